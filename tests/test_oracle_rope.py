"""Pins of the oracle's key re-rotation for position-aware affix registration.

Source: "Affix Cache for Diffusion Large Language Models", Sec. 4 (opening) and Limitations:
the cache is kept after the rotary position rotation, so an affix reused at another offset
needs its keys moved.  Reading R8: rotate every frequency pair i by delta * theta^(-2i/d).

Pins: delta 0 is the identity, the first pair's frequency is 1 (a closed-form rotation by
delta radians), rotations compose, pair norms are preserved, and the half-split layout equals
multiplying by exp(i w) with torch's complex arithmetic.
"""
import math

import numpy as np
import pytest
import torch

import oracle


def test_delta_zero_is_identity():
    k = torch.randn((5, 3, 16), generator=torch.Generator().manual_seed(1))
    assert np.array_equal(oracle.rerotate(k, 0, 10000.0), k.double().numpy())


@pytest.mark.parametrize("interleaved", [False, True])
def test_first_pair_rotates_by_delta_radians(interleaved):
    k = torch.zeros((1, 1, 2))
    k[0, 0, 0] = 1.0
    out = oracle.rerotate(k, 3, 500000.0, interleaved)
    np.testing.assert_allclose(out[0, 0], [math.cos(3.0), math.sin(3.0)], atol=1e-15)


@pytest.mark.parametrize("interleaved", [False, True])
def test_rotations_compose_and_preserve_pair_norms(interleaved):
    k = torch.randn((7, 2, 32), generator=torch.Generator().manual_seed(2))
    a = oracle.rerotate(k, 11, 1e6, interleaved)
    ab = oracle.rerotate(torch.from_numpy(a).float(), 29, 1e6, interleaved)   # float32 rounding of a
    direct = oracle.rerotate(k, 40, 1e6, interleaved)
    np.testing.assert_allclose(ab, direct, atol=1e-5)
    back = oracle.rerotate(torch.from_numpy(a).float(), -11, 1e6, interleaved)
    np.testing.assert_allclose(back, k.double().numpy(), atol=1e-5)
    half = 16
    if interleaved:
        na = a[..., 0::2] ** 2 + a[..., 1::2] ** 2
        nk = k.double().numpy()[..., 0::2] ** 2 + k.double().numpy()[..., 1::2] ** 2
    else:
        na = a[..., :half] ** 2 + a[..., half:] ** 2
        nk = k.double().numpy()[..., :half] ** 2 + k.double().numpy()[..., half:] ** 2
    np.testing.assert_allclose(na, nk, rtol=1e-12)


def test_half_split_equals_complex_multiplication():
    d, delta, theta = 64, 1234, 10000.0
    k = torch.randn((4, 3, d), generator=torch.Generator().manual_seed(3)).double()
    z = torch.complex(k[..., : d // 2], k[..., d // 2:])
    freq = theta ** (-2.0 * torch.arange(d // 2, dtype=torch.float64) / d)
    rot = z * torch.polar(torch.ones(d // 2, dtype=torch.float64), delta * freq)
    want = torch.cat([rot.real, rot.imag], dim=-1).numpy()
    np.testing.assert_allclose(oracle.rerotate(k.float(), delta, theta), want, atol=1e-6)
