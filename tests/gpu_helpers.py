"""Helpers shared by the GPU parity tests: run each step of the path through the C ABI on
the same seeded inputs the oracle sees, and compare with the tolerances of the path.

Tolerances (stated for the path): slot tables, scatter destinations and anchor sets are
bit-exact (anchor offsets whose oracle score lies within 1e-3 relative of the K-th
oracle score are exempt); importance scores agree within 1e-3 relative (plus a floor
of 1e-7 of the largest score for entries that underflow); attention outputs within
2e-2 absolute for bf16 inputs and 1e-5 absolute for float32.
"""
from __future__ import annotations

import numpy as np
import torch

import affix_kv_cache_gb300 as ac
import oracle
from affix_kv_cache_gb300 import workloads as wl

OUT_TOL = {"bf16": 2e-2, "f32": 1e-5}
SCORE_RTOL = 1e-3
SCORE_FLOOR = 1e-7
TIE_BAND = 1e-3


def dev(x, device="cuda"):
    return x.to(device, non_blocking=False).contiguous()


def desc_of(w: wl.Workload):
    return ac.attn_desc(w.hq, w.hkv, w.d, w.scale, w.dtype)


def status_tensor():
    return torch.zeros(1, dtype=torch.int32, device="cuda")


def probe_layer_gpu(w, inp, scores, masked=None, out=True, workspace=None, dev_status=None):
    """One probe layer through the C ABI; returns the probe output (or None)."""
    d = desc_of(w)
    q, kr, vr, ka, va = (dev(inp[k]) for k in ("q", "k_req", "v_req", "k_aff", "v_aff"))
    if masked is None:
        masked = torch.tensor(w.masked_rows(), dtype=torch.int32).expand(w.batch, -1)
    masked = dev(masked.to(torch.int32))
    o = torch.empty_like(q) if out else None
    need = ac.acache_probe_workspace_bytes(d, w.batch, w.T, w.L, masked.shape[1])
    if workspace is None:
        workspace = torch.empty(max(need, 1), dtype=torch.uint8, device="cuda")
    ac.acache_probe_scores(d, w.batch, w.T, w.l, w.L, masked, masked.shape[1], q, kr, vr, ka, va,
                           o, scores, workspace, dev_status=dev_status)
    return o


def assert_scores_close(got, want, what=""):
    got = np.asarray(got, np.float64)
    want = np.asarray(want, np.float64)
    floor = SCORE_FLOOR * max(float(np.abs(want).max()), 1e-30)
    err = np.abs(got - want)
    tol = SCORE_RTOL * np.abs(want) + floor
    bad = err > tol
    assert not bad.any(), (f"{what}: {bad.sum()} scores outside 1e-3 rel; worst "
                           f"{(err / np.maximum(np.abs(want), 1e-300)).max():.3e}")


def assert_out_close(got, want, dtype, what=""):
    got = np.asarray(got, np.float64)
    err = np.abs(got - want)
    tol = OUT_TOL[dtype]
    assert err.max() <= tol, f"{what}: max |err| {err.max():.3e} > {tol}"


def assert_anchors_match(got, oracle_scores, K, what=""):
    """Anchor sets bit-exact except offsets within the tie band of the K-th oracle score."""
    got = np.asarray(got)
    s = np.asarray(oracle_scores, np.float64)
    want = oracle.topk_anchors(s, K)
    for b in range(s.shape[0]):
        assert np.all(np.diff(got[b]) > 0), f"{what}: anchors of request {b} not ascending"
        if K == 0:
            continue
        kth = np.sort(s[b])[::-1][K - 1]
        diff = set(got[b].tolist()) ^ set(want[b].tolist())
        for j in diff:
            assert abs(s[b, j] - kth) <= TIE_BAND * abs(kth), (
                f"{what}: request {b} offset {j} differs outside the tie band "
                f"(score {s[b, j]:.6e}, K-th {kth:.6e})")


def register_shared(w, lay, k_aff, v_aff, kc, vc):
    """Store the shared precomputed affix K/V into the pool's shared region (admission)."""
    d = desc_of(w)
    ac.acache_write_slots(d, 1, w.L, dev(lay.shared_slot), dev(k_aff), dev(v_aff), kc, vc,
                          lay.num_slots, 0)
