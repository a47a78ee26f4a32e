"""Pins of the oracle's CacheBlend-style selector (high KV deviation).

Source: "Affix Cache for Diffusion Large Language Models", App. B.5: the variant ranks affix
tokens by the KV difference between the affix-only cache and the full-prompt cache, and then
takes the same Top-K as ACache (Eq. 6).  Reading taken: per KV head, the L2 norm of the key
difference plus the L2 norm of the value difference, summed over KV heads and layers.

Pins: exact closed forms (Pythagorean triples), zero for identical caches, additivity over
layers, homogeneity (a norm, not a squared norm), invariance under permuting KV heads, and a
planted set of high-deviation tokens that must come out as the Top-K.
"""
import numpy as np
import pytest
import torch

import oracle


def _zeros(B, L, hkv, d, dtype):
    ks = torch.zeros((L, hkv, d), dtype=dtype)
    return ks, ks.clone(), torch.zeros((B, L, hkv, d), dtype=dtype), torch.zeros((B, L, hkv, d), dtype=dtype)


@pytest.mark.parametrize("dtype", [torch.float32, torch.bfloat16])
def test_pythagorean_closed_form(dtype):
    ks, vs, kf, vf = _zeros(1, 2, 2, 4, dtype)
    kf[0, 0, 0, :2] = torch.tensor([3.0, 4.0])        # head 0 key: |(3,4)| = 5
    vf[0, 0, 0, 0] = 1.0                               # head 0 value: 1
    vf[0, 0, 1, 1:3] = torch.tensor([6.0, 8.0])       # head 1 value: |(6,8)| = 10
    ks[1, 1, 3] = 2.0                                  # token 1: shared key differs by -2 -> 2
    s = oracle.kv_deviation(ks, vs, kf, vf)
    assert s.tolist() == [[16.0, 2.0]]


def test_identical_caches_score_zero_and_topk_takes_lowest_offsets():
    g = torch.Generator().manual_seed(3)
    ks = torch.randn((11, 2, 8), generator=g)
    vs = torch.randn((11, 2, 8), generator=g)
    s = oracle.kv_deviation(ks, vs, ks[None].repeat(2, 1, 1, 1), vs[None].repeat(2, 1, 1, 1))
    assert np.all(s == 0.0)
    assert oracle.topk_anchors(s, 4).tolist() == [[0, 1, 2, 3]] * 2


def test_accumulates_over_layers():
    g = torch.Generator().manual_seed(4)
    args = [torch.randn(sh, generator=g) for sh in ((7, 3, 8), (7, 3, 8), (2, 7, 3, 8), (2, 7, 3, 8))]
    one = oracle.kv_deviation(*args)
    two = oracle.kv_deviation(*args, scores=one)
    np.testing.assert_allclose(two, 2 * one, rtol=1e-15)


def test_norm_not_squared_norm_and_both_k_and_v_count():
    ks, vs, kf, vf = _zeros(1, 1, 1, 4, torch.float32)
    kf[0, 0, 0, 0] = 1.0
    base = oracle.kv_deviation(ks, vs, kf, vf)[0, 0]
    kf3 = kf * 3
    assert oracle.kv_deviation(ks, vs, kf3, vf)[0, 0] == 3 * base      # homogeneous of degree 1
    vf[0, 0, 0, 2] = 0.5
    assert oracle.kv_deviation(ks, vs, kf, vf)[0, 0] == base + 0.5     # the value term adds


def test_kv_head_permutation_invariance():
    g = torch.Generator().manual_seed(5)
    ks, vs = torch.randn((9, 4, 16), generator=g), torch.randn((9, 4, 16), generator=g)
    kf, vf = torch.randn((2, 9, 4, 16), generator=g), torch.randn((2, 9, 4, 16), generator=g)
    perm = torch.tensor([2, 0, 3, 1])
    a = oracle.kv_deviation(ks, vs, kf, vf)
    b = oracle.kv_deviation(ks[:, perm], vs[:, perm], kf[:, :, perm], vf[:, :, perm])
    np.testing.assert_allclose(a, b, rtol=1e-13)


def test_planted_high_deviation_tokens_are_the_topk():
    g = torch.Generator().manual_seed(6)
    B, L, hkv, d = 3, 64, 2, 32
    ks, vs = torch.randn((L, hkv, d), generator=g), torch.randn((L, hkv, d), generator=g)
    kf = ks[None].repeat(B, 1, 1, 1) + 0.01 * torch.randn((B, L, hkv, d), generator=g)
    vf = vs[None].repeat(B, 1, 1, 1) + 0.01 * torch.randn((B, L, hkv, d), generator=g)
    planted = [sorted(torch.randperm(L, generator=g)[:6].tolist()) for _ in range(B)]
    for b in range(B):
        for j in planted[b]:
            kf[b, j] += torch.randn((hkv, d), generator=g)
    s = oracle.kv_deviation(ks, vs, kf, vf)
    assert oracle.topk_anchors(s, 6).tolist() == planted


# ----------------------------------------------------------------------------- DropNA
# Sec. 5.3 (Figure 5): DropNA recomputes the same anchors but discards every non-anchor affix
# entry.  Reading: a discarded position has no key; a row with no key left outputs zeros.
def _pool(num_slots, hkv, d, seed):
    g = torch.Generator().manual_seed(seed)
    return torch.randn((num_slots, hkv, d), generator=g), torch.randn((num_slots, hkv, d), generator=g)


def _sdpa(q, k, v, scale):
    """torch float64 attention; q [n][Hq][d], k/v [T][Hkv][d]."""
    g = q.shape[1] // k.shape[1]
    kk = k.double().repeat_interleave(g, dim=1).permute(1, 0, 2).unsqueeze(0)
    vv = v.double().repeat_interleave(g, dim=1).permute(1, 0, 2).unsqueeze(0)
    o = torch.nn.functional.scaled_dot_product_attention(q.double().permute(1, 0, 2).unsqueeze(0), kk, vv,
                                                         scale=scale)
    return o.squeeze(0).permute(1, 0, 2)


@pytest.mark.parametrize("hq,hkv", [(2, 2), (4, 2)])
def test_dropna_equals_attention_over_the_kept_keys(hq, hkv):
    B, nq, T, d, ns = 2, 5, 23, 8, 40
    kc, vc = _pool(ns, hkv, d, 7)
    g = torch.Generator().manual_seed(8)
    q = torch.randn((B, nq, hq, d), generator=g)
    rs = torch.randint(0, ns, (B, T), generator=g, dtype=torch.int32)
    rs[0, 3:11] = -1
    rs[1, ::3] = -1
    got = oracle.slot_attention(q, rs, kc, vc, scale=d ** -0.5, drop_none=True)
    for b in range(B):
        keep = rs[b][rs[b] >= 0].long()
        want = _sdpa(q[b], kc[keep], vc[keep], d ** -0.5)
        np.testing.assert_allclose(got[b], want.numpy(), atol=1e-12)


def test_dropna_key_is_not_a_zero_row():
    kc, vc = _pool(10, 1, 4, 9)
    kc[9] = 0.0
    vc[9] = 0.0
    q = torch.randn((1, 1, 1, 4), generator=torch.Generator().manual_seed(10))
    drop = oracle.slot_attention(q, torch.tensor([[0, 1, -1]], dtype=torch.int32), kc, vc, scale=0.5,
                                 drop_none=True)
    zero = oracle.slot_attention(q, torch.tensor([[0, 1, 9]], dtype=torch.int32), kc, vc, scale=0.5)
    two = oracle.slot_attention(q, torch.tensor([[0, 1]], dtype=torch.int32), kc, vc, scale=0.5)
    np.testing.assert_allclose(drop, two, atol=1e-14)
    assert np.abs(drop - zero).max() > 1e-3


def test_dropna_row_without_keys_outputs_zeros():
    kc, vc = _pool(4, 1, 4, 11)
    q = torch.randn((1, 2, 1, 4), generator=torch.Generator().manual_seed(12))
    out = oracle.slot_attention(q, torch.full((1, 6), -1, dtype=torch.int32), kc, vc, scale=0.5,
                                drop_none=True)
    assert np.all(out == 0.0)


def test_dropna_equals_keepna_at_ratio_one():
    # K = L: every affix position is an anchor, no shared entry is left to discard
    T, l, L, B = 20, 4, 9, 2
    K = L
    R = K + T - L
    anchors = np.tile(np.arange(L, dtype=np.int32), (B, 1))
    shared = np.arange(100, 100 + L, dtype=np.int32)
    priv = np.arange(B * R, dtype=np.int32).reshape(B, R)
    _, keep = oracle.build_slot_maps(anchors, shared, priv, T=T, l=l, L=L)
    _, drop = oracle.build_slot_maps(anchors, np.full(L, -1, np.int32), priv, T=T, l=l, L=L)
    assert np.array_equal(keep, drop)
    kc, vc = _pool(B * R, 2, 8, 13)
    q = torch.randn((B, 3, 2, 8), generator=torch.Generator().manual_seed(14))
    a = oracle.slot_attention(q, keep, kc, vc, scale=0.3)
    b = oracle.slot_attention(q, drop, kc, vc, scale=0.3, drop_none=True)
    assert np.array_equal(a, b)


def test_dropna_map_discards_exactly_the_non_anchor_affix_positions():
    T, l, L, B, K = 30, 5, 16, 2, 4
    R = K + T - L
    g = np.random.default_rng(15)
    anchors = np.stack([np.sort(g.choice(L, K, replace=False)) for _ in range(B)]).astype(np.int32)
    priv = np.arange(B * R, dtype=np.int32).reshape(B, R)
    _, rs = oracle.build_slot_maps(anchors, np.full(L, -1, np.int32), priv, T=T, l=l, L=L)
    for b in range(B):
        dropped = {t for t in range(T) if rs[b, t] == -1}
        assert dropped == {l + j for j in range(L) if j not in set(anchors[b].tolist())}
