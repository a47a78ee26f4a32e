"""GPU parity of the CacheBlend-style (high KV deviation) selector against the oracle.

Scores within 1e-3 relative (the path's score tolerance), bit-reproducible across runs,
accumulated over layers; the anchors the GPU Top-K picks from the GPU scores equal the
oracle's ranking of the very same float32 scores.
"""
import numpy as np
import pytest
import torch

import affix_kv_cache_gb300 as ac
import oracle

from gpu_helpers import assert_scores_close, dev

pytestmark = pytest.mark.gpu


def _inputs(B, L, hkv, d, dtype, seed):
    g = torch.Generator().manual_seed(seed)
    ks, vs = torch.randn((L, hkv, d), generator=g), torch.randn((L, hkv, d), generator=g)
    kf = ks[None] + torch.randn((B, L, hkv, d), generator=g) * torch.rand((B, L, 1, 1), generator=g)
    vf = vs[None] + torch.randn((B, L, hkv, d), generator=g) * torch.rand((B, L, 1, 1), generator=g)
    return [x.to(dtype) for x in (ks, vs, kf, vf)]


@pytest.mark.parametrize("dtype,d,hkv,B,L", [(torch.bfloat16, 128, 32, 2, 300), (torch.bfloat16, 128, 4, 3, 37),
                                             (torch.bfloat16, 128, 1, 2, 129), (torch.bfloat16, 64, 2, 2, 50),
                                             (torch.float32, 64, 2, 1, 128), (torch.float32, 128, 3, 2, 33)])
def test_kv_deviation_parity(dtype, d, hkv, B, L):
    layers = [_inputs(B, L, hkv, d, dtype, seed) for seed in (1, 2)]
    desc = ac.attn_desc(hkv, hkv, d, d ** -0.5, dtype)
    scores = torch.zeros((B, L), dtype=torch.float32, device="cuda")
    ref = None
    for ks, vs, kf, vf in layers:
        ac.acache_kv_deviation_scores(desc, B, L, dev(ks), dev(vs), dev(kf), dev(vf), scores)
        ref = oracle.kv_deviation(ks, vs, kf, vf, scores=ref)
    got = scores.cpu().numpy()
    assert_scores_close(got, ref, "kv deviation")
    again = torch.zeros_like(scores)
    for ks, vs, kf, vf in layers:
        ac.acache_kv_deviation_scores(desc, B, L, dev(ks), dev(vs), dev(kf), dev(vf), again)
    assert torch.equal(again, scores), "not bit-reproducible"
    K = max(1, L // 5)
    anchors = torch.empty((B, K), dtype=torch.int32, device="cuda")
    st = torch.zeros(1, dtype=torch.int32, device="cuda")
    ac.acache_topk_anchors(scores, B, L, K, anchors, dev_status=st)
    torch.cuda.synchronize()
    assert st.item() == 0
    want = oracle.topk_anchors(got.astype(np.float64), K)
    assert np.array_equal(anchors.cpu().numpy(), want)


# ----------------------------------------------------------------------------- DropNA
# (B, n_q, Hq, Hkv, T, dtype, d): the recompute-point kernel (many query rows), the block-decode
# kernel (32 queries, GQA and MHA with clusters) and the float32 CUDA-core kernel.
DROP_CASES = [(2, 300, 4, 2, 700, torch.bfloat16, 128), (2, 32, 8, 4, 500, torch.bfloat16, 128),
              (1, 32, 4, 4, 1408, torch.bfloat16, 128), (2, 40, 2, 2, 200, torch.float32, 64),
              (3, 5, 2, 2, 37, torch.bfloat16, 128)]


@pytest.mark.parametrize("B,n_q,hq,hkv,T,dtype,d", DROP_CASES)
def test_dropna_slot_attention_parity(B, n_q, hq, hkv, T, dtype, d):
    ns = 3000
    g = torch.Generator().manual_seed(B * 100 + n_q + T)
    kc = torch.randn((ns, hkv, d), generator=g).to(dtype)
    vc = torch.randn((ns, hkv, d), generator=g).to(dtype)
    q = (torch.randn((B, n_q, hq, d), generator=g) * 2).to(dtype)
    rs = torch.randint(0, ns, (B, T), generator=g, dtype=torch.int32)
    rs[0, :min(T, 128)] = -1                                                  # a whole key tile discarded
    rs[0, 130::3] = -1
    if B > 1:
        rs[B - 1, :] = -1                                                      # no key left: zeros
    ref = oracle.slot_attention(q, rs, kc, vc, scale=d ** -0.5, drop_none=True)
    out = torch.full((B, n_q, hq, d), float("nan"), dtype=dtype, device="cuda")
    st = torch.zeros(1, dtype=torch.int32, device="cuda")
    ac.acache_slot_attention_dropna(ac.attn_desc(hq, hkv, d, d ** -0.5, dtype), B, n_q, dev(q), T, dev(rs),
                                    dev(kc), dev(vc), ns, out, dev_status=st)
    torch.cuda.synchronize()
    assert st.item() == 0
    tol = 2e-2 if dtype == torch.bfloat16 else 1e-5
    err = (out.double().cpu().numpy() - ref)
    assert np.abs(err).max() <= tol, f"max |err| {np.abs(err).max():.3e}"
    if B > 1:
        assert torch.all(out[B - 1] == 0)


@pytest.mark.parametrize("lo,hi", [(384, 700), (0, 384), (0, 700), (383, 385)])
def test_dropna_lone_query_tile_with_a_discarded_key_half(lo, hi):
    # One query tile and six key tiles: the kernel gives each of its two chains three key tiles
    # and merges their partial softmax states, so discarding keys [384, 700) or [0, 384) leaves
    # one chain with no key at all, and [0, 700) both.
    d, hq, hkv, T, ns, n_q = 128, 2, 2, 700, 2000, 100
    g = torch.Generator().manual_seed(lo * 7 + hi)
    kc = torch.randn((ns, hkv, d), generator=g).to(torch.bfloat16)
    vc = torch.randn((ns, hkv, d), generator=g).to(torch.bfloat16)
    q = (torch.randn((1, n_q, hq, d), generator=g) * 2).to(torch.bfloat16)
    rs = torch.randint(0, ns, (1, T), generator=g, dtype=torch.int32)
    rs[0, lo:hi] = -1
    ref = oracle.slot_attention(q, rs, kc, vc, scale=d ** -0.5, drop_none=True)
    out = torch.full((1, n_q, hq, d), float("nan"), dtype=torch.bfloat16, device="cuda")
    st = torch.zeros(1, dtype=torch.int32, device="cuda")
    ac.acache_slot_attention_dropna(ac.attn_desc(hq, hkv, d, d ** -0.5, "bf16"), 1, n_q, dev(q), T, dev(rs),
                                    dev(kc), dev(vc), ns, out, dev_status=st)
    torch.cuda.synchronize()
    assert st.item() == 0
    err = np.abs(out.double().cpu().numpy() - ref)
    assert err.max() <= 2e-2, f"max |err| {err.max():.3e}"
    if hi - lo == T:
        assert torch.all(out == 0)


def test_dropna_other_negative_slots_still_flag():
    d, hq, hkv, T, ns = 128, 2, 2, 150, 300
    g = torch.Generator().manual_seed(21)
    kc = torch.randn((ns, hkv, d), generator=g).to(torch.bfloat16)
    vc = torch.randn((ns, hkv, d), generator=g).to(torch.bfloat16)
    q = torch.randn((1, 40, hq, d), generator=g).to(torch.bfloat16)
    rs = torch.randint(0, ns, (1, T), generator=g, dtype=torch.int32)
    rs[0, 7] = -2
    out = torch.empty((1, 40, hq, d), dtype=torch.bfloat16, device="cuda")
    st = torch.zeros(1, dtype=torch.int32, device="cuda")
    ac.acache_slot_attention_dropna(ac.attn_desc(hq, hkv, d, d ** -0.5, "bf16"), 1, 40, dev(q), T, dev(rs),
                                    dev(kc), dev(vc), ns, out, dev_status=st)
    torch.cuda.synchronize()
    assert st.item() == 1   # ACACHE_DEV_BAD_SLOT
