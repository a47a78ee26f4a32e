"""GPU parity: every entry point of the C ABI against the CPU oracle on the same seeded inputs.

Sizes are small enough for the oracle to finish in seconds but span several 128-row /
128-key tiles with ragged tails.  Tolerances are those of the path (see gpu_helpers).
"""
import numpy as np
import pytest
import torch

import affix_kv_cache_gb300 as ac
import oracle
from affix_kv_cache_gb300 import workloads as wl

from gpu_helpers import (assert_anchors_match, assert_out_close, assert_scores_close, desc_of, dev,
                         probe_layer_gpu, register_shared, status_tensor)

pytestmark = pytest.mark.gpu


def tiny(segments, hq=4, hkv=2, d=128, batch=2, ratio=200, dtype="bf16", **kw):
    return wl.Workload(name="parity", dtype=dtype, layers=1, hq=hq, hkv=hkv, d=d, batch=batch,
                       segments=tuple(segments), ratio_permille=ratio, recompute_points=1, **kw)


# several tiles with ragged tails: P = 300 probe rows, m = 150 masked, L = 400, T = 700
RAGGED = {
    "prefix": [(wl.SEG_AFFIX, 400), (wl.SEG_REQ, 150), (wl.SEG_MASK, 150)],
    "infix": [(wl.SEG_REQ, 100), (wl.SEG_AFFIX, 400), (wl.SEG_REQ, 50), (wl.SEG_MASK, 150)],
    "suffix": [(wl.SEG_REQ, 150), (wl.SEG_MASK, 150), (wl.SEG_AFFIX, 400)],
}
SMALL = [(wl.SEG_REQ, 5), (wl.SEG_AFFIX, 37), (wl.SEG_REQ, 3), (wl.SEG_MASK, 19)]


# ------------------------------------------------------------------ store / gather / maps
@pytest.mark.parametrize("dtype,d,heads", [("bf16", 128, (4, 2)), ("f32", 64, (2, 2)),
                                           ("bf16", 64, (8, 8))])
def test_write_slots_bit_exact(dtype, d, heads):
    w = tiny(RAGGED["infix"], hq=heads[0], hkv=heads[1], d=d, dtype=dtype, batch=3, page=64)
    lay = wl.slot_layout(w)
    rec = wl.recompute_inputs(w, 0)
    g = torch.Generator().manual_seed(3)
    kc = torch.randn((lay.num_slots, w.hkv, w.d), generator=g).to(w.torch_dtype)
    vc = torch.randn((lay.num_slots, w.hkv, w.d), generator=g).to(w.torch_dtype)
    kb, vb, flags = oracle.write_slots(lay.private_slots, rec["k_new"], rec["v_new"], kc, vc,
                                       private_begin=lay.private_begin)
    kd, vd = dev(kc), dev(vc)
    st = status_tensor()
    ac.acache_write_slots(desc_of(w), w.batch, w.R, dev(lay.private_slots), dev(rec["k_new"]),
                          dev(rec["v_new"]), kd, vd, lay.num_slots, lay.private_begin, dev_status=st)
    torch.cuda.synchronize()
    assert st.item() == 0 and flags == 0
    assert np.array_equal(kd.cpu().view(torch.uint8).reshape(-1).numpy(), kb)
    assert np.array_equal(vd.cpu().view(torch.uint8).reshape(-1).numpy(), vb)


def test_write_slots_skips_and_flags_bad_slots():
    w = tiny(SMALL, batch=2, page=16)
    lay = wl.slot_layout(w)
    rec = wl.recompute_inputs(w, 0)
    ws = lay.private_slots.clone()
    ws[0, 0] = 1                         # inside the shared region
    ws[1, 3] = lay.num_slots + 5         # outside the pool
    ws[1, 4] = -2
    kc = torch.zeros((lay.num_slots, w.hkv, w.d), dtype=w.torch_dtype)
    kb, vb, flags = oracle.write_slots(ws, rec["k_new"], rec["v_new"], kc, kc,
                                       private_begin=lay.private_begin)
    kd, vd = dev(kc), dev(kc.clone())
    st = status_tensor()
    ac.acache_write_slots(desc_of(w), w.batch, w.R, dev(ws), dev(rec["k_new"]), dev(rec["v_new"]),
                          kd, vd, lay.num_slots, lay.private_begin, dev_status=st)
    torch.cuda.synchronize()
    assert st.item() == (ac._lib.DEV_BAD_SLOT | ac._lib.DEV_SHARED_WRITE) == flags
    assert np.array_equal(kd.cpu().view(torch.uint8).reshape(-1).numpy(), kb)
    assert np.array_equal(vd.cpu().view(torch.uint8).reshape(-1).numpy(), vb)


@pytest.mark.parametrize("dtype,d", [("bf16", 128), ("f32", 64)])
def test_gather_slots_bit_exact(dtype, d):
    w = tiny(RAGGED["prefix"], d=d, dtype=dtype, batch=3, page=64)
    lay = wl.slot_layout(w)
    g = torch.Generator().manual_seed(5)
    kc = torch.randn((lay.num_slots, w.hkv, w.d), generator=g).to(w.torch_dtype)
    vc = torch.randn((lay.num_slots, w.hkv, w.d), generator=g).to(w.torch_dtype)
    rs = torch.randint(0, lay.num_slots, (w.batch, w.T), generator=g, dtype=torch.int32)
    ko, vo, flags = oracle.gather_slots(rs, kc, vc)
    kd = torch.empty((w.batch, w.T, w.hkv, w.d), dtype=w.torch_dtype, device="cuda")
    vd = torch.empty_like(kd)
    ac.acache_gather_slots(desc_of(w), w.batch, w.T, dev(rs), dev(kc), dev(vc), lay.num_slots, kd, vd)
    torch.cuda.synchronize()
    assert np.array_equal(kd.cpu().view(torch.uint8).reshape(-1).numpy(), ko)
    assert np.array_equal(vd.cpu().view(torch.uint8).reshape(-1).numpy(), vo)


@pytest.mark.parametrize("layout", list(RAGGED))
@pytest.mark.parametrize("ratio", [0, 200, 1000])
def test_build_slot_maps_bit_exact(layout, ratio):
    w = tiny(RAGGED[layout], ratio=ratio, batch=3, page=64)
    lay = wl.slot_layout(w)
    rng = np.random.default_rng(ratio + len(layout))
    anchors = np.stack([np.sort(rng.choice(w.L, w.K, replace=False))
                        for _ in range(w.batch)]).astype(np.int32).reshape(w.batch, w.K)
    wp, rs = oracle.build_slot_maps(anchors, lay.shared_slot, lay.private_slots, T=w.T, l=w.l, L=w.L)
    wpd = torch.full((w.batch, w.R), -7, dtype=torch.int32, device="cuda")
    rsd = torch.full((w.batch, w.T), -7, dtype=torch.int32, device="cuda")
    st = status_tensor()
    ac.acache_build_slot_maps(w.batch, w.T, w.l, w.L, w.K, dev(torch.from_numpy(anchors)),
                              dev(lay.shared_slot), dev(lay.private_slots), wpd, rsd, dev_status=st)
    torch.cuda.synchronize()
    assert st.item() == 0
    assert np.array_equal(wpd.cpu().numpy(), wp)
    assert np.array_equal(rsd.cpu().numpy(), rs)


def test_build_slot_maps_flags_bad_anchors():
    w = tiny(SMALL, ratio=500, batch=2)
    lay = wl.slot_layout(w)
    anchors = torch.stack([torch.arange(w.K, dtype=torch.int32)] * 2)
    anchors[1, 2] = anchors[1, 1]                    # not strictly ascending
    rsd = torch.full((w.batch, w.T), -7, dtype=torch.int32, device="cuda")
    wpd = torch.full((w.batch, w.R), -7, dtype=torch.int32, device="cuda")
    st = status_tensor()
    ac.acache_build_slot_maps(w.batch, w.T, w.l, w.L, w.K, dev(anchors), dev(lay.shared_slot),
                              dev(lay.private_slots), wpd, rsd, dev_status=st)
    torch.cuda.synchronize()
    assert st.item() == ac._lib.DEV_BAD_ANCHOR
    assert (rsd[1] == -7).all() and (rsd[0] != -7).all()     # request 1 untouched


# ------------------------------------------------------------------ Top-K
@pytest.mark.parametrize("L,K", [(1, 1), (37, 0), (37, 8), (400, 80), (1024, 205), (8192, 1639),
                                 (3000, 3000), (50000, 777)])
def test_topk_bit_exact(L, K):
    g = torch.Generator().manual_seed(L + K)
    s = torch.rand((4, L), generator=g)
    s[1] = torch.round(s[1] * 8) / 8                 # heavy exact ties
    s[2] = 0.5                                        # all equal
    s[3, ::3] = 0.0
    s[3, 1::3] = -0.0                                 # -0.0 ranks as +0.0
    sd = dev(s)
    a = torch.empty((4, K), dtype=torch.int32, device="cuda")
    st = status_tensor()
    ac.acache_topk_anchors(sd, 4, L, K, a, dev_status=st)
    torch.cuda.synchronize()
    assert st.item() == 0
    # the oracle decides on the very same float32 values (exact in float64)
    want = oracle.topk_anchors(s.double().numpy(), K)
    assert np.array_equal(a.cpu().numpy(), want)


def test_topk_flags_nan():
    s = torch.rand((1, 100))
    s[0, 7] = float("nan")
    a = torch.empty((1, 10), dtype=torch.int32, device="cuda")
    st = status_tensor()
    ac.acache_topk_anchors(dev(s), 1, 100, 10, a, dev_status=st)
    torch.cuda.synchronize()
    assert st.item() == ac._lib.DEV_NAN
    assert 7 not in a.cpu().numpy()[0].tolist()


# ------------------------------------------------------------------ probe
@pytest.mark.parametrize("layout", list(RAGGED))
@pytest.mark.parametrize("dtype,d,heads", [("bf16", 128, (4, 2)), ("f32", 64, (2, 2)),
                                           ("bf16", 128, (7, 1))])
def test_probe_parity(layout, dtype, d, heads):
    w = tiny(RAGGED[layout], hq=heads[0], hkv=heads[1], d=d, dtype=dtype, batch=2)
    inp = wl.probe_inputs(w, 0)
    ref = oracle.probe_layer(inp["q"], inp["k_req"], inp["v_req"], inp["k_aff"], inp["v_aff"],
                             T=w.T, l=w.l, masked_rows=w.masked_rows(), scale=w.scale)
    scores = torch.zeros((w.batch, w.L), dtype=torch.float32, device="cuda")
    o = probe_layer_gpu(w, inp, scores)
    torch.cuda.synchronize()
    assert_out_close(o.float().cpu().numpy(), ref["out"], dtype, "probe output")
    assert_scores_close(scores.cpu().numpy(), ref["scores"], "probe scores")


# More 256-row blocks of probe rows than SMs (4 requests x 32 query heads x 2 blocks = 256):
# the forward runs in two waves, the last block of a (request, head) a one-tile block whose keys
# the two chains split.  GQA (8 KV heads) and MHA; the affix as prefix and as infix.
@pytest.mark.parametrize("layout,hkv", [("prefix", 8), ("infix", 32)])
def test_probe_parity_more_blocks_than_sms(layout, hkv):
    w = tiny(RAGGED[layout], hq=32, hkv=hkv, batch=4)
    inp = wl.probe_inputs(w, 0)
    ref = oracle.probe_layer(inp["q"], inp["k_req"], inp["v_req"], inp["k_aff"], inp["v_aff"],
                             T=w.T, l=w.l, masked_rows=w.masked_rows(), scale=w.scale)
    scores = torch.zeros((w.batch, w.L), dtype=torch.float32, device="cuda")
    st = status_tensor()
    o = probe_layer_gpu(w, inp, scores, dev_status=st)
    torch.cuda.synchronize()
    assert st.item() == 0
    assert_out_close(o.float().cpu().numpy(), ref["out"], "bf16", "probe output")
    assert_scores_close(scores.cpu().numpy(), ref["scores"], "probe scores")


@pytest.mark.parametrize("m,consecutive", [(256, True), (257, True), (400, True), (200, False), (300, False)])
def test_probe_parity_masked_row_counts(m, consecutive):
    """Up to 256 masked rows (two 128-row chunks) the masked-to-affix mass keeps them resident
    in shared memory; more go through the one-tile-per-CTA kernel.  Consecutive masked rows
    are box loads, scattered ones gathered."""
    w = tiny([(wl.SEG_AFFIX, 400), (wl.SEG_REQ, 100), (wl.SEG_MASK, 300)], batch=2)
    if consecutive:
        rows = list(range(w.P - m, w.P))
    else:
        rows = sorted(np.random.default_rng(m).choice(w.P, m, replace=False).tolist())
    inp = wl.probe_inputs(w, 0)
    ref = oracle.probe_layer(inp["q"], inp["k_req"], inp["v_req"], inp["k_aff"], inp["v_aff"],
                             T=w.T, l=w.l, masked_rows=rows, scale=w.scale, want_out=False)
    scores = torch.zeros((w.batch, w.L), dtype=torch.float32, device="cuda")
    st = status_tensor()
    probe_layer_gpu(w, inp, scores, masked=torch.tensor(rows, dtype=torch.int32).expand(w.batch, -1),
                    out=False, dev_status=st)
    torch.cuda.synchronize()
    assert st.item() == 0
    assert_scores_close(scores.cpu().numpy(), ref["scores"], f"{m} masked rows")


def test_probe_accumulates_over_layers_and_is_deterministic():
    w = tiny(RAGGED["infix"], batch=2).replace(layers=3)
    ref = None
    s1 = torch.zeros((w.batch, w.L), dtype=torch.float32, device="cuda")
    s2 = torch.zeros_like(s1)
    for n in range(w.layers):
        inp = wl.probe_inputs(w, n)
        ref = oracle.probe_layer(inp["q"], inp["k_req"], inp["v_req"], inp["k_aff"], inp["v_aff"],
                                 T=w.T, l=w.l, masked_rows=w.masked_rows(), scale=w.scale,
                                 scores=None if ref is None else ref["scores"], want_out=False)
        o1 = probe_layer_gpu(w, inp, s1)
        o2 = probe_layer_gpu(w, inp, s2)
        torch.cuda.synchronize()
        assert torch.equal(o1, o2)
    assert torch.equal(s1, s2)
    assert_scores_close(s1.cpu().numpy(), ref["scores"], "3-layer scores")


@pytest.mark.parametrize("dtype,d,heads,feed", [("bf16", 128, (4, 2), False), ("bf16", 128, (4, 2), True),
                                                ("f32", 64, (2, 2), False)])
def test_probe_layers_matches_per_layer_calls(dtype, d, heads, feed):
    """acache_probe_scores_layers is bit-identical to one acache_probe_scores call per layer.
    feed: layer n's output buffer is layer n+1's query buffer, so the call must not chain
    (the host's overlap check) and each layer reads what the previous one wrote."""
    w = tiny(RAGGED["suffix"], hq=heads[0], hkv=heads[1], d=d, dtype=dtype, batch=2).replace(layers=4)
    inps = [wl.probe_inputs(w, n) for n in range(w.layers)]
    masked = dev(torch.tensor(w.masked_rows(), dtype=torch.int32).expand(w.batch, -1))
    desc = desc_of(w)
    need = ac.acache_probe_workspace_bytes(desc, w.batch, w.T, w.L, w.m)

    def buffers():
        qs = [dev(i["q"]) for i in inps]
        outs = [torch.empty_like(q) for q in qs]
        if feed:
            outs = qs[1:] + [outs[-1]]
        return qs, outs

    ka = [dev(i["k_aff"]) for i in inps]
    va = [dev(i["v_aff"]) for i in inps]
    kr = [dev(i["k_req"]) for i in inps]
    vr = [dev(i["v_req"]) for i in inps]
    ws = torch.empty(need, dtype=torch.uint8, device="cuda")
    s1 = torch.zeros((w.batch, w.L), dtype=torch.float32, device="cuda")
    st1 = status_tensor()
    q1, o1 = buffers()
    for n in range(w.layers):
        ac.acache_probe_scores(desc, w.batch, w.T, w.l, w.L, masked, w.m, q1[n], kr[n], vr[n], ka[n], va[n],
                               o1[n], s1, ws, dev_status=st1)
    s2 = torch.zeros_like(s1)
    st2 = status_tensor()
    q2, o2 = buffers()
    ac.acache_probe_scores_layers(desc, w.batch, w.T, w.l, w.L, masked, w.m, q2, kr, vr, ka, va, o2, s2,
                                  ws, dev_status=st2)
    torch.cuda.synchronize()
    assert st1.item() == 0 and st2.item() == 0
    assert torch.equal(s1, s2)
    for a, b in zip(o1, o2):
        assert torch.equal(a, b)
    if not feed:
        # again, without outputs, accumulating onto the first call's scores
        ac.acache_probe_scores_layers(desc, w.batch, w.T, w.l, w.L, masked, w.m, q2, kr, vr, ka, va, None,
                                      s2, ws, dev_status=st2)
        for n in range(w.layers):
            ac.acache_probe_scores(desc, w.batch, w.T, w.l, w.L, masked, w.m, q1[n], kr[n], vr[n], ka[n],
                                   va[n], None, s1, ws, dev_status=st1)
        torch.cuda.synchronize()
        assert st1.item() == 0 and st2.item() == 0
        assert torch.equal(s1, s2)
        s2 = s2 / 2
    if not feed:
        ref = None
        for n, inp in enumerate(inps):
            ref = oracle.probe_layer(inp["q"], inp["k_req"], inp["v_req"], inp["k_aff"], inp["v_aff"],
                                     T=w.T, l=w.l, masked_rows=w.masked_rows(), scale=w.scale,
                                     scores=None if ref is None else ref["scores"], want_out=n == w.layers - 1)
        assert_scores_close(s2.cpu().numpy(), ref["scores"], "4-layer scores")
        assert_out_close(o2[-1].float().cpu().numpy(), ref["out"], dtype, "last layer's probe output")


def test_probe_bad_masked_row_is_skipped_and_flagged():
    w = tiny(SMALL, batch=2, d=64, dtype="f32")
    inp = wl.probe_inputs(w, 0)
    masked = torch.tensor(w.masked_rows(), dtype=torch.int32).expand(w.batch, -1).clone()
    masked[1, 0] = w.P + 3
    ok_rows = masked[1, 1:].tolist()
    ref0 = oracle.probe_layer(inp["q"], inp["k_req"], inp["v_req"], inp["k_aff"], inp["v_aff"],
                              T=w.T, l=w.l, masked_rows=w.masked_rows(), scale=w.scale, want_out=False)
    ref1 = oracle.probe_layer(inp["q"][1:], inp["k_req"][1:], inp["v_req"][1:], inp["k_aff"],
                              inp["v_aff"], T=w.T, l=w.l, masked_rows=ok_rows, scale=w.scale,
                              want_out=False)
    scores = torch.zeros((w.batch, w.L), dtype=torch.float32, device="cuda")
    st = status_tensor()
    probe_layer_gpu(w, inp, scores, masked=masked, dev_status=st)
    torch.cuda.synchronize()
    assert st.item() == ac._lib.DEV_BAD_ROW
    assert_scores_close(scores[0].cpu().numpy()[None], ref0["scores"][:1], "request 0")
    assert_scores_close(scores[1].cpu().numpy()[None], ref1["scores"], "request 1")


# ------------------------------------------------------------------ slot attention
@pytest.mark.parametrize("dtype,d,heads", [("bf16", 128, (4, 2)), ("f32", 64, (2, 2)),
                                           ("bf16", 128, (7, 1)), ("bf16", 64, (2, 1))])
@pytest.mark.parametrize("n_q,T", [(300, 700), (1, 129), (129, 1)])
def test_slot_attention_parity(dtype, d, heads, n_q, T):
    hq, hkv = heads
    g = torch.Generator().manual_seed(n_q * 7 + T)
    B, num_slots = 2, 1500
    td = torch.float32 if dtype == "f32" else torch.bfloat16
    kc = torch.randn((num_slots, hkv, d), generator=g).to(td)
    vc = torch.randn((num_slots, hkv, d), generator=g).to(td)
    q = torch.randn((B, n_q, hq, d), generator=g).to(td)
    rs = torch.randint(0, num_slots, (B, T), generator=g, dtype=torch.int32)
    scale = d ** -0.5
    ref = oracle.slot_attention(q, rs, kc, vc, scale=scale)
    out = torch.empty((B, n_q, hq, d), dtype=td, device="cuda")
    st = status_tensor()
    ac.acache_slot_attention(ac.attn_desc(hq, hkv, d, scale, dtype), B, n_q, dev(q), T, dev(rs),
                             dev(kc), dev(vc), num_slots, out, dev_status=st)
    torch.cuda.synchronize()
    assert st.item() == 0
    assert_out_close(out.float().cpu().numpy(), ref, dtype, "slot attention")


# More 256-row query blocks of a (request, head) than SMs: the persistent kernel, each CTA
# working through several blocks, up to 20 key tiles; past that the fresh-CTA kernel in several
# waves.  (B, n_q, Hq, Hkv, T): two-tile blocks followed by one-tile blocks whose keys the two
# chains split; one key tile only (the one-tile blocks then have a single chain); the fewest
# key tiles a split takes (2, 3); four to five blocks per CTA; one-tile blocks only; 17 key
# tiles (still persistent); 21 key tiles (the fresh-CTA kernel); one-tile blocks of 22 key
# tiles (persistent: with one query tile per block there is no key-tile limit).
WAVE_CASES = [
    (4, 600, 32, 8, 700),
    (4, 300, 32, 32, 100),
    (4, 300, 32, 4, 200),
    (2, 1100, 64, 8, 300),
    (8, 100, 32, 8, 500),
    (2, 260, 64, 8, 2100),
    (2, 260, 64, 8, 2600),
    (6, 40, 32, 8, 2700),
]


@pytest.mark.parametrize("B,n_q,hq,hkv,T", WAVE_CASES)
def test_slot_attention_more_blocks_than_sms(B, n_q, hq, hkv, T):
    d, num_slots = 128, 3000
    g = torch.Generator().manual_seed(B * 100 + n_q + hq + T)
    kc = torch.randn((num_slots, hkv, d), generator=g).to(torch.bfloat16)
    vc = torch.randn((num_slots, hkv, d), generator=g).to(torch.bfloat16)
    q = (torch.randn((B, n_q, hq, d), generator=g) * 2).to(torch.bfloat16)
    rs = torch.randint(0, num_slots, (B, T), generator=g, dtype=torch.int32)
    ref = oracle.slot_attention(q, rs, kc, vc, scale=d ** -0.5)
    out = torch.full((B, n_q, hq, d), float("nan"), dtype=torch.bfloat16, device="cuda")
    st = status_tensor()
    ac.acache_slot_attention(ac.attn_desc(hq, hkv, d, d ** -0.5, "bf16"), B, n_q, dev(q), T, dev(rs),
                             dev(kc), dev(vc), num_slots, out, dev_status=st)
    torch.cuda.synchronize()
    assert st.item() == 0
    assert_out_close(out.float().cpu().numpy(), ref, "bf16", "slot attention, several waves")


# Few query rows per KV head (the block-decode step): (B, n_q, Hq, Hkv, T).  The cases span
# 4 / 2 / 1 replicas of the packed rows, key ranges split over clusters of 1, 2 and 4 CTAs,
# GQA groups packed into one or two row blocks, and ragged last key tiles.
DECODE_CASES = [
    (2, 32, 4, 4, 1408),     # MHA block of 32: four replicas, clusters of 4
    (1, 32, 2, 2, 4480),     # two units only: clusters of 4, 35 key tiles
    (3, 5, 4, 4, 37),        # one ragged key tile
    (2, 32, 8, 4, 300),      # g = 2: 64 packed rows, two replicas
    (2, 32, 28, 4, 2624),    # g = 7: row blocks of 18 and 14 queries (126 + 98 rows)
    (2, 100, 4, 4, 700),     # 100 rows: no replicas
    (1, 1, 1, 1, 1),         # one query, one key
    (2, 64, 4, 2, 129),      # g = 2, 128 packed rows, one key past a tile
    (4, 32, 32, 32, 1408),   # the LLaDA-8B head geometry at T = 1408
]


@pytest.mark.parametrize("B,n_q,hq,hkv,T", DECODE_CASES)
def test_decode_slot_attention_parity(B, n_q, hq, hkv, T):
    d, num_slots = 128, 5000
    g = torch.Generator().manual_seed(B * 1000 + n_q * 10 + hq + T)
    kc = torch.randn((num_slots, hkv, d), generator=g).to(torch.bfloat16)
    vc = torch.randn((num_slots, hkv, d), generator=g).to(torch.bfloat16)
    q = (torch.randn((B, n_q, hq, d), generator=g) * 2).to(torch.bfloat16)
    rs = torch.randint(0, num_slots, (B, T), generator=g, dtype=torch.int32)
    scale = d ** -0.5
    ref = oracle.slot_attention(q, rs, kc, vc, scale=scale)
    out = torch.full((B, n_q, hq, d), float("nan"), dtype=torch.bfloat16, device="cuda")
    st = status_tensor()
    ac.acache_slot_attention(ac.attn_desc(hq, hkv, d, scale, "bf16"), B, n_q, dev(q), T, dev(rs),
                             dev(kc), dev(vc), num_slots, out, dev_status=st)
    torch.cuda.synchronize()
    assert st.item() == 0
    assert_out_close(out.float().cpu().numpy(), ref, "bf16", "decode slot attention")


def test_decode_slot_attention_peaked_rows():
    """Rows whose maximum moves late (forces the in-TMEM rescale) and rows dominated by one
    key: the replicas' and cluster ranks' partial maxima differ by large amounts."""
    B, n_q, hq, hkv, T, d, num_slots = 1, 32, 4, 4, 2000, 128, 2500
    g = torch.Generator().manual_seed(5)
    kc = torch.randn((num_slots, hkv, d), generator=g)
    vc = torch.randn((num_slots, hkv, d), generator=g)
    q = torch.randn((B, n_q, hq, d), generator=g)
    rs = torch.arange(T, dtype=torch.int32)[None].repeat(B, 1)
    # key 1900 (last cluster rank, late tile) aligned with query 3; key 40 with query 7
    kc[1900] = q[0, 3].reshape(hq, d)[:hkv] * 3
    kc[40] = q[0, 7].reshape(hq, d)[:hkv] * 3
    kc, vc, q = kc.to(torch.bfloat16), vc.to(torch.bfloat16), q.to(torch.bfloat16)
    ref = oracle.slot_attention(q, rs, kc, vc, scale=d ** -0.5)
    out = torch.empty((B, n_q, hq, d), dtype=torch.bfloat16, device="cuda")
    st = status_tensor()
    ac.acache_slot_attention(ac.attn_desc(hq, hkv, d, d ** -0.5, "bf16"), B, n_q, dev(q), T, dev(rs),
                             dev(kc), dev(vc), num_slots, out, dev_status=st)
    torch.cuda.synchronize()
    assert st.item() == 0
    assert_out_close(out.float().cpu().numpy(), ref, "bf16", "peaked decode rows")


def test_slot_attention_peaked_rows_many_queries():
    """The 128-row tile kernel with rows whose maximum jumps late: the lazy rescale of O in TMEM
    runs, and in the one-tile last query block (rows 256-299, keys split between two chains)
    the two halves' maxima differ by tens of powers of two when they are merged."""
    B, n_q, hq, hkv, T, d, num_slots = 1, 300, 2, 2, 2000, 128, 2500
    g = torch.Generator().manual_seed(17)
    kc = torch.randn((num_slots, hkv, d), generator=g)
    vc = torch.randn((num_slots, hkv, d), generator=g)
    q = torch.randn((B, n_q, hq, d), generator=g)
    rs = torch.arange(T, dtype=torch.int32)[None].repeat(B, 1)
    kc[1900] = q[0, 3] * 3        # two-tile block, a late key tile
    kc[1500] = q[0, 290] * 3      # last block: in the second chain's half of the keys
    kc[100] = q[0, 291] * 3       # last block: in the first chain's half
    kc[130] = q[0, 200] * 2
    kc[1990] = q[0, 200] * 3      # a second, larger jump in the same row
    kc, vc, q = kc.to(torch.bfloat16), vc.to(torch.bfloat16), q.to(torch.bfloat16)
    ref = oracle.slot_attention(q, rs, kc, vc, scale=d ** -0.5)
    out = torch.empty((B, n_q, hq, d), dtype=torch.bfloat16, device="cuda")
    st = status_tensor()
    ac.acache_slot_attention(ac.attn_desc(hq, hkv, d, d ** -0.5, "bf16"), B, n_q, dev(q), T, dev(rs),
                             dev(kc), dev(vc), num_slots, out, dev_status=st)
    torch.cuda.synchronize()
    assert st.item() == 0
    assert_out_close(out.float().cpu().numpy(), ref, "bf16", "peaked rows")


@pytest.mark.parametrize("drop", [False, True])
def test_slot_attention_consecutive_slot_tiles(drop):
    """Read-slot tiles whose 128 slots are consecutive load as tiled boxes, others gather: tiles
    consecutive from slot 100, from slot 0, and ending on the pool's last slot; one with a single
    key out of order; a random one; a ragged last tile that is consecutive; with DropNA, a
    consecutive tile with one discarded key."""
    B, n_q, hq, hkv, T, d, num_slots = 2, 300, 2, 2, 700, 128, 1200
    g = torch.Generator().manual_seed(23 + drop)
    kc = torch.randn((num_slots, hkv, d), generator=g).to(torch.bfloat16)
    vc = torch.randn((num_slots, hkv, d), generator=g).to(torch.bfloat16)
    q = torch.randn((B, n_q, hq, d), generator=g).to(torch.bfloat16)
    rs = torch.randint(0, num_slots, (B, T), generator=g, dtype=torch.int32)
    ar = torch.arange(128, dtype=torch.int32)
    rs[:, 0:128] = 100 + ar                          # consecutive
    rs[:, 128:256] = 400 + ar
    rs[:, 200], rs[:, 201] = rs[:, 201].clone(), rs[:, 200].clone()   # one pair swapped: gathers
    rs[:, 256:384] = num_slots - 128 + ar            # ends on the last slot
    rs[1, 512:640] = ar                              # request 1: consecutive from 0
    rs[:, 640:700] = 700 + ar[:60]                   # ragged last tile, consecutive
    if drop:
        rs[0, 300] = -1                              # a discarded key inside a consecutive tile
    ref = oracle.slot_attention(q, rs, kc, vc, scale=d ** -0.5, drop_none=drop)
    out = torch.empty((B, n_q, hq, d), dtype=torch.bfloat16, device="cuda")
    st = status_tensor()
    desc = ac.attn_desc(hq, hkv, d, d ** -0.5, "bf16")
    fn = ac.acache_slot_attention_dropna if drop else ac.acache_slot_attention
    fn(desc, B, n_q, dev(q), T, dev(rs), dev(kc), dev(vc), num_slots, out, dev_status=st)
    torch.cuda.synchronize()
    assert st.item() == 0
    assert_out_close(out.float().cpu().numpy(), ref, "bf16", "consecutive-slot tiles")


def test_slot_attention_bad_slot_reads_zero_row():
    B, n_q, T, hq, hkv, d, num_slots = 1, 40, 150, 2, 2, 128, 300
    g = torch.Generator().manual_seed(11)
    kc = torch.randn((num_slots, hkv, d), generator=g).to(torch.bfloat16)
    vc = torch.randn((num_slots, hkv, d), generator=g).to(torch.bfloat16)
    q = torch.randn((B, n_q, hq, d), generator=g).to(torch.bfloat16)
    rs = torch.randint(0, num_slots, (B, T), generator=g, dtype=torch.int32)
    rs[0, 17] = num_slots + 100
    # the oracle sees an extra all-zero slot in place of the bad one
    kz = torch.cat([kc, torch.zeros(1, hkv, d, dtype=kc.dtype)])
    vz = torch.cat([vc, torch.zeros(1, hkv, d, dtype=vc.dtype)])
    rz = rs.clone()
    rz[0, 17] = num_slots
    ref = oracle.slot_attention(q, rz, kz, vz, scale=d ** -0.5)
    out = torch.empty((B, n_q, hq, d), dtype=torch.bfloat16, device="cuda")
    st = status_tensor()
    ac.acache_slot_attention(ac.attn_desc(hq, hkv, d, d ** -0.5, "bf16"), B, n_q, dev(q), T,
                             dev(rs), dev(kc), dev(vc), num_slots, out, dev_status=st)
    torch.cuda.synchronize()
    assert st.item() == ac._lib.DEV_BAD_SLOT
    assert_out_close(out.float().cpu().numpy(), ref, "bf16", "bad-slot attention")


# ------------------------------------------------------------------ the tiny workload end to end
def test_tiny_prefix_f32_pipeline():
    """Probe -> scores -> Top-K(26) -> maps -> write 122 rows -> slot attention (122 x 224).

    The oracle runs its own chain from the generator's inputs; each GPU stage is compared
    with the oracle's stage.  No GPU result is fed to the oracle."""
    w = wl.TINY_PREFIX_F32
    lay = wl.slot_layout(w)
    inp = wl.probe_inputs(w, 0)
    rec = wl.recompute_inputs(w, 0)
    # ---- oracle chain
    ref = oracle.probe_layer(inp["q"], inp["k_req"], inp["v_req"], inp["k_aff"], inp["v_aff"],
                             T=w.T, l=w.l, masked_rows=w.masked_rows(), scale=w.scale)
    a_ref = oracle.topk_anchors(ref["scores"], w.K)
    wp_ref, rs_ref = oracle.build_slot_maps(a_ref, lay.shared_slot, lay.private_slots, T=w.T, l=w.l, L=w.L)
    kc0 = torch.zeros((lay.num_slots, w.hkv, w.d))
    vc0 = torch.zeros_like(kc0)
    kb, vb, _ = oracle.write_slots(lay.shared_slot[None], inp["k_aff"][None], inp["v_aff"][None],
                                   kc0, vc0, private_begin=0)
    kc0 = torch.from_numpy(kb).view(torch.float32).view(kc0.shape)
    vc0 = torch.from_numpy(vb).view(torch.float32).view(vc0.shape)
    kb, vb, flags = oracle.write_slots(lay.private_slots, rec["k_new"], rec["v_new"], kc0, vc0,
                                       private_begin=lay.private_begin)
    assert flags == 0
    kc_ref = torch.from_numpy(kb).view(torch.float32).view(kc0.shape)
    vc_ref = torch.from_numpy(vb).view(torch.float32).view(vc0.shape)
    o_ref = oracle.slot_attention(rec["q_r"], rs_ref, kc_ref, vc_ref, scale=w.scale)
    # ---- GPU chain
    scores = torch.zeros((w.batch, w.L), dtype=torch.float32, device="cuda")
    o = probe_layer_gpu(w, inp, scores)
    anchors = torch.empty((w.batch, w.K), dtype=torch.int32, device="cuda")
    ac.acache_topk_anchors(scores, w.batch, w.L, w.K, anchors)
    wp = torch.empty((w.batch, w.R), dtype=torch.int32, device="cuda")
    rs = torch.empty((w.batch, w.T), dtype=torch.int32, device="cuda")
    ac.acache_build_slot_maps(w.batch, w.T, w.l, w.L, w.K, anchors, dev(lay.shared_slot),
                              dev(lay.private_slots), wp, rs)
    kc = torch.zeros((lay.num_slots, w.hkv, w.d), dtype=torch.float32, device="cuda")
    vc = torch.zeros_like(kc)
    register_shared(w, lay, inp["k_aff"], inp["v_aff"], kc, vc)
    ac.acache_write_slots(desc_of(w), w.batch, w.R, dev(lay.private_slots), dev(rec["k_new"]),
                          dev(rec["v_new"]), kc, vc, lay.num_slots, lay.private_begin)
    out = torch.empty((w.batch, w.R, w.hq, w.d), dtype=torch.float32, device="cuda")
    ac.acache_slot_attention(desc_of(w), w.batch, w.R, dev(rec["q_r"]), w.T, rs, kc, vc,
                             lay.num_slots, out)
    torch.cuda.synchronize()
    # ---- stage by stage
    assert_out_close(o.cpu().numpy(), ref["out"], "f32", "probe output")
    assert_scores_close(scores.cpu().numpy(), ref["scores"], "scores")
    assert_anchors_match(anchors.cpu().numpy(), ref["scores"], w.K, "anchors")
    # this seeded case has no near-tie at the K-th score, so the sets are identical and
    # every later stage is compared bit for bit / within tolerance
    assert np.array_equal(anchors.cpu().numpy(), a_ref)
    assert np.array_equal(wp.cpu().numpy(), wp_ref) and np.array_equal(rs.cpu().numpy(), rs_ref)
    assert torch.equal(kc.cpu(), kc_ref) and torch.equal(vc.cpu(), vc_ref)
    assert_out_close(out.cpu().numpy(), o_ref, "f32", "slot attention")


@pytest.mark.parametrize("case", ["no_masked_rows", "no_affix", "one_layer"])
def test_probe_layers_edge_cases(case):
    """The chained probe of several layers at its edges: no masked row (every score stays 0), no
    affix (only the request's own keys: no mass, no head sum; the forwards chain directly) and a
    single layer -- each equal to the per-layer calls bit for bit and to the oracle."""
    segs = {"no_masked_rows": [(wl.SEG_AFFIX, 300), (wl.SEG_REQ, 200)],
            "no_affix": [(wl.SEG_REQ, 150), (wl.SEG_MASK, 150)],
            "one_layer": [(wl.SEG_REQ, 60), (wl.SEG_AFFIX, 300), (wl.SEG_MASK, 140)]}[case]
    w = tiny(segs, batch=2).replace(layers=1 if case == "one_layer" else 3)
    inps = [wl.probe_inputs(w, n) for n in range(w.layers)]
    desc = desc_of(w)
    masked = dev(torch.tensor(w.masked_rows(), dtype=torch.int32).reshape(1, -1).expand(w.batch, -1).contiguous())
    ws = torch.empty(max(1, ac.acache_probe_workspace_bytes(desc, w.batch, w.T, w.L, w.m)), dtype=torch.uint8,
                     device="cuda")
    lists = [[dev(i[k]) if i[k].numel() else None for i in inps] for k in ("q", "k_req", "v_req", "k_aff", "v_aff")]
    s1 = torch.zeros((w.batch, max(w.L, 1)), dtype=torch.float32, device="cuda")
    s2 = torch.zeros_like(s1)
    o1 = [torch.empty_like(q) for q in lists[0]]
    o2 = [torch.empty_like(q) for q in lists[0]]
    st = status_tensor()
    sc1 = s1 if w.L else None
    sc2 = s2 if w.L else None
    for n in range(w.layers):
        ac.acache_probe_scores(desc, w.batch, w.T, w.l, w.L, masked, w.m, lists[0][n], lists[1][n], lists[2][n],
                               lists[3][n], lists[4][n], o1[n], sc1, ws, dev_status=st)
    ac.acache_probe_scores_layers(desc, w.batch, w.T, w.l, w.L, masked, w.m,
                                  *[lst if any(x is not None for x in lst) else None for lst in lists],
                                  o2, sc2, ws, dev_status=st)
    torch.cuda.synchronize()
    assert st.item() == 0
    assert torch.equal(s1, s2)
    for a, b in zip(o1, o2):
        assert torch.equal(a, b)
    ref = None
    for n, inp in enumerate(inps):
        ref = oracle.probe_layer(inp["q"], inp["k_req"], inp["v_req"], inp["k_aff"], inp["v_aff"], T=w.T, l=w.l,
                                 masked_rows=w.masked_rows(), scale=w.scale,
                                 scores=None if ref is None else ref["scores"])
        assert_out_close(o2[n].float().cpu().numpy(), ref["out"], "bf16", f"{case} layer {n} output")
    if w.L:
        if w.m == 0:
            assert not s2.any()
        else:
            assert_scores_close(s2.cpu().numpy(), ref["scores"], f"{case} scores")
