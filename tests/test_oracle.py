"""Pins of the CPU oracle against what the page and the mathematics fix.

Source: "Affix Cache for Diffusion Large Language Models" (arXiv 2608.26140), Sec. 3.2
(Eq. 4-6), Sec. 4.1-4.3 and App. C.1.  The page prints no worked numeric example, so the
oracle is pinned by library routines (torch float64 attention and softmax, a stable sort,
torch index ops), closed forms, invariants and the semantic end points of the anchor ratio
(Sec. 5.1: ratio 0 is direct reuse, ratio 1 is full recomputation).
"""
import math

import numpy as np
import pytest
import torch

import oracle
from affix_kv_cache_gb300 import workloads as wl


def tiny(segments, hq=2, hkv=2, d=16, batch=2, ratio=200, dtype="f32", **kw):
    return wl.Workload(name="tiny", dtype=dtype, layers=1, hq=hq, hkv=hkv, d=d, batch=batch,
                       segments=tuple(segments), ratio_permille=ratio, recompute_points=1, **kw)


LAYOUTS = {
    "prefix": [(wl.SEG_AFFIX, 9), (wl.SEG_REQ, 4), (wl.SEG_MASK, 6)],
    "infix": [(wl.SEG_REQ, 3), (wl.SEG_AFFIX, 8), (wl.SEG_REQ, 2), (wl.SEG_MASK, 5)],
    "suffix": [(wl.SEG_REQ, 3), (wl.SEG_MASK, 6), (wl.SEG_AFFIX, 10)],
}


def logical_kv(w, inp, b):
    """Logical key/value rows of request b, built here from the layout (test-side)."""
    ks, vs = [], []
    pr = 0
    for t in range(w.T):
        if w.l <= t < w.l + w.L:
            ks.append(inp["k_aff"][t - w.l])
            vs.append(inp["v_aff"][t - w.l])
        else:
            ks.append(inp["k_req"][b, pr])
            vs.append(inp["v_req"][b, pr])
            pr += 1
    return torch.stack(ks).double(), torch.stack(vs).double()   # [T][Hkv][d]


def sdpa64(q, k, v, scale):
    """torch float64 attention; q [n][Hq][d], k/v [T][Hkv][d] (KV heads repeated)."""
    g = q.shape[1] // k.shape[1]
    kk = k.double().repeat_interleave(g, dim=1).permute(1, 0, 2)
    vv = v.double().repeat_interleave(g, dim=1).permute(1, 0, 2)
    o = torch.nn.functional.scaled_dot_product_attention(
        q.double().permute(1, 0, 2).unsqueeze(0), kk.unsqueeze(0), vv.unsqueeze(0), scale=scale)
    return o.squeeze(0).permute(1, 0, 2)


# ------------------------------------------------------------------------ probe
@pytest.mark.parametrize("layout", list(LAYOUTS))
@pytest.mark.parametrize("heads", [(2, 2), (4, 2), (6, 1)])
@pytest.mark.parametrize("dtype", ["f32", "bf16"])
def test_probe_output_matches_torch_attention(layout, heads, dtype):
    w = tiny(LAYOUTS[layout], hq=heads[0], hkv=heads[1], dtype=dtype)
    inp = wl.probe_inputs(w, 0)
    r = oracle.probe_layer(inp["q"], inp["k_req"], inp["v_req"], inp["k_aff"], inp["v_aff"],
                           T=w.T, l=w.l, masked_rows=w.masked_rows(), scale=w.scale)
    for b in range(w.batch):
        k, v = logical_kv(w, inp, b)
        ref = sdpa64(inp["q"][b], k, v, w.scale).numpy()
        np.testing.assert_allclose(r["out"][b], ref, rtol=0, atol=1e-12)


@pytest.mark.parametrize("layout", list(LAYOUTS))
def test_probe_scores_equal_masked_affix_probability_mass(layout):
    # Eq. 4-5 against torch float64 softmax of the full logical row (reading: the row
    # softmax runs over affix keys and the request's own keys), summed over heads and the
    # initially masked rows only.
    w = tiny(LAYOUTS[layout], hq=4, hkv=2)
    inp = wl.probe_inputs(w, 0)
    r = oracle.probe_layer(inp["q"], inp["k_req"], inp["v_req"], inp["k_aff"], inp["v_aff"],
                           T=w.T, l=w.l, masked_rows=w.masked_rows(), scale=w.scale)
    g = w.hq // w.hkv
    for b in range(w.batch):
        k, _ = logical_kv(w, inp, b)
        q = inp["q"][b].double()                                   # [P][Hq][d]
        kk = k.repeat_interleave(g, dim=1)                          # [T][Hq][d]
        logits = torch.einsum("phc,thc->hpt", q, kk) * w.scale
        prob = torch.softmax(logits, dim=-1)                        # [Hq][P][T]
        rows = torch.tensor(w.masked_rows())
        expect = prob[:, rows, w.l:w.l + w.L].sum(dim=(0, 1)).numpy()
        np.testing.assert_allclose(r["scores"][b], expect, rtol=1e-12, atol=1e-15)


def test_probe_rows_sum_to_one_via_constant_values():
    # invariant (i): with every value row equal to 1, the output equals the row sum of the
    # probabilities, which must be 1 for every probe row and head.
    w = tiny(LAYOUTS["infix"], hq=4, hkv=2)
    inp = wl.probe_inputs(w, 0)
    r = oracle.probe_layer(inp["q"], inp["k_req"], torch.ones_like(inp["v_req"]), inp["k_aff"],
                           torch.ones_like(inp["v_aff"]), T=w.T, l=w.l,
                           masked_rows=w.masked_rows(), scale=w.scale, want_stats=True)
    np.testing.assert_allclose(r["out"], 1.0, rtol=0, atol=1e-12)
    # the stats are the row max and the sum of exp(logit - max): at least one term is 1
    assert np.all(r["row_sum"] >= 1.0) and np.all(r["row_sum"] <= w.T)


@pytest.mark.parametrize("layout", list(LAYOUTS))
def test_probe_scores_through_indicator_values(layout):
    # invariant (v) column by column: with v_aff[j] = e_j and v_req = 0, the output of row k
    # is the vector (a_{l+j,k})_j, so the masked-row sum of outputs over heads is s_j.
    w = tiny(LAYOUTS[layout], hq=4, hkv=2, d=16)
    assert w.L <= w.d
    inp = wl.probe_inputs(w, 0)
    v_aff = torch.zeros_like(inp["v_aff"])
    for j in range(w.L):
        v_aff[j, :, j] = 1.0
    r = oracle.probe_layer(inp["q"], inp["k_req"], torch.zeros_like(inp["v_req"]), inp["k_aff"],
                           v_aff, T=w.T, l=w.l, masked_rows=w.masked_rows(), scale=w.scale)
    rows = w.masked_rows()
    via_out = r["out"][:, rows, :, : w.L].sum(axis=(1, 2))         # [B][L]
    np.testing.assert_allclose(r["scores"], via_out, rtol=1e-12, atol=1e-15)
    # total masked mass on the affix is at most heads * masked rows, strictly below it
    # because the request's own keys also take mass (full-row normaliser)
    assert np.all(r["scores"].sum(axis=1) < w.hq * w.m)


def test_probe_equal_keys_closed_form():
    # all T keys equal: every probability is 1/T, the output is the mean value row, and
    # s_j = layers * Hq * m / T for every affix offset.
    w = tiny(LAYOUTS["suffix"], hq=2, hkv=1, d=8)
    inp = wl.probe_inputs(w, 0)
    key = torch.randn(w.d)
    k_aff = key.expand_as(inp["k_aff"]).contiguous()
    k_req = key.expand_as(inp["k_req"]).contiguous()
    r = oracle.probe_layer(inp["q"], k_req, inp["v_req"], k_aff, inp["v_aff"], T=w.T, l=w.l,
                           masked_rows=w.masked_rows(), scale=w.scale)
    np.testing.assert_allclose(r["scores"], w.hq * w.m / w.T, rtol=1e-12)
    for b in range(w.batch):
        _, v = logical_kv(w, inp, b)
        meanv = v.mean(dim=0).numpy()                              # [Hkv][d]
        np.testing.assert_allclose(r["out"][b], np.broadcast_to(meanv[None, :, :], r["out"][b].shape),
                                   atol=1e-12)


def test_probe_dominant_key_takes_all_mass():
    # one affix key aligned with every masked query at a huge logit takes essentially all the
    # mass: s_j0 -> Hq * m, every other s_j -> 0.
    w = tiny(LAYOUTS["prefix"], hq=2, hkv=2, d=8, batch=1)
    inp = wl.probe_inputs(w, 0)
    q = torch.zeros_like(inp["q"])
    q[..., 0] = 1.0
    k_aff = torch.zeros_like(inp["k_aff"])
    j0 = 5
    k_aff[j0, :, 0] = 400.0                                        # logit 400/sqrt(8) vs 0
    r = oracle.probe_layer(q, torch.zeros_like(inp["k_req"]), inp["v_req"], k_aff, inp["v_aff"],
                           T=w.T, l=w.l, masked_rows=w.masked_rows(), scale=w.scale)
    expect = np.zeros(w.L)
    expect[j0] = w.hq * w.m
    np.testing.assert_allclose(r["scores"][0], expect, rtol=1e-12, atol=1e-12)


def test_probe_scores_accumulate_over_layers_in_call_order():
    w = tiny(LAYOUTS["infix"], hq=2, hkv=2).replace(layers=3)
    total = None
    parts = []
    for n in range(w.layers):
        inp = wl.probe_inputs(w, n)
        r = oracle.probe_layer(inp["q"], inp["k_req"], inp["v_req"], inp["k_aff"], inp["v_aff"],
                               T=w.T, l=w.l, masked_rows=w.masked_rows(), scale=w.scale,
                               scores=total, want_out=False)
        total = r["scores"]
        parts.append(oracle.probe_layer(inp["q"], inp["k_req"], inp["v_req"], inp["k_aff"],
                                        inp["v_aff"], T=w.T, l=w.l, masked_rows=w.masked_rows(),
                                        scale=w.scale, want_out=False)["scores"])
    np.testing.assert_allclose(total, parts[0] + parts[1] + parts[2], rtol=1e-14)


def test_probe_affix_only_normaliser_flag():
    # the literal reading of Eq. 4 normalises over affix keys only: every masked row then
    # spends exactly one unit of mass per head on the affix.
    w = tiny(LAYOUTS["infix"], hq=4, hkv=2)
    inp = wl.probe_inputs(w, 0)
    r = oracle.probe_layer(inp["q"], inp["k_req"], inp["v_req"], inp["k_aff"], inp["v_aff"],
                           T=w.T, l=w.l, masked_rows=w.masked_rows(), scale=w.scale,
                           affix_only_norm=True, want_out=False)
    np.testing.assert_allclose(r["scores"].sum(axis=1), w.hq * w.m, rtol=1e-12)


def test_probe_row_subset_matches_full():
    w = tiny(LAYOUTS["suffix"], hq=2, hkv=2)
    inp = wl.probe_inputs(w, 0)
    full = oracle.probe_layer(inp["q"], inp["k_req"], inp["v_req"], inp["k_aff"], inp["v_aff"],
                              T=w.T, l=w.l, masked_rows=w.masked_rows(), scale=w.scale)
    rows = [1, 4, 7]
    sub = oracle.probe_layer(inp["q"], inp["k_req"], inp["v_req"], inp["k_aff"], inp["v_aff"],
                             T=w.T, l=w.l, masked_rows=w.masked_rows(), scale=w.scale, rows=rows)
    np.testing.assert_array_equal(sub["out"][:, rows], full["out"][:, rows])
    # only masked rows among the subset contribute to the scores
    only = oracle.probe_layer(inp["q"], inp["k_req"], inp["v_req"], inp["k_aff"], inp["v_aff"],
                              T=w.T, l=w.l, masked_rows=w.masked_rows(), scale=w.scale,
                              rows=w.masked_rows())
    np.testing.assert_array_equal(only["scores"], full["scores"])


def test_probe_rejects_bad_arguments():
    w = tiny(LAYOUTS["prefix"])
    inp = wl.probe_inputs(w, 0)
    with pytest.raises(ValueError):
        oracle.probe_layer(inp["q"], inp["k_req"], inp["v_req"], inp["k_aff"], inp["v_aff"],
                           T=w.T, l=w.l, masked_rows=[w.P], scale=w.scale)


# ------------------------------------------------------------------------ Top-K
def _stable_topk(s, K):
    order = np.argsort(-s, kind="stable")       # ties keep ascending index
    return np.sort(order[:K])


@pytest.mark.parametrize("L,K", [(1, 0), (1, 1), (17, 5), (64, 13), (300, 61), (300, 300)])
def test_topk_matches_stable_sort(L, K):
    rng = np.random.default_rng(L * 1000 + K)
    s = rng.standard_normal((3, L)) ** 2
    s[1] = np.round(s[1] * 4) / 4                     # many exact ties
    a = oracle.topk_anchors(s, K)
    for b in range(3):
        np.testing.assert_array_equal(a[b], _stable_topk(s[b], K))


def test_topk_special_cases():
    s = np.full((1, 40), 0.25)
    np.testing.assert_array_equal(oracle.topk_anchors(s, 7)[0], np.arange(7))
    assert oracle.topk_anchors(s, 0).shape == (1, 0)
    np.testing.assert_array_equal(oracle.topk_anchors(s, 40)[0], np.arange(40))
    s = np.arange(40, dtype=np.float64)[None, ::-1].copy()
    np.testing.assert_array_equal(oracle.topk_anchors(s, 3)[0], [0, 1, 2])
    s[0, 39] = np.nan
    with pytest.raises(ValueError):
        oracle.topk_anchors(s, 3)


# ------------------------------------------------------------------------ maps
def _maps_by_definition(anchors, shared, private, T, l, L):
    B, K = anchors.shape
    R = K + T - L
    wp = np.zeros((B, R), np.int64)
    rs = np.zeros((B, T), np.int64)
    for b in range(B):
        recomputed = [t for t in range(T) if not (l <= t < l + L) or (t - l) in set(anchors[b])]
        assert len(recomputed) == R
        for i, t in enumerate(recomputed):
            wp[b, i] = t
            rs[b, t] = private[b, i]
        for t in range(l, l + L):
            if (t - l) not in set(anchors[b]):
                rs[b, t] = shared[t - l]
    return wp, rs


@pytest.mark.parametrize("layout", list(LAYOUTS))
@pytest.mark.parametrize("ratio", [0, 200, 500, 1000])
def test_slot_maps(layout, ratio):
    w = tiny(LAYOUTS[layout], ratio=ratio, batch=3, page=4)
    lay = wl.slot_layout(w)
    rng = np.random.default_rng(ratio)
    anchors = np.stack([np.sort(rng.choice(w.L, w.K, replace=False)) for _ in range(w.batch)]).astype(np.int32)
    wp, rs = oracle.build_slot_maps(anchors, lay.shared_slot, lay.private_slots, T=w.T, l=w.l, L=w.L)
    ewp, ers = _maps_by_definition(anchors, lay.shared_slot.numpy(), lay.private_slots.numpy(), w.T, w.l, w.L)
    np.testing.assert_array_equal(wp, ewp)
    np.testing.assert_array_equal(rs, ers)
    for b in range(w.batch):
        priv = rs[b][rs[b] >= lay.private_begin]
        assert len(priv) == w.R and len(set(priv.tolist())) == w.R       # injective on private
        shared_pos = [t for t in range(w.l, w.l + w.L) if (t - w.l) not in set(anchors[b])]
        assert all(rs[b, t] == lay.shared_slot[t - w.l] for t in shared_pos)
        assert np.all(np.diff(wp[b]) > 0)


def test_slot_maps_reject_unsorted_anchors():
    w = tiny(LAYOUTS["prefix"], ratio=500, batch=1)
    lay = wl.slot_layout(w)
    bad = np.array([[3, 1, 4, 5, 7]], np.int32)[:, : w.K]
    with pytest.raises(ValueError):
        oracle.build_slot_maps(bad, lay.shared_slot, lay.private_slots, T=w.T, l=w.l, L=w.L)


# ------------------------------------------------------------------------ write / gather
@pytest.mark.parametrize("dtype", ["f32", "bf16"])
def test_write_and_gather_match_index_ops(dtype):
    w = tiny(LAYOUTS["infix"], ratio=500, batch=3, page=4, dtype=dtype, hkv=2, d=8)
    lay = wl.slot_layout(w)
    rec = wl.recompute_inputs(w, 0)
    g = torch.Generator().manual_seed(1)
    kc = torch.randn((lay.num_slots, w.hkv, w.d), generator=g).to(w.torch_dtype)
    vc = torch.randn((lay.num_slots, w.hkv, w.d), generator=g).to(w.torch_dtype)
    kb, vb, flags = oracle.write_slots(lay.private_slots, rec["k_new"], rec["v_new"], kc, vc,
                                       private_begin=lay.private_begin)
    assert flags == 0
    ek, ev = kc.clone(), vc.clone()
    idx = lay.private_slots.reshape(-1).long()
    ek.index_copy_(0, idx, rec["k_new"].reshape(-1, w.hkv, w.d))
    ev.index_copy_(0, idx, rec["v_new"].reshape(-1, w.hkv, w.d))
    np.testing.assert_array_equal(kb, ek.view(torch.uint8).reshape(-1).numpy())
    np.testing.assert_array_equal(vb, ev.view(torch.uint8).reshape(-1).numpy())
    # gather through a read map equals index_select
    rs = torch.randint(0, lay.num_slots, (w.batch, w.T), generator=g, dtype=torch.int32)
    ko, vo, f2 = oracle.gather_slots(rs, ek, ev)
    assert f2 == 0
    np.testing.assert_array_equal(ko, ek.index_select(0, rs.reshape(-1).long()).view(torch.uint8).reshape(-1).numpy())
    np.testing.assert_array_equal(vo, ev.index_select(0, rs.reshape(-1).long()).view(torch.uint8).reshape(-1).numpy())


def test_write_flags_bad_slots():
    w = tiny(LAYOUTS["prefix"], ratio=200, batch=1, hkv=1, d=4)
    lay = wl.slot_layout(w)
    rec = wl.recompute_inputs(w, 0)
    kc = torch.zeros((lay.num_slots, 1, 4))
    ws = lay.private_slots.clone()
    ws[0, 0] = 0                       # inside the shared region
    ws[0, 1] = lay.num_slots           # out of range
    kb, _, flags = oracle.write_slots(ws, rec["k_new"], rec["v_new"], kc, kc,
                                      private_begin=lay.private_begin)
    assert flags == 3
    # the shared region is untouched
    assert np.all(kb.view(np.float32)[: lay.private_begin * 4] == 0)


# ------------------------------------------------------------------------ slot attention
@pytest.mark.parametrize("heads", [(2, 2), (6, 2)])
@pytest.mark.parametrize("dtype", ["f32", "bf16"])
def test_slot_attention_equals_dense_attention_over_gathered_kv(heads, dtype):
    # invariant (iv): attention through the read map equals plain attention over the
    # gathered logical KV (two separate oracle paths), and both equal torch float64 SDPA.
    w = tiny(LAYOUTS["infix"], hq=heads[0], hkv=heads[1], batch=2, dtype=dtype, page=4)
    lay = wl.slot_layout(w)
    g = torch.Generator().manual_seed(7)
    kc = torch.randn((lay.num_slots, w.hkv, w.d), generator=g).to(w.torch_dtype)
    vc = torch.randn((lay.num_slots, w.hkv, w.d), generator=g).to(w.torch_dtype)
    rs = torch.randint(0, lay.num_slots, (w.batch, w.T), generator=g, dtype=torch.int32)
    q = torch.randn((w.batch, 11, w.hq, w.d), generator=g).to(w.torch_dtype)
    o = oracle.slot_attention(q, rs, kc, vc, scale=w.scale)
    kl = kc.index_select(0, rs.reshape(-1).long()).view(w.batch, w.T, w.hkv, w.d)
    vl = vc.index_select(0, rs.reshape(-1).long()).view(w.batch, w.T, w.hkv, w.d)
    od = oracle.dense_attention(q, kl, vl, scale=w.scale)
    np.testing.assert_allclose(o, od, rtol=0, atol=1e-12)
    for b in range(w.batch):
        ref = sdpa64(q[b], kl[b], vl[b], w.scale).numpy()
        np.testing.assert_allclose(o[b], ref, rtol=0, atol=1e-12)
    sub = oracle.slot_attention(q, rs, kc, vc, scale=w.scale, rows=[0, 5, 10])
    np.testing.assert_array_equal(sub[:, [0, 5, 10]], o[:, [0, 5, 10]])


def test_slot_attention_rejects_out_of_range_slot():
    q = torch.randn(1, 2, 1, 4)
    kc = torch.randn(5, 1, 4)
    with pytest.raises(ValueError):
        oracle.slot_attention(q, torch.tensor([[0, 5]], dtype=torch.int32), kc, kc, scale=0.5)


# ------------------------------------------------------------------------ end-to-end semantics
def _selective_recompute_output(w, layer, anchors_fn):
    """Run the oracle's admission + recompute path for one layer; return the attention
    output of the recomputed rows and the pieces used to build it."""
    lay = wl.slot_layout(w)
    inp = wl.probe_inputs(w, layer)
    fresh = wl.fresh_context(w, layer)
    q_r = wl.recompute_inputs(w, layer)["q_r"]
    anchors = anchors_fn(w, inp)
    wp, rs = oracle.build_slot_maps(anchors, lay.shared_slot, lay.private_slots, T=w.T, l=w.l, L=w.L)
    kc = torch.zeros((lay.num_slots, w.hkv, w.d), dtype=w.torch_dtype)
    vc = torch.zeros_like(kc)
    # the shared region holds the precomputed affix cache
    kc[lay.shared_slot.long()] = inp["k_aff"]
    vc[lay.shared_slot.long()] = inp["v_aff"]
    # the fresh K/V of each recomputed position, in write order
    k_new = torch.stack([fresh["k_fresh"][b, torch.from_numpy(wp[b]).long()] for b in range(w.batch)])
    v_new = torch.stack([fresh["v_fresh"][b, torch.from_numpy(wp[b]).long()] for b in range(w.batch)])
    kb, vb, flags = oracle.write_slots(lay.private_slots, k_new, v_new, kc, vc,
                                       private_begin=lay.private_begin)
    assert flags == 0
    kc = torch.from_numpy(kb).view(w.torch_dtype).view(kc.shape)
    vc = torch.from_numpy(vb).view(w.torch_dtype).view(vc.shape)
    o = oracle.slot_attention(q_r, rs, kc, vc, scale=w.scale)
    return o, inp, fresh, q_r, wp


def _probe_anchors(w, inp):
    s = oracle.probe_layer(inp["q"], inp["k_req"], inp["v_req"], inp["k_aff"], inp["v_aff"],
                           T=w.T, l=w.l, masked_rows=w.masked_rows(), scale=w.scale,
                           want_out=False)["scores"]
    return oracle.topk_anchors(s, w.K)


@pytest.mark.parametrize("layout", list(LAYOUTS))
def test_ratio_one_is_full_recompute(layout):
    # invariant (ii): with every affix token an anchor, each logical position reads fresh K/V
    w = tiny(LAYOUTS[layout], ratio=1000, hq=4, hkv=2, page=4)
    assert w.K == w.L
    o, inp, fresh, q_r, wp = _selective_recompute_output(w, 0, _probe_anchors)
    assert wp.shape[1] == w.T
    # full recompute: dense attention over the fresh K/V of the whole sequence
    full = oracle.dense_attention(q_r, fresh["k_fresh"], fresh["v_fresh"], scale=w.scale)
    np.testing.assert_allclose(o, full, rtol=0, atol=1e-12)
    # and through the slot path with an identity map, bit for bit
    ident = torch.arange(w.batch * w.T, dtype=torch.int32).view(w.batch, w.T)
    o2 = oracle.slot_attention(q_r, ident, fresh["k_fresh"].reshape(-1, w.hkv, w.d),
                               fresh["v_fresh"].reshape(-1, w.hkv, w.d), scale=w.scale)
    np.testing.assert_array_equal(o, o2)


@pytest.mark.parametrize("layout", list(LAYOUTS))
def test_ratio_zero_is_direct_reuse(layout):
    # invariant (iii): with no anchors, affix positions read the shared cache and every
    # other position reads its fresh K/V
    w = tiny(LAYOUTS[layout], ratio=0, hq=4, hkv=2, page=4)
    assert w.K == 0
    o, inp, fresh, q_r, wp = _selective_recompute_output(
        w, 0, lambda w, inp: np.zeros((w.batch, 0), np.int32))
    k = fresh["k_fresh"].clone()
    v = fresh["v_fresh"].clone()
    k[:, w.l:w.l + w.L] = inp["k_aff"]
    v[:, w.l:w.l + w.L] = inp["v_aff"]
    direct = oracle.dense_attention(q_r, k, v, scale=w.scale)
    np.testing.assert_allclose(o, direct, rtol=0, atol=1e-12)


def test_partial_ratio_mixes_shared_and_fresh():
    w = tiny(LAYOUTS["infix"], ratio=500, hq=2, hkv=2, page=4)
    o, inp, fresh, q_r, wp = _selective_recompute_output(w, 0, _probe_anchors)
    k = fresh["k_fresh"].clone()
    v = fresh["v_fresh"].clone()
    for b in range(w.batch):
        anchors = set((wp[b][(wp[b] >= w.l) & (wp[b] < w.l + w.L)] - w.l).tolist())
        assert len(anchors) == w.K
        for j in range(w.L):
            if j not in anchors:
                k[b, w.l + j] = inp["k_aff"][j]
                v[b, w.l + j] = inp["v_aff"][j]
    expect = oracle.dense_attention(q_r, k, v, scale=w.scale)
    np.testing.assert_allclose(o, expect, rtol=0, atol=1e-12)


def test_thread_count_does_not_change_results():
    w = tiny(LAYOUTS["infix"], hq=4, hkv=2, batch=3)
    inp = wl.probe_inputs(w, 0)
    n0 = oracle.get_threads()
    try:
        res = []
        for n in (1, 3):
            oracle.set_threads(n)
            res.append(oracle.probe_layer(inp["q"], inp["k_req"], inp["v_req"], inp["k_aff"],
                                          inp["v_aff"], T=w.T, l=w.l,
                                          masked_rows=w.masked_rows(), scale=w.scale))
    finally:
        oracle.set_threads(n0)
    np.testing.assert_array_equal(res[0]["out"], res[1]["out"])
    np.testing.assert_array_equal(res[0]["scores"], res[1]["scores"])
