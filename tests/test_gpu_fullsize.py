"""GPU parity at the full workload sizes, in the launch configuration the benchmark times.

Every entry point runs over the whole batch of each bf16 workload (LLaDA-8B prefix,
Dream-7B GQA infix, LLaDA-8B paged, LLaDA-8B long suffix).  The oracle then checks
sampled outputs it can afford: the first and last request, every masked row's importance
scores, and a spread of query rows that includes the ragged last tile.  Integer outputs
(anchors on identical scores, maps, stores) are checked bit for bit over the whole batch.

Inputs come from the seeded generator on the GPU (the same bits are copied to the
oracle); the oracle never receives a value computed by the CUDA path.
"""
import numpy as np
import pytest
import torch

import affix_kv_cache_gb300 as ac
import oracle
from affix_kv_cache_gb300 import workloads as wl

from gpu_helpers import assert_out_close, assert_scores_close, desc_of, status_tensor

pytestmark = pytest.mark.gpu

FULL = [wl.LLADA_PREFIX, wl.DREAM_INFIX, wl.LLADA_PAGED, wl.LLADA_SUFFIX]
IDS = [w.name for w in FULL]
# the long-suffix workload's anchor-ratio sweep (0.1 and 0.3 besides the default 0.2): K and R
# change, and with them the recomputed query rows' tiling and the private pages
RATIO_SWEEP = [wl.LLADA_SUFFIX.replace(ratio_permille=r) for r in (100, 300)]
STORE_ATTEND = FULL + RATIO_SWEEP
STORE_ATTEND_IDS = IDS + [f"{w.name}_ratio{w.ratio_permille / 1000:g}" for w in RATIO_SWEEP]


def sample_rows(n, seed, count=12):
    g = np.random.default_rng(seed)
    tail = list(range(max(0, n - 5), n))                       # the ragged last tile
    mid = sorted(set(g.choice(n, size=min(count, n), replace=False).tolist()))
    return sorted(set([0, 1, n // 2] + mid + tail))


def seeded_anchors(w, seed=1234):
    g = np.random.default_rng(seed)
    return np.stack([np.sort(g.choice(w.L, w.K, replace=False)) for _ in range(w.batch)]).astype(np.int32)


@pytest.mark.parametrize("w", FULL, ids=IDS)
def test_fullsize_probe_layer(w):
    inp = wl.probe_inputs(w, 0, device="cuda")
    d = desc_of(w)
    masked = torch.tensor(w.masked_rows(), dtype=torch.int32, device="cuda").expand(w.batch, -1).contiguous()
    scores = torch.zeros((w.batch, w.L), dtype=torch.float32, device="cuda")
    out = torch.empty_like(inp["q"])
    ws = torch.empty(ac.acache_probe_workspace_bytes(d, w.batch, w.T, w.L, w.m), dtype=torch.uint8,
                     device="cuda")
    st = status_tensor()
    ac.acache_probe_scores(d, w.batch, w.T, w.l, w.L, masked, w.m, inp["q"], inp["k_req"], inp["v_req"],
                           inp["k_aff"], inp["v_aff"], out, scores, ws, dev_status=st)
    torch.cuda.synchronize()
    assert st.item() == 0
    # scores: the oracle's full masked-row sum for the first and last request; output rows:
    # a sample of probe rows (request tokens and masked rows, incl. the ragged tail)
    checked = [0, w.batch - 1]
    rows = sorted(set(w.masked_rows()) | set(sample_rows(w.P, 7, 8)))
    cpu = {k: v[checked].cpu() if k in ("q", "k_req", "v_req") else v.cpu() for k, v in inp.items()}
    ref = oracle.probe_layer(cpu["q"], cpu["k_req"], cpu["v_req"], cpu["k_aff"], cpu["v_aff"], T=w.T,
                             l=w.l, masked_rows=w.masked_rows(), scale=w.scale, rows=rows)
    assert_scores_close(scores[checked].cpu().numpy(), ref["scores"], f"{w.name} scores")
    got = out[checked].float().cpu().numpy()[:, rows]
    assert_out_close(got, ref["out"][:, rows], "bf16", f"{w.name} probe output")
    # Top-K over the whole batch, decided on the very same float32 scores on both sides
    anchors = torch.empty((w.batch, w.K), dtype=torch.int32, device="cuda")
    ac.acache_topk_anchors(scores, w.batch, w.L, w.K, anchors, dev_status=st)
    torch.cuda.synchronize()
    want = oracle.topk_anchors(scores.cpu().double().numpy(), w.K)
    assert np.array_equal(anchors.cpu().numpy(), want)


@pytest.mark.parametrize("w", STORE_ATTEND, ids=STORE_ATTEND_IDS)
def test_fullsize_store_and_slot_attention(w):
    lay = wl.slot_layout(w)
    inp = wl.probe_inputs(w, 0, device="cuda")
    rec = wl.recompute_inputs(w, 0, 0, device="cuda")
    anchors = seeded_anchors(w)
    d = desc_of(w)
    st = status_tensor()
    # admission maps for the whole batch, bit for bit
    wp = torch.empty((w.batch, w.R), dtype=torch.int32, device="cuda")
    rs = torch.empty((w.batch, w.T), dtype=torch.int32, device="cuda")
    ac.acache_build_slot_maps(w.batch, w.T, w.l, w.L, w.K, torch.from_numpy(anchors).cuda(),
                              lay.shared_slot.cuda(), lay.private_slots.cuda(), wp, rs, dev_status=st)
    wp_ref, rs_ref = oracle.build_slot_maps(anchors, lay.shared_slot, lay.private_slots, T=w.T, l=w.l, L=w.L)
    torch.cuda.synchronize()
    assert np.array_equal(wp.cpu().numpy(), wp_ref) and np.array_equal(rs.cpu().numpy(), rs_ref)
    # store: register the shared affix, then write every request's R fresh rows
    kc = torch.zeros((lay.num_slots, w.hkv, w.d), dtype=torch.bfloat16, device="cuda")
    vc = torch.zeros_like(kc)
    ac.acache_write_slots(d, 1, w.L, lay.shared_slot.cuda(), inp["k_aff"], inp["v_aff"], kc, vc,
                          lay.num_slots, 0, dev_status=st)
    ac.acache_write_slots(d, w.batch, w.R, lay.private_slots.cuda(), rec["k_new"], rec["v_new"], kc, vc,
                          lay.num_slots, lay.private_begin, dev_status=st)
    out = torch.empty_like(rec["q_r"])
    ac.acache_slot_attention(d, w.batch, w.R, rec["q_r"], w.T, rs, kc, vc, lay.num_slots, out,
                             dev_status=st)
    torch.cuda.synchronize()
    assert st.item() == 0
    # every stored row, whole batch (a property that holds at any size)
    ps = lay.private_slots.cuda().long()
    assert torch.equal(kc[ps], rec["k_new"]) and torch.equal(vc[ps], rec["v_new"])
    assert torch.equal(kc[lay.shared_slot.cuda().long()], inp["k_aff"])
    # sampled attention rows of the first and last request: the oracle builds its own pool
    # for the request (shared affix + the request's fresh rows) from the generator's data
    rows = sample_rows(w.R, 11)
    for b in (0, w.batch - 1):
        pool_k = torch.cat([inp["k_aff"].cpu(), rec["k_new"][b].cpu()])
        pool_v = torch.cat([inp["v_aff"].cpu(), rec["v_new"][b].cpu()])
        _, rmap = oracle.build_slot_maps(anchors[b:b + 1], np.arange(w.L, dtype=np.int32),
                                         (w.L + np.arange(w.R, dtype=np.int32))[None], T=w.T, l=w.l, L=w.L)
        ref = oracle.slot_attention(rec["q_r"][b:b + 1].cpu(), rmap, pool_k, pool_v, scale=w.scale, rows=rows)
        got = out[b:b + 1].float().cpu().numpy()[:, rows]
        assert_out_close(got, ref[:, rows], "bf16", f"{w.name} slot attention request {b}")


@pytest.mark.parametrize("w", FULL, ids=IDS)
def test_fullsize_block_decode(w):
    """One block-decode step over the whole batch: the block's fresh K/V are written into the
    private slots of its positions, then its 32 queries attend over all T logical keys."""
    lay = wl.slot_layout(w)
    inp = wl.probe_inputs(w, 0, device="cuda")
    rec = wl.recompute_inputs(w, 0, 0, device="cuda")
    blk = wl.decode_inputs(w, 0, 3, device="cuda")
    pos = wl.decode_block_positions(w, 3)
    anchors = seeded_anchors(w)
    d = desc_of(w)
    st = status_tensor()
    _, rs = oracle.build_slot_maps(anchors, lay.shared_slot, lay.private_slots, T=w.T, l=w.l, L=w.L)
    rsd = torch.from_numpy(rs).cuda()
    kc = torch.zeros((lay.num_slots, w.hkv, w.d), dtype=torch.bfloat16, device="cuda")
    vc = torch.zeros_like(kc)
    ac.acache_write_slots(d, 1, w.L, lay.shared_slot.cuda(), inp["k_aff"], inp["v_aff"], kc, vc,
                          lay.num_slots, 0, dev_status=st)
    ac.acache_write_slots(d, w.batch, w.R, lay.private_slots.cuda(), rec["k_new"], rec["v_new"], kc, vc,
                          lay.num_slots, lay.private_begin, dev_status=st)
    wslot = rsd[:, pos].contiguous()
    ac.acache_write_slots(d, w.batch, len(pos), wslot, blk["k_blk"], blk["v_blk"], kc, vc, lay.num_slots,
                          lay.private_begin, dev_status=st)
    out = torch.empty_like(blk["q_blk"])
    ac.acache_slot_attention(d, w.batch, len(pos), blk["q_blk"], w.T, rsd, kc, vc, lay.num_slots, out,
                             dev_status=st)
    torch.cuda.synchronize()
    assert st.item() == 0
    ws = wslot.long()
    assert torch.equal(kc[ws], blk["k_blk"]) and torch.equal(vc[ws], blk["v_blk"])
    # the first and last request against the oracle's own pool: shared affix + the request's
    # fresh rows, with the block's rows overwritten in place
    for b in (0, w.batch - 1):
        pool_k = torch.cat([inp["k_aff"].cpu(), rec["k_new"][b].cpu()])
        pool_v = torch.cat([inp["v_aff"].cpu(), rec["v_new"][b].cpu()])
        _, rmap = oracle.build_slot_maps(anchors[b:b + 1], np.arange(w.L, dtype=np.int32),
                                         (w.L + np.arange(w.R, dtype=np.int32))[None], T=w.T, l=w.l, L=w.L)
        bslots = torch.from_numpy(rmap[0, pos].astype(np.int32))[None]
        kb, vb, flags = oracle.write_slots(bslots, blk["k_blk"][b:b + 1].cpu(), blk["v_blk"][b:b + 1].cpu(),
                                           pool_k, pool_v, private_begin=w.L)
        assert flags == 0
        pool_k = torch.from_numpy(kb).view(torch.bfloat16).reshape(pool_k.shape)
        pool_v = torch.from_numpy(vb).view(torch.bfloat16).reshape(pool_v.shape)
        ref = oracle.slot_attention(blk["q_blk"][b:b + 1].cpu(), rmap, pool_k, pool_v, scale=w.scale)
        got = out[b:b + 1].float().cpu().numpy()
        assert_out_close(got, ref, "bf16", f"{w.name} block decode request {b}")


def test_fullsize_gather_matches_store():
    w = wl.LLADA_PAGED
    lay = wl.slot_layout(w)
    g = torch.Generator(device="cuda").manual_seed(3)
    kc = torch.randn((lay.num_slots, w.hkv, w.d), generator=g, device="cuda").to(torch.bfloat16)
    vc = torch.randn((lay.num_slots, w.hkv, w.d), generator=g, device="cuda").to(torch.bfloat16)
    anchors = seeded_anchors(w)
    _, rs = oracle.build_slot_maps(anchors, lay.shared_slot, lay.private_slots, T=w.T, l=w.l, L=w.L)
    rsd = torch.from_numpy(rs).cuda()
    ko = torch.empty((w.batch, w.T, w.hkv, w.d), dtype=torch.bfloat16, device="cuda")
    vo = torch.empty_like(ko)
    ac.acache_gather_slots(desc_of(w), w.batch, w.T, rsd, kc, vc, lay.num_slots, ko, vo)
    torch.cuda.synchronize()
    assert torch.equal(ko, kc[rsd.long()]) and torch.equal(vo, vc[rsd.long()])


def test_fullsize_chained_layers_repeat():
    """One recompute point over 8 layers of the LLaDA-8B prefix workload in one call (chained
    grids, each released once its predecessor's CTAs have all started), repeated: every run
    ends with no device error and matches the per-layer calls bit for bit.  Its lone query
    tiles split their keys, and the second half of those keys is box-loaded (the request's
    own rows sit in consecutive slots) -- the case whose producer warps once fell two barrier
    phases behind and stalled the CTA."""
    w = wl.LLADA_PREFIX
    layers, reps = 8, 6
    lay = wl.slot_layout(w)
    anchors = seeded_anchors(w)
    d = desc_of(w)
    st = status_tensor()
    _, rs = oracle.build_slot_maps(anchors, lay.shared_slot, lay.private_slots, T=w.T, l=w.l, L=w.L)
    rsd = torch.from_numpy(rs).cuda()
    wslot = lay.private_slots.cuda()
    kc, vc, kn, vn, q = [], [], [], [], []
    for n in range(layers):
        inp = wl.probe_inputs(w, n, device="cuda")
        rec = wl.recompute_inputs(w, n, 0, device="cuda")
        k = torch.zeros((lay.num_slots, w.hkv, w.d), dtype=torch.bfloat16, device="cuda")
        v = torch.zeros_like(k)
        ac.acache_write_slots(d, 1, w.L, lay.shared_slot.cuda(), inp["k_aff"], inp["v_aff"], k, v,
                              lay.num_slots, 0, dev_status=st)
        kc.append(k), vc.append(v), kn.append(rec["k_new"]), vn.append(rec["v_new"]), q.append(rec["q_r"])
    ref = [torch.empty_like(x) for x in q]
    for n in range(layers):
        ac.acache_store_attend(d, w.batch, w.R, wslot, kn[n], vn[n], kc[n], vc[n], lay.num_slots,
                               lay.private_begin, w.R, q[n], w.T, rsd, ref[n], dev_status=st)
    torch.cuda.synchronize()
    assert st.item() == 0
    out = [torch.empty_like(x) for x in q]
    for r in range(reps):
        for o in out:
            o.zero_()
        ac.acache_store_attend_layers(d, w.batch, w.R, wslot, kn, vn, kc, vc, lay.num_slots, lay.private_begin,
                                      w.R, q, w.T, rsd, out, dev_status=st)
        torch.cuda.synchronize()
        assert st.item() == 0, f"device status {st.item()} in run {r}"
        for n in range(layers):
            assert torch.equal(out[n], ref[n]), f"run {r}, layer {n}"


@pytest.mark.parametrize("w", FULL, ids=IDS)
def test_fullsize_probe_layers_chained(w):
    """The probe of four layers in one call (each layer's forward chained behind the previous
    layer's head sum, starting while the previous layer's mass pass runs), repeated: no device
    error, and scores and outputs equal the per-layer calls bit for bit every time.  The first
    request's scores are checked against the oracle's four-layer sum."""
    layers, reps = 4, 3
    d = desc_of(w)
    inps = [wl.probe_inputs(w, n, device="cuda") for n in range(layers)]
    lists = [[i[k] for i in inps] for k in ("q", "k_req", "v_req", "k_aff", "v_aff")]
    masked = torch.tensor(w.masked_rows(), dtype=torch.int32, device="cuda").expand(w.batch, -1).contiguous()
    ws = torch.empty(ac.acache_probe_workspace_bytes(d, w.batch, w.T, w.L, w.m), dtype=torch.uint8,
                     device="cuda")
    st = status_tensor()
    ref_s = torch.zeros((w.batch, w.L), dtype=torch.float32, device="cuda")
    ref_o = [torch.empty_like(i["q"]) for i in inps]
    for n, i in enumerate(inps):
        ac.acache_probe_scores(d, w.batch, w.T, w.l, w.L, masked, w.m, i["q"], i["k_req"], i["v_req"],
                               i["k_aff"], i["v_aff"], ref_o[n], ref_s, ws, dev_status=st)
    torch.cuda.synchronize()
    assert st.item() == 0
    out = [torch.empty_like(o) for o in ref_o]
    for r in range(reps):
        s = torch.zeros_like(ref_s)
        for o in out:
            o.zero_()
        ac.acache_probe_scores_layers(d, w.batch, w.T, w.l, w.L, masked, w.m, *lists, out, s, ws, dev_status=st)
        torch.cuda.synchronize()
        assert st.item() == 0, f"device status {st.item()} in run {r}"
        assert torch.equal(s, ref_s), f"scores, run {r}"
        for n in range(layers):
            assert torch.equal(out[n], ref_o[n]), f"run {r}, layer {n}"
    ref = None
    for i in inps:
        cpu = {k: v[:1].cpu() if k in ("q", "k_req", "v_req") else v.cpu() for k, v in i.items()}
        ref = oracle.probe_layer(cpu["q"], cpu["k_req"], cpu["v_req"], cpu["k_aff"], cpu["v_aff"], T=w.T, l=w.l,
                                 masked_rows=w.masked_rows(), scale=w.scale, want_out=False,
                                 scores=None if ref is None else ref["scores"])
    assert_scores_close(ref_s[:1].cpu().numpy(), ref["scores"], f"{w.name} four-layer scores")
