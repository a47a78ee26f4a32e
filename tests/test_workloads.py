"""The seeded input generator: geometry, determinism and slot layouts."""
import json
import os

import torch

from affix_kv_cache_gb300 import workloads as wl

GOLDEN = os.path.join(os.path.dirname(__file__), "golden", "workload_geometry.json")


def test_geometry_matches_fixture():
    g = json.load(open(GOLDEN))
    for name, w in wl.CATALOGUE.items():
        exp = g[name]
        got = {k: getattr(w, k) for k in ("T", "L", "l", "P", "m", "K", "R")}
        assert got == exp, name
        assert len(w.masked_rows()) == w.m and len(w.probe_positions()) == w.P
    for r, exp in g["llada8b_suffix_L8192_ratio_sweep"].items():
        w = wl.LLADA_SUFFIX.replace(ratio_permille=int(r))
        assert (w.K, w.R) == (exp["K"], exp["R"])


def test_masked_rows_are_generation_positions():
    w = wl.DREAM_INFIX
    pos = w.probe_positions()
    assert [pos[i] for i in w.masked_rows()] == list(range(w.T - 256, w.T))
    w = wl.LLADA_SUFFIX
    assert [w.probe_positions()[i] for i in w.masked_rows()] == list(range(256, 512))


def test_generation_is_seeded_and_layer_dependent():
    w = wl.TINY_PREFIX_F32
    a = wl.probe_inputs(w, 0)
    b = wl.probe_inputs(w, 0)
    c = wl.probe_inputs(w.replace(layers=2), 1)
    for k in a:
        assert torch.equal(a[k], b[k])
    assert not torch.equal(a["q"], c["q"][:, :, :, :])


def test_planted_keys_are_aligned_with_masked_queries():
    w = wl.TINY_PREFIX_F32
    inp = wl.probe_inputs(w, 0)
    pos = wl.plant_positions(w)
    assert len(pos) == 8
    rows = torch.tensor(w.masked_rows())
    qbar = inp["q"][0, rows].mean(dim=0)                     # [Hq][d]
    dots = torch.einsum("jhd,hd->jh", inp["k_aff"], qbar)
    planted = dots[pos].mean()
    others = dots[[j for j in range(w.L) if j not in set(pos.tolist())]].mean()
    assert planted > others


def test_prototype_mixture_has_near_duplicates():
    w = wl.LLADA_SUFFIX.replace(batch=1, segments=((wl.SEG_REQ, 4), (wl.SEG_MASK, 4), (wl.SEG_AFFIX, 640)),
                                plant_count=64 * 2, hq=2, hkv=2, d=16)
    inp = wl.probe_inputs(w, 0)
    pos = wl.plant_positions(w)
    k = inp["k_aff"][pos].float()                            # [n][Hkv][d]
    dist = torch.cdist(k[:, 0], k[:, 0])
    dist.fill_diagonal_(1e9)
    assert (dist.min(dim=1).values < 1.0).all()              # each has a sibling of its prototype


def test_slot_layout_paged():
    w = wl.LLADA_PAGED.replace(batch=3)
    lay = wl.slot_layout(w)
    assert lay.private_begin == 4096 and lay.shared_slot.shape == (w.L,)
    assert sorted(lay.shared_slot.tolist()) == list(range(w.L))
    priv = lay.private_slots.reshape(-1).tolist()
    assert len(set(priv)) == len(priv) and min(priv) >= lay.private_begin and max(priv) < lay.num_slots
    # pages are shuffled: consecutive private rows are not all physically consecutive
    d = torch.diff(lay.private_slots[0].long())
    assert (d != 1).any()
