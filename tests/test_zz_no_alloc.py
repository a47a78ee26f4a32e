"""The scratch-free probe entry point, acache_probe_scores_noalloc, through the C ABI.

Some callers of this library cannot allocate device memory when they probe -- an engine that
hands the library only tensors it already owns (a memory budget split up at start-up, an
allocator the library cannot reach, or code that must stay out of the CUDA allocator).  This
entry point keeps the probe's scratch in a fixed 16 MiB array inside the library instead of a
caller-provided workspace.  These tests check that it returns the same importance scores and
probe outputs as acache_probe_scores -- bit for bit, and so within the path's tolerances -- on
two calls in a row with different inputs, that a larger call's leftovers in the array do not
reach the smaller call after it (which also matches the oracle), and that a request too large
for the fixed array is refused.

This file is collected last on purpose: if it fails, a run that stops at the first failure
has already run every other test.
"""
import pytest
import torch

import affix_kv_cache_gb300 as ac
import oracle
from affix_kv_cache_gb300 import workloads as wl

from gpu_helpers import assert_out_close, assert_scores_close, desc_of

pytestmark = pytest.mark.gpu

SMALL_BF16 = wl.Workload(
    name="noalloc_infix_bf16", dtype="bf16", layers=2, hq=4, hkv=2, d=128, batch=2,
    segments=((wl.SEG_REQ, 100), (wl.SEG_AFFIX, 400), (wl.SEG_REQ, 50), (wl.SEG_MASK, 150)),
    ratio_permille=200, recompute_points=1, plant="aligned", plant_count=20, plant_scale=1.5)
# a larger call first, so that the fixed array still holds its leftovers beyond the extent of
# the smaller call that follows
LARGER_BF16 = wl.Workload(
    name="noalloc_prefix_bf16_larger", dtype="bf16", layers=1, hq=8, hkv=8, d=128, batch=3,
    segments=((wl.SEG_AFFIX, 1100), (wl.SEG_REQ, 90), (wl.SEG_MASK, 230)),
    ratio_permille=200, recompute_points=1, plant="aligned", plant_count=30, plant_scale=1.5)
TINY_F32 = wl.TINY_PREFIX_F32.replace(layers=2)


def probe_both(w, layer):
    inp = wl.probe_inputs(w, layer, device="cuda")
    d = desc_of(w)
    masked = torch.tensor(w.masked_rows(), dtype=torch.int32, device="cuda").expand(w.batch, -1).contiguous()
    s_ws = torch.zeros((w.batch, w.L), dtype=torch.float32, device="cuda")
    o_ws = torch.empty_like(inp["q"])
    ws = torch.empty(ac.acache_probe_workspace_bytes(d, w.batch, w.T, w.L, w.m), dtype=torch.uint8,
                     device="cuda")
    ac.acache_probe_scores(d, w.batch, w.T, w.l, w.L, masked, w.m, inp["q"], inp["k_req"], inp["v_req"],
                           inp["k_aff"], inp["v_aff"], o_ws, s_ws, ws)
    s_na = torch.zeros_like(s_ws)
    o_na = torch.empty_like(o_ws)
    st = torch.zeros(1, dtype=torch.int32, device="cuda")
    ac.acache_probe_scores_noalloc(d, w.batch, w.T, w.l, w.L, masked, w.m, inp["q"], inp["k_req"],
                                   inp["v_req"], inp["k_aff"], inp["v_aff"], o_na, s_na, dev_status=st)
    torch.cuda.synchronize()
    assert st.item() == 0
    return inp, s_ws, o_ws, s_na, o_na


@pytest.mark.parametrize("w", [SMALL_BF16, TINY_F32], ids=lambda w: w.name)
def test_noalloc_probe_matches_workspace_probe_on_two_calls(w):
    for layer in (0, 1):      # two calls in a row on different inputs share the fixed scratch
        _, s_ws, o_ws, s_na, o_na = probe_both(w, layer)
        # the same kernels on the same inputs: the same bits, whichever memory holds the scratch
        assert torch.equal(s_na, s_ws), f"scores, call {layer + 1}"
        assert torch.equal(o_na, o_ws), f"probe output, call {layer + 1}"
        assert_scores_close(s_na.cpu().numpy(), s_ws.cpu().numpy(), f"scores, call {layer + 1}")
        assert_out_close(o_na.float().cpu().numpy(), o_ws.float().cpu().numpy(), w.dtype,
                         f"probe output, call {layer + 1}")


def test_noalloc_larger_call_then_smaller_call_matches_oracle():
    """Leftovers of a larger earlier call in the fixed scratch do not reach a smaller call."""
    for w in (LARGER_BF16, SMALL_BF16):
        inp, s_ws, o_ws, s_na, o_na = probe_both(w, 0)
        assert torch.equal(s_na, s_ws) and torch.equal(o_na, o_ws), w.name
    cpu = {k: v.cpu() for k, v in inp.items()}
    ref = oracle.probe_layer(cpu["q"], cpu["k_req"], cpu["v_req"], cpu["k_aff"], cpu["v_aff"], T=w.T,
                             l=w.l, masked_rows=w.masked_rows(), scale=w.scale)
    assert_scores_close(s_na.cpu().numpy(), ref["scores"], "scores of the smaller call vs the oracle")
    assert_out_close(o_na.float().cpu().numpy(), ref["out"], "bf16", "output of the smaller call vs the oracle")


def test_noalloc_refuses_requests_beyond_its_scratch():
    # the long-suffix workload needs about 38 MB of scratch (> 16 MiB): refused before launch
    w = wl.LLADA_SUFFIX
    buf = torch.zeros(64, dtype=torch.bfloat16, device="cuda")
    sc = torch.zeros(64, dtype=torch.float32, device="cuda")
    masked = torch.zeros(64, dtype=torch.int32, device="cuda")
    st = ac.acache_probe_scores_noalloc(desc_of(w), w.batch, w.T, w.l, w.L, masked, w.m, buf, buf, buf,
                                        buf, buf, None, sc, check=False)
    assert st == ac._lib.ACACHE_ERR_WORKSPACE
