"""End-to-end anchor selection at the bf16 workload sizes: importance scores summed over
every probed layer, then Top-K, against the oracle.

Page: "Affix Cache for Diffusion Large Language Models", Sec. 3.2, Eq. 5 (s_j sums the
masked-to-affix attention over the layers, heads and initially masked rows) and Eq. 6
(A = TopK(s_j, K)).

For the first and last request of a batch the oracle sums, layer after layer, the
full-row softmax mass of every initially masked row on every affix key (float64), and
ranks those sums itself.  The CUDA path probes every layer of the whole batch in order on
one stream (the launch configuration the benchmark times), then selects anchors on its
own float32 sums.  Checked:
  - accumulated scores within 1e-3 relative of the oracle's (floor 1e-7 of the largest);
  - the GPU anchor set equals the oracle's Top-K of the ORACLE scores, except affix offsets
    whose oracle score lies within 1e-3 relative of the oracle's K-th score (the tie band);
  - the GPU Top-K over the whole batch equals the oracle's Top-K of the same float32
    scores, bit for bit.

Workloads: the LLaDA-8B prefix workload over all 32 layers; the Dream-7B GQA infix workload
and the long-suffix workload (its prototype mixture makes near-tied scores) over their
first layers, each ranked at anchor ratios 0.1, 0.2 and 0.3 (the scores do not depend on
the ratio; K does).
"""
import numpy as np
import pytest
import torch

import affix_kv_cache_gb300 as ac
import oracle
from affix_kv_cache_gb300 import workloads as wl

from gpu_helpers import assert_anchors_match, assert_scores_close, desc_of, status_tensor

pytestmark = pytest.mark.gpu

RATIOS = (100, 200, 300)
CASES = [
    (wl.LLADA_PREFIX, wl.LLADA_PREFIX.layers, (200,)),
    (wl.DREAM_INFIX, 4, RATIOS),
    (wl.LLADA_SUFFIX, 4, RATIOS),
]


def k_of(w, ratio):
    return (ratio * w.L + 999) // 1000


@pytest.mark.parametrize("w,layers,ratios", CASES, ids=[c[0].name for c in CASES])
def test_layer_summed_scores_and_anchor_sets(w, layers, ratios):
    d = desc_of(w)
    masked_rows = w.masked_rows()
    masked = torch.tensor(masked_rows, dtype=torch.int32, device="cuda").expand(w.batch, -1).contiguous()
    scores = torch.zeros((w.batch, w.L), dtype=torch.float32, device="cuda")
    ws = torch.empty(ac.acache_probe_workspace_bytes(d, w.batch, w.T, w.L, w.m), dtype=torch.uint8,
                     device="cuda")
    st = status_tensor()
    checked = [0, w.batch - 1]
    ref = None
    for n in range(layers):
        inp = wl.probe_inputs(w, n, device="cuda")
        out = torch.empty_like(inp["q"])
        ac.acache_probe_scores(d, w.batch, w.T, w.l, w.L, masked, w.m, inp["q"], inp["k_req"],
                               inp["v_req"], inp["k_aff"], inp["v_aff"], out, scores, ws, dev_status=st)
        cpu = {k: (v[checked] if k in ("q", "k_req", "v_req") else v).cpu() for k, v in inp.items()}
        # the oracle needs only the masked rows' softmax rows for the scores
        ref = oracle.probe_layer(cpu["q"], cpu["k_req"], cpu["v_req"], cpu["k_aff"], cpu["v_aff"], T=w.T,
                                 l=w.l, masked_rows=masked_rows, scale=w.scale, rows=masked_rows,
                                 want_out=False, scores=None if ref is None else ref["scores"])
        del inp, out
    torch.cuda.synchronize()
    assert st.item() == 0
    got = scores.cpu().numpy()
    assert_scores_close(got[checked], ref["scores"], f"{w.name}: scores over {layers} layers")
    for ratio in ratios:
        K = k_of(w, ratio)
        anchors = torch.empty((w.batch, K), dtype=torch.int32, device="cuda")
        ac.acache_topk_anchors(scores, w.batch, w.L, K, anchors, dev_status=st)
        torch.cuda.synchronize()
        assert st.item() == 0
        a = anchors.cpu().numpy()
        # the whole batch, decided on the very same float32 scores on both sides
        assert np.array_equal(a, oracle.topk_anchors(got.astype(np.float64), K)), f"ratio {ratio / 1000}"
        # the first and last request against the oracle's own scores, with the tie band
        assert_anchors_match(a[checked], ref["scores"], K, f"{w.name} ratio {ratio / 1000}")
