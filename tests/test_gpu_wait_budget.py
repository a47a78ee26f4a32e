"""Failure detection on the GPU without a fault: a bounded wait that runs out.

Every wait of the tensor-core attention kernel's pipeline is bounded by the budget that
acache_wait_budget sets (default about a second).  With a budget of a few hundred cycles the
first wait of a launch -- the MMA thread waiting for the query tiles' TMA loads, which take
microseconds -- runs out on a healthy kernel: the kernel must flag ACACHE_DEV_TIMEOUT, let the
copies it issued land, release its tensor memory and exit, leaving no CUDA error behind.  The
same call with the default budget on the same stream must then match the oracle.
"""
import pytest
import torch

import affix_kv_cache_gb300 as ac
import oracle

from gpu_helpers import assert_out_close, dev, status_tensor

pytestmark = pytest.mark.gpu


def _case(B=2, n_q=300, T=700, hq=4, hkv=2):
    g = torch.Generator().manual_seed(77)
    d, num_slots = 128, 1500
    kc = torch.randn((num_slots, hkv, d), generator=g).to(torch.bfloat16)
    vc = torch.randn((num_slots, hkv, d), generator=g).to(torch.bfloat16)
    q = torch.randn((B, n_q, hq, d), generator=g).to(torch.bfloat16)
    rs = torch.randint(0, num_slots, (B, T), generator=g, dtype=torch.int32)
    return B, n_q, T, hq, hkv, d, num_slots, kc, vc, q, rs


# (B, n_q, T, Hq, Hkv): one wave of CTAs; several waves (384 CTAs)
@pytest.mark.parametrize("shape", [(2, 300, 700, 4, 2), (4, 600, 700, 32, 8)])
def test_wait_that_runs_out_flags_timeout_and_leaves_the_context_usable(shape):
    B, n_q, T, hq, hkv, d, num_slots, kc, vc, q, rs = _case(*shape)
    desc = ac.attn_desc(hq, hkv, d, d ** -0.5, "bf16")
    args = (desc, B, n_q, dev(q), T, dev(rs), dev(kc), dev(vc), num_slots)
    out = torch.zeros((B, n_q, hq, d), dtype=torch.bfloat16, device="cuda")
    st = status_tensor()
    prev = ac.acache_wait_budget(300)
    try:
        ac.acache_slot_attention(*args, out, dev_status=st)
        torch.cuda.synchronize()          # raises if the kernel left a CUDA error
    finally:
        ac.acache_wait_budget(prev)
    assert st.item() & ac._lib.DEV_TIMEOUT, f"device status {st.item()}"
    # the context is intact: the same call with the default budget is correct
    st2 = status_tensor()
    out2 = torch.empty_like(out)
    for _ in range(2):
        ac.acache_slot_attention(*args, out2, dev_status=st2)
    torch.cuda.synchronize()
    assert st2.item() == 0
    ref = oracle.slot_attention(q, rs, kc, vc, scale=d ** -0.5)
    assert_out_close(out2.float().cpu().numpy(), ref, "bf16", "slot attention after a timeout")


def test_probe_waits_that_run_out_flag_timeout():
    """The probe forward and the mass kernel under a 300-cycle budget: both give up their
    first waits, flag ACACHE_DEV_TIMEOUT, let their issued loads land and exit cleanly; the
    same probe with the default budget then matches the oracle."""
    from affix_kv_cache_gb300 import workloads as wl
    from gpu_helpers import assert_scores_close, probe_layer_gpu

    w = wl.Workload(name="budget", dtype="bf16", layers=1, hq=4, hkv=2, d=128, batch=2,
                    segments=((wl.SEG_AFFIX, 400), (wl.SEG_REQ, 150), (wl.SEG_MASK, 150)),
                    ratio_permille=200, recompute_points=1)
    inp = wl.probe_inputs(w, 0)
    scores = torch.zeros((w.batch, w.L), dtype=torch.float32, device="cuda")
    st = status_tensor()
    prev = ac.acache_wait_budget(300)
    try:
        probe_layer_gpu(w, inp, scores, dev_status=st)
        torch.cuda.synchronize()
    finally:
        ac.acache_wait_budget(prev)
    assert st.item() & ac._lib.DEV_TIMEOUT, f"device status {st.item()}"
    st2 = status_tensor()
    scores.zero_()
    probe_layer_gpu(w, inp, scores, dev_status=st2)
    torch.cuda.synchronize()
    assert st2.item() == 0
    ref = oracle.probe_layer(inp["q"], inp["k_req"], inp["v_req"], inp["k_aff"], inp["v_aff"], T=w.T, l=w.l,
                             masked_rows=w.masked_rows(), scale=w.scale, want_out=False)
    assert_scores_close(scores.cpu().numpy(), ref["scores"], "probe scores after a timeout")



def test_block_decode_waits_that_run_out_flag_timeout():
    """The block-decode kernel (GQA group of 2, few requests: key range split over a
    cluster) under a 300-cycle budget: every CTA of the cluster still reaches the cluster
    barriers, the launch flags ACACHE_DEV_TIMEOUT and leaves no CUDA error; the default
    budget then gives the oracle's result."""
    g = torch.Generator().manual_seed(78)
    B, n_q, T, hq, hkv, d, num_slots = 2, 32, 1408, 8, 4, 128, 3000
    kc = torch.randn((num_slots, hkv, d), generator=g).to(torch.bfloat16)
    vc = torch.randn((num_slots, hkv, d), generator=g).to(torch.bfloat16)
    q = torch.randn((B, n_q, hq, d), generator=g).to(torch.bfloat16)
    rs = torch.randint(0, num_slots, (B, T), generator=g, dtype=torch.int32)
    desc = ac.attn_desc(hq, hkv, d, d ** -0.5, "bf16")
    assert ac.acache_slot_attention_path(desc, B, n_q, T) == ac._lib.ACACHE_PATH_BLOCK_DECODE
    args = (desc, B, n_q, dev(q), T, dev(rs), dev(kc), dev(vc), num_slots)
    out = torch.zeros((B, n_q, hq, d), dtype=torch.bfloat16, device="cuda")
    st = status_tensor()
    prev = ac.acache_wait_budget(300)
    try:
        ac.acache_slot_attention(*args, out, dev_status=st)
        torch.cuda.synchronize()
    finally:
        ac.acache_wait_budget(prev)
    assert st.item() & ac._lib.DEV_TIMEOUT, f"device status {st.item()}"
    st2 = status_tensor()
    out2 = torch.empty_like(out)
    ac.acache_slot_attention(*args, out2, dev_status=st2)
    torch.cuda.synchronize()
    assert st2.item() == 0
    ref = oracle.slot_attention(q, rs, kc, vc, scale=d ** -0.5)
    assert_out_close(out2.float().cpu().numpy(), ref, "bf16", "block decode after a timeout")
