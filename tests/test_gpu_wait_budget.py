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


def _case():
    g = torch.Generator().manual_seed(77)
    B, n_q, T, hq, hkv, d, num_slots = 2, 300, 700, 4, 2, 128, 1500
    kc = torch.randn((num_slots, hkv, d), generator=g).to(torch.bfloat16)
    vc = torch.randn((num_slots, hkv, d), generator=g).to(torch.bfloat16)
    q = torch.randn((B, n_q, hq, d), generator=g).to(torch.bfloat16)
    rs = torch.randint(0, num_slots, (B, T), generator=g, dtype=torch.int32)
    return B, n_q, T, hq, hkv, d, num_slots, kc, vc, q, rs


def test_wait_that_runs_out_flags_timeout_and_leaves_the_context_usable():
    B, n_q, T, hq, hkv, d, num_slots, kc, vc, q, rs = _case()
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
