"""GPU parity of the key re-rotation and an admission flow through the host runtime.

Sources: "Affix Cache for Diffusion Large Language Models", Sec. 4 (opening) and Limitations
(position-aware registration of a cached affix) and Sec. 4.1-4.3 (shared region, private
slots, maps recorded at admission, store-then-attend).
"""
import numpy as np
import pytest
import torch

import affix_kv_cache_gb300 as ac
import oracle

from gpu_helpers import assert_out_close, dev

pytestmark = pytest.mark.gpu


@pytest.mark.parametrize("dtype,d,hkv", [(torch.bfloat16, 128, 32), (torch.bfloat16, 64, 4), (torch.float32, 128, 1),
                                         (torch.float32, 64, 2)])
@pytest.mark.parametrize("interleaved", [False, True])
@pytest.mark.parametrize("delta", [0, 1, -17, 256, 8192])
def test_rerotate_parity(dtype, d, hkv, interleaved, delta):
    rows = 300
    k = torch.randn((rows, hkv, d), generator=torch.Generator().manual_seed(delta + d + hkv)).to(dtype)
    desc = ac.attn_desc(hkv, hkv, d, d ** -0.5, dtype)
    out = torch.empty((rows, hkv, d), dtype=dtype, device="cuda")
    ac.acache_rerotate_keys(desc, rows, dev(k), out, delta, 500000.0, interleaved)
    inplace = dev(k)
    ac.acache_rerotate_keys(desc, rows, inplace, inplace, delta, 500000.0, interleaved)
    torch.cuda.synchronize()
    ref = oracle.rerotate(k, delta, 500000.0, interleaved)
    got = out.double().cpu().numpy()
    if dtype == torch.bfloat16:      # one rounding to bf16 (half a unit in the last place) plus
        # the float32 arithmetic before it (a floor for results that cancel to near zero)
        assert np.all(np.abs(got - ref) <= 2.0 ** -8 * np.abs(ref) + 1e-6)
    else:
        assert np.abs(got - ref).max() <= 1e-5
    assert torch.equal(inplace, out)
    if delta == 0:
        assert torch.equal(out.cpu(), k)


def test_admission_flow_with_an_affix_moved_to_a_new_offset():
    """An affix cached for offset 0 is reused as an infix at offset 40: the runtime registers
    it, its keys are re-rotated into the shared slots, the request gets private pages, the
    maps are built from those slot lists, and store-then-attend matches the oracle."""
    g = torch.Generator().manual_seed(17)
    hq, hkv, d, L, l, n_req, n_mask, B, K = 4, 2, 128, 300, 40, 25, 120, 2, 60
    T = l + L + n_req + n_mask
    R = K + T - L
    desc = ac.attn_desc(hq, hkv, d, d ** -0.5, "bf16")
    pool = ac.Pool(num_slots=4096 + 8 * 256, private_begin=4096, page_slots=256)
    base, created = pool.register_affix(0xAF1, L)
    assert created
    k_aff = torch.randn((L, hkv, d), generator=g).to(torch.bfloat16)     # cached for offset 0
    v_aff = torch.randn((L, hkv, d), generator=g).to(torch.bfloat16)
    kc = torch.zeros((4096 + 8 * 256, hkv, d), dtype=torch.bfloat16, device="cuda")
    vc = torch.zeros_like(kc)
    k_moved = torch.empty((L, hkv, d), dtype=torch.bfloat16, device="cuda")
    ac.acache_rerotate_keys(desc, L, dev(k_aff), k_moved, l, 500000.0)
    shared_slot = torch.arange(base, base + L, dtype=torch.int32)
    ac.acache_write_slots(desc, 1, L, dev(shared_slot), k_moved, dev(v_aff), kc, vc, kc.shape[0], 0)
    priv, rids = [], []
    for b in range(B):
        s, rid = pool.alloc_private(R)
        priv.append(s)
        rids.append(rid)
    priv = torch.stack(priv)
    anchors = torch.stack([torch.sort(torch.randperm(L, generator=g)[:K]).values for _ in range(B)]).to(torch.int32)
    wp = torch.empty((B, R), dtype=torch.int32, device="cuda")
    rs = torch.empty((B, T), dtype=torch.int32, device="cuda")
    st = torch.zeros(1, dtype=torch.int32, device="cuda")
    ac.acache_build_slot_maps(B, T, l, L, K, dev(anchors), dev(shared_slot), dev(priv), wp, rs, dev_status=st)
    k_new = torch.randn((B, R, hkv, d), generator=g).to(torch.bfloat16)
    v_new = torch.randn((B, R, hkv, d), generator=g).to(torch.bfloat16)
    q = torch.randn((B, R, hq, d), generator=g).to(torch.bfloat16)
    out = torch.empty((B, R, hq, d), dtype=torch.bfloat16, device="cuda")
    ac.acache_store_attend(desc, B, R, dev(priv), dev(k_new), dev(v_new), kc, vc, kc.shape[0], 4096, R, dev(q), T,
                           rs, out, dev_status=st)
    torch.cuda.synchronize()
    assert st.item() == 0
    # oracle side: its own rotation (rounded to bf16 here), its own maps and pool
    k_rot = torch.from_numpy(oracle.rerotate(k_aff, l, 500000.0)).to(torch.bfloat16)
    _, rmap = oracle.build_slot_maps(anchors, shared_slot, priv, T=T, l=l, L=L)
    assert np.array_equal(rs.cpu().numpy(), rmap)
    pk = torch.zeros((kc.shape[0], hkv, d), dtype=torch.bfloat16)
    pv = torch.zeros_like(pk)
    pk[base:base + L], pv[base:base + L] = k_rot, v_aff
    kb, vb, flags = oracle.write_slots(priv, k_new, v_new, pk, pv, private_begin=4096)
    assert flags == 0
    pk = torch.from_numpy(kb).view(torch.bfloat16).reshape(pk.shape)
    pv = torch.from_numpy(vb).view(torch.bfloat16).reshape(pv.shape)
    ref = oracle.slot_attention(q, rmap, pk, pv, scale=d ** -0.5)
    assert_out_close(out.double().cpu().numpy(), ref, "bf16", "admission flow")
    for rid in rids:
        pool.free_private(rid)
    pool.release_affix(0xAF1)
    assert pool.stats() == {"free_shared": 4096, "free_private": 8 * 256, "affixes": 0, "requests": 0}
