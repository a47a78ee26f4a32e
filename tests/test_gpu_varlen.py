"""GPU parity of the ragged-batch read-slot attention and of store-then-attend in one call.

Ragged batches (App. C.1: ragged query / KV lengths next to the read-slot map): every request
has its own row and key counts in one launch; each request's rows are compared with the
oracle run on that request alone.  Store-then-attend (Sec. 4.3, App. C.1): one call must give
exactly what the store followed by the attention gives, and match the oracle.
"""
import numpy as np
import pytest
import torch

import affix_kv_cache_gb300 as ac
import oracle
from affix_kv_cache_gb300 import _lib

from gpu_helpers import assert_out_close, dev

pytestmark = pytest.mark.gpu


def _ragged(n_rows, n_keys, hq, hkv, d, dtype, num_slots, seed, drop_every=0):
    g = torch.Generator().manual_seed(seed)
    total_q, total_t = sum(n_rows), sum(n_keys)
    q = (torch.randn((max(total_q, 1), hq, d), generator=g) * 2).to(dtype)
    kc = torch.randn((num_slots, hkv, d), generator=g).to(dtype)
    vc = torch.randn((num_slots, hkv, d), generator=g).to(dtype)
    rs = torch.randint(0, num_slots, (max(total_t, 1),), generator=g, dtype=torch.int32)
    if drop_every:
        rs[::drop_every] = -1
    q_start = torch.tensor([0] + list(np.cumsum(n_rows)), dtype=torch.int32)
    kv_start = torch.tensor([0] + list(np.cumsum(n_keys)), dtype=torch.int32)
    return q, kc, vc, rs, q_start, kv_start


# per-request (rows, keys): empty requests, one key, ragged key tiles, several Q blocks
CASES = [
    ("bf16-gqa", torch.bfloat16, 128, 8, 2, [(300, 700), (0, 50), (5, 1), (589, 1408), (128, 129)]),
    ("bf16-mha", torch.bfloat16, 128, 4, 4, [(32, 4480), (1, 37), (257, 256)]),
    ("f32", torch.float32, 64, 2, 2, [(40, 200), (0, 0), (7, 33), (1, 1)]),
]


@pytest.mark.parametrize("name,dtype,d,hq,hkv,reqs", CASES, ids=[c[0] for c in CASES])
@pytest.mark.parametrize("drop", [False, True])
def test_varlen_slot_attention_parity(name, dtype, d, hq, hkv, reqs, drop):
    n_rows, n_keys = [r for r, _ in reqs], [k for _, k in reqs]
    B, ns = len(reqs), 5000
    q, kc, vc, rs, qs, ks = _ragged(n_rows, n_keys, hq, hkv, d, dtype, ns, seed=len(name) + 7 * B,
                                    drop_every=5 if drop else 0)
    out = torch.full((q.shape[0], hq, d), float("nan"), dtype=dtype, device="cuda")
    st = torch.zeros(1, dtype=torch.int32, device="cuda")
    desc = ac.attn_desc(hq, hkv, d, d ** -0.5, dtype)
    ac.acache_slot_attention_varlen(desc, B, dev(qs), max(n_rows), sum(n_rows), dev(q), dev(ks), max(n_keys),
                                    dev(rs), dev(kc), dev(vc), ns, out, drop_none=drop, dev_status=st)
    torch.cuda.synchronize()
    assert st.item() == 0
    got = out.double().cpu().numpy()
    tol = "bf16" if dtype == torch.bfloat16 else "f32"
    for b in range(B):
        if n_rows[b] == 0:
            continue
        q0, q1, k0, k1 = int(qs[b]), int(qs[b + 1]), int(ks[b]), int(ks[b + 1])
        ref = oracle.slot_attention(q[q0:q1][None], rs[k0:k1][None], kc, vc, scale=d ** -0.5, drop_none=drop)
        assert_out_close(got[q0:q1], ref[0], tol, f"{name} request {b}")


def test_varlen_bad_length_is_skipped_and_flagged():
    reqs = [(40, 300), (50, 300), (30, 0)]        # request 1 exceeds max_q_rows; request 2 has no key
    n_rows, n_keys = [r for r, _ in reqs], [k for _, k in reqs]
    q, kc, vc, rs, qs, ks = _ragged(n_rows, n_keys, 2, 2, 128, torch.bfloat16, 2000, seed=3)
    out = torch.full((q.shape[0], 2, 128), float("nan"), dtype=torch.bfloat16, device="cuda")
    st = torch.zeros(1, dtype=torch.int32, device="cuda")
    ac.acache_slot_attention_varlen(ac.attn_desc(2, 2, 128, 128 ** -0.5, "bf16"), 3, dev(qs), 45, sum(n_rows),
                                    dev(q), dev(ks), 300, dev(rs), dev(kc), dev(vc), 2000, out, dev_status=st)
    torch.cuda.synchronize()
    assert st.item() == _lib.DEV_BAD_LENGTH
    got = out.double().cpu().numpy()
    assert np.isnan(got[40:120]).all()            # skipped requests: rows untouched
    ref = oracle.slot_attention(q[:40][None], rs[:300][None], kc, vc, scale=128 ** -0.5)
    assert_out_close(got[:40], ref[0], "bf16", "request 0")


# ------------------------------------------------------------------------ store-then-attend
@pytest.mark.parametrize("B,rows,n_q,hq,hkv,T,dtype,d", [(2, 589, 589, 4, 4, 1408, torch.bfloat16, 128),
                                                        (3, 32, 32, 8, 4, 600, torch.bfloat16, 128),
                                                        (2, 40, 40, 2, 2, 150, torch.float32, 64)])
def test_store_attend_equals_store_then_attention(B, rows, n_q, hq, hkv, T, dtype, d):
    g = torch.Generator().manual_seed(B + rows + T)
    ns, priv0 = 6000, 2000
    kc = torch.randn((ns, hkv, d), generator=g).to(dtype)
    vc = torch.randn((ns, hkv, d), generator=g).to(dtype)
    # private slots for the fresh rows (disjoint per request), read map mixing shared and private
    ws = (priv0 + torch.randperm(ns - priv0, generator=g)[:B * rows]).to(torch.int32).reshape(B, rows)
    rs = torch.randint(0, priv0, (B, T), generator=g, dtype=torch.int32)
    for b in range(B):
        pos = torch.randperm(T, generator=g)[:min(rows, T)]
        rs[b, pos] = ws[b, :len(pos)]
    kn = torch.randn((B, rows, hkv, d), generator=g).to(dtype)
    vn = torch.randn((B, rows, hkv, d), generator=g).to(dtype)
    q = (torch.randn((B, n_q, hq, d), generator=g) * 2).to(dtype)
    desc = ac.attn_desc(hq, hkv, d, d ** -0.5, dtype)
    st = torch.zeros(1, dtype=torch.int32, device="cuda")
    # one call
    k1, v1 = dev(kc), dev(vc)
    o1 = torch.empty((B, n_q, hq, d), dtype=dtype, device="cuda")
    ac.acache_store_attend(desc, B, rows, dev(ws), dev(kn), dev(vn), k1, v1, ns, priv0, n_q, dev(q), T, dev(rs),
                           o1, dev_status=st)
    # the two calls
    k2, v2 = dev(kc), dev(vc)
    o2 = torch.empty_like(o1)
    ac.acache_write_slots(desc, B, rows, dev(ws), dev(kn), dev(vn), k2, v2, ns, priv0, dev_status=st)
    ac.acache_slot_attention(desc, B, n_q, dev(q), T, dev(rs), k2, v2, ns, o2, dev_status=st)
    torch.cuda.synchronize()
    assert st.item() == 0
    assert torch.equal(k1, k2) and torch.equal(v1, v2)
    assert torch.equal(o1, o2)
    ref = oracle.slot_attention(q, rs, k1.cpu(), v1.cpu(), scale=d ** -0.5)
    assert_out_close(o1.double().cpu().numpy(), ref, "bf16" if dtype == torch.bfloat16 else "f32", "store_attend")


def test_store_attend_one_half_only():
    d, hq, hkv, ns = 128, 2, 2, 400
    g = torch.Generator().manual_seed(9)
    kc = torch.randn((ns, hkv, d), generator=g).to(torch.bfloat16).cuda()
    vc = torch.randn((ns, hkv, d), generator=g).to(torch.bfloat16).cuda()
    kn = torch.randn((1, 3, hkv, d), generator=g).to(torch.bfloat16).cuda()
    ws = torch.tensor([[300, 301, 302]], dtype=torch.int32, device="cuda")
    desc = ac.attn_desc(hq, hkv, d, d ** -0.5, "bf16")
    ac.acache_store_attend(desc, 1, 3, ws, kn, kn, kc, vc, ns, 256, 0, None, 0, None, None)   # store only
    torch.cuda.synchronize()
    assert torch.equal(kc[300:303], kn[0]) and torch.equal(vc[300:303], kn[0])
    q = torch.randn((1, 5, hq, d), generator=g).to(torch.bfloat16).cuda()
    rs = torch.arange(0, 50, dtype=torch.int32, device="cuda")[None]
    o = torch.empty_like(q)
    ac.acache_store_attend(desc, 1, 0, None, None, None, kc, vc, ns, 256, 5, q, 50, rs, o)      # attend only
    torch.cuda.synchronize()
    ref = oracle.slot_attention(q.cpu(), rs.cpu(), kc.cpu(), vc.cpu(), scale=d ** -0.5)
    assert_out_close(o.double().cpu().numpy(), ref, "bf16", "attend only")


# ----------------------------------------------------------- store-then-attend over layers
def _layers_case(L, B, rows, n_q, hq, hkv, T, d, ns, priv0, seed):
    g = torch.Generator().manual_seed(seed)
    dt = torch.bfloat16
    kc = [torch.randn((ns, hkv, d), generator=g).to(dt) for _ in range(L)]
    vc = [torch.randn((ns, hkv, d), generator=g).to(dt) for _ in range(L)]
    ws = (priv0 + torch.randperm(ns - priv0, generator=g)[:B * rows]).to(torch.int32).reshape(B, rows)
    rs = torch.randint(0, priv0, (B, T), generator=g, dtype=torch.int32)
    for b in range(B):
        pos = torch.randperm(T, generator=g)[:min(rows, T)]
        rs[b, pos] = ws[b, :len(pos)]
    kn = [torch.randn((B, rows, hkv, d), generator=g).to(dt) for _ in range(L)]
    vn = [torch.randn((B, rows, hkv, d), generator=g).to(dt) for _ in range(L)]
    q = [(torch.randn((B, n_q, hq, d), generator=g) * 2).to(dt) for _ in range(L)]
    return kc, vc, ws, rs, kn, vn, q


@pytest.mark.parametrize("L,B,rows,n_q,T", [(3, 2, 300, 300, 700), (4, 1, 40, 40, 1408), (2, 3, 0, 129, 300),
                                            (3, 2, 77, 0, 300)])
def test_store_attend_layers_equals_per_layer_calls(L, B, rows, n_q, T):
    hq, hkv, d, ns, priv0 = 4, 2, 128, 3000, 1000
    kc, vc, ws, rs, kn, vn, q = _layers_case(L, B, rows, n_q, hq, hkv, T, d, ns, priv0, seed=L * 10 + rows)
    desc = ac.attn_desc(hq, hkv, d, d ** -0.5, "bf16")
    st = torch.zeros(1, dtype=torch.int32, device="cuda")
    # one call over all layers (chained grids)
    k1, v1 = [dev(x) for x in kc], [dev(x) for x in vc]
    o1 = [torch.empty((B, n_q, hq, d), dtype=torch.bfloat16, device="cuda") for _ in range(L)]
    ac.acache_store_attend_layers(desc, B, rows, dev(ws), [dev(x) for x in kn] if rows else None,
                                  [dev(x) for x in vn] if rows else None, k1, v1, ns, priv0, n_q,
                                  [dev(x) for x in q] if n_q else None, T, dev(rs), o1 if n_q else None,
                                  dev_status=st)
    # one call per layer
    k2, v2 = [dev(x) for x in kc], [dev(x) for x in vc]
    o2 = [torch.empty_like(o) for o in o1]
    for l in range(L):
        ac.acache_store_attend(desc, B, rows, dev(ws), dev(kn[l]) if rows else None, dev(vn[l]) if rows else None,
                               k2[l], v2[l], ns, priv0, n_q, dev(q[l]) if n_q else None, T, dev(rs),
                               o2[l] if n_q else None, dev_status=st)
    torch.cuda.synchronize()
    assert st.item() == 0
    # the same copies and the same attention grids (only their launch order differs): identical
    # bits, and each layer's output within the oracle's tolerance
    for l in range(L):
        assert torch.equal(k1[l], k2[l]) and torch.equal(v1[l], v2[l]), f"pool of layer {l}"
        if n_q:
            assert torch.equal(o1[l], o2[l]), f"output of layer {l}"
            ref = oracle.slot_attention(q[l], rs, k1[l].cpu(), v1[l].cpu(), scale=d ** -0.5)
            assert_out_close(o1[l].double().cpu().numpy(), ref, "bf16", f"layer {l}")


def test_store_attend_layers_shared_pool_runs_in_order():
    # two layers on the same pool: the call must behave as the per-layer calls in order (the
    # second store lands after the first attention has read the pool)
    L, B, rows, n_q, T, hq, hkv, d, ns, priv0 = 2, 2, 100, 100, 400, 2, 2, 128, 1500, 500
    kc, vc, ws, rs, kn, vn, q = _layers_case(L, B, rows, n_q, hq, hkv, T, d, ns, priv0, seed=5)
    desc = ac.attn_desc(hq, hkv, d, d ** -0.5, "bf16")
    st = torch.zeros(1, dtype=torch.int32, device="cuda")
    kp, vp = dev(kc[0]), dev(vc[0])
    o1 = [torch.empty((B, n_q, hq, d), dtype=torch.bfloat16, device="cuda") for _ in range(L)]
    ac.acache_store_attend_layers(desc, B, rows, dev(ws), [dev(x) for x in kn], [dev(x) for x in vn], [kp, kp],
                                  [vp, vp], ns, priv0, n_q, [dev(x) for x in q], T, dev(rs), o1, dev_status=st)
    kp2, vp2 = dev(kc[0]), dev(vc[0])
    o2 = [torch.empty_like(o) for o in o1]
    for l in range(L):
        ac.acache_store_attend(desc, B, rows, dev(ws), dev(kn[l]), dev(vn[l]), kp2, vp2, ns, priv0, n_q, dev(q[l]),
                               T, dev(rs), o2[l], dev_status=st)
    torch.cuda.synchronize()
    assert st.item() == 0
    assert torch.equal(kp, kp2) and torch.equal(vp, vp2)
    for l in range(L):          # overlapping buffers: the call runs the per-layer calls themselves
        assert torch.equal(o1[l], o2[l])
