"""CPU oracle of the affix-cache attention path -- TEST INFRASTRUCTURE ONLY.

Only the test suite, ``__graft_entry__.smoke()`` and the benchmark's CPU-baseline /
reference leg may import this package.  The product (the CUDA library and its Python
binding) never imports it, and it never imports the product.

The arithmetic lives in ``acache_ref.c`` (plain float64 loops, see its header for the
page passages each function follows and the readings taken).  This module only builds
that file with the host C compiler and marshals arrays to it.

Every function here is pinned by ``tests/test_oracle.py`` against closed forms,
invariants, library routines (torch float64 attention, a stable sort) and brute force.
"""
from __future__ import annotations

import ctypes
import os
import subprocess
import threading

import numpy as np
import torch

_HERE = os.path.dirname(os.path.abspath(__file__))
_SRC = os.path.join(_HERE, "acache_ref.c")
_BUILD_DIR = os.path.join(_HERE, "_build")
_LIB_PATH = os.path.join(_BUILD_DIR, "libacache_ref.so")
_lock = threading.Lock()
_lib = None

F32, BF16 = 0, 1


def build(force: bool = False) -> str:
    """Compile acache_ref.c into a shared library (gcc, -O2, OpenMP, no fast-math)."""
    os.makedirs(_BUILD_DIR, exist_ok=True)
    if (not force and os.path.exists(_LIB_PATH)
            and os.path.getmtime(_LIB_PATH) >= os.path.getmtime(_SRC)):
        return _LIB_PATH
    tmp = _LIB_PATH + f".tmp{os.getpid()}"
    cmd = ["gcc", "-O2", "-fopenmp", "-fPIC", "-shared", "-std=c11", "-o", tmp, _SRC, "-lm"]
    subprocess.run(cmd, check=True)
    os.replace(tmp, _LIB_PATH)
    return _LIB_PATH


def _load():
    global _lib
    with _lock:
        if _lib is None:
            lib = ctypes.CDLL(build())
            P, I, D, L = ctypes.c_void_p, ctypes.c_int, ctypes.c_double, ctypes.c_int64
            lib.ref_probe_layer.argtypes = [I, I, I, I, I, I, I, D, I, P, P, P, P, P, I, P, P, I,
                                            I, P, P, P, P]
            lib.ref_topk.argtypes = [I, I, I, P, P]
            lib.ref_build_slot_maps.argtypes = [I, I, I, I, I, P, P, P, P, P]
            lib.ref_write_slots.argtypes = [I, I, I, I, I, P, P, P, P, P, L, L]
            lib.ref_gather_slots.argtypes = [I, I, I, I, I, P, P, P, L, P, P]
            lib.ref_slot_attention.argtypes = [I, I, I, I, I, I, D, I, P, P, P, P, L, P, I, I, P]
            lib.ref_dense_attention.argtypes = [I, I, I, I, I, I, D, I, P, P, P, P]
            lib.ref_kv_deviation.argtypes = [I, I, I, I, I, P, P, P, P, P]
            lib.ref_rerotate.argtypes = [L, I, I, I, P, I, D, I, P]
            lib.ref_set_threads.argtypes = [I]
            for f in ("ref_probe_layer", "ref_topk", "ref_build_slot_maps", "ref_write_slots",
                      "ref_gather_slots", "ref_slot_attention", "ref_dense_attention",
                      "ref_kv_deviation", "ref_rerotate",
                      "ref_version", "ref_get_threads"):
                getattr(lib, f).restype = ctypes.c_int
            _lib = lib
    return _lib


def set_threads(n: int) -> None:
    _load().ref_set_threads(int(n))


def get_threads() -> int:
    return int(_load().ref_get_threads())


# ---- marshalling ---------------------------------------------------------------
def _raw(x):
    """Return (contiguous numpy array holding the raw element bits, dtype code)."""
    if isinstance(x, torch.Tensor):
        x = x.detach().cpu().contiguous()
        if x.dtype == torch.bfloat16:
            return x.view(torch.int16).numpy().view(np.uint16), BF16
        if x.dtype == torch.float32:
            return x.numpy(), F32
        raise TypeError(f"unsupported dtype {x.dtype}")
    x = np.ascontiguousarray(x)
    if x.dtype == np.float32:
        return x, F32
    raise TypeError(f"unsupported dtype {x.dtype}")


def _i32(x):
    if x is None:
        return None
    if isinstance(x, torch.Tensor):
        x = x.detach().cpu()
    return np.ascontiguousarray(np.asarray(x, dtype=np.int32))


def _bytes(x):
    if isinstance(x, torch.Tensor):
        x = x.detach().cpu().contiguous()
        return (x.view(torch.uint8) if x.dtype != torch.uint8 else x).reshape(-1).numpy()
    return np.ascontiguousarray(x).view(np.uint8).reshape(-1)


def _p(a):
    return None if a is None else a.ctypes.data_as(ctypes.c_void_p)


# ---- the oracle functions --------------------------------------------------------
def probe_layer(q, k_req, v_req, k_aff, v_aff, *, T, l, masked_rows, scale, rows=None,
                want_out=True, scores=None, affix_only_norm=False, want_stats=False):
    """One probe layer (Eq. 4-5).  q [B][P][Hq][d]; k_req/v_req [B][P][Hkv][d];
    k_aff/v_aff [L][Hkv][d]; masked_rows [B][m] (or [m], shared by all requests).

    Returns dict(out [B][P][Hq][d] float64 or None, scores [B][L] float64 (accumulated
    onto ``scores`` if given), row_max / row_sum [B][Hq][P] if want_stats).
    """
    qa, dt = _raw(q)
    kr, dt2 = _raw(k_req)
    vr, _ = _raw(v_req)
    ka, _ = _raw(k_aff)
    va, _ = _raw(v_aff)
    assert dt == dt2
    B, P, Hq, d = qa.shape
    L, Hkv = ka.shape[0], ka.shape[1]
    assert T - L == P
    mr = _i32(masked_rows)
    if mr.ndim == 1:
        mr = np.ascontiguousarray(np.broadcast_to(mr, (B, mr.shape[0])))
    m = mr.shape[1]
    rw = _i32(rows)
    n_rows = 0 if rw is None else rw.shape[0]
    out = np.zeros((B, P, Hq, d), np.float64) if want_out else None
    sc = np.zeros((B, L), np.float64) if scores is None else np.ascontiguousarray(scores, np.float64).copy()
    rmax = np.zeros((B, Hq, P), np.float64) if want_stats else None
    rsum = np.zeros((B, Hq, P), np.float64) if want_stats else None
    rc = _load().ref_probe_layer(B, T, l, L, Hq, Hkv, d, float(scale), dt, _p(qa), _p(kr), _p(vr),
                                 _p(ka), _p(va), m, _p(mr), _p(rw), n_rows,
                                 int(affix_only_norm), _p(out), _p(sc), _p(rmax), _p(rsum))
    if rc != 0:
        raise ValueError(f"ref_probe_layer rejected its arguments (rc={rc})")
    return {"out": out, "scores": sc, "row_max": rmax, "row_sum": rsum}


def topk_anchors(scores, K):
    """Eq. 6: anchors [B][K] int32, ascending offsets; ties to the lower offset."""
    if isinstance(scores, torch.Tensor):
        scores = scores.detach().cpu().double().numpy()
    s = np.ascontiguousarray(scores, np.float64)
    B, L = s.shape
    out = np.zeros((B, K), np.int32)
    rc = _load().ref_topk(B, L, K, _p(s), _p(out))
    if rc != 0:
        raise ValueError(f"ref_topk failed (rc={rc})")
    return out


def build_slot_maps(anchors, shared_slot, private_slots, *, T, l, L):
    a = _i32(anchors)
    B, K = a.shape
    R = K + T - L
    ss, ps = _i32(shared_slot), _i32(private_slots)
    assert ps.shape == (B, R), (ps.shape, (B, R))
    wp = np.zeros((B, R), np.int32)
    rs = np.zeros((B, T), np.int32)
    rc = _load().ref_build_slot_maps(B, T, l, L, K, _p(a), _p(ss), _p(ps), _p(wp), _p(rs))
    if rc != 0:
        raise ValueError("ref_build_slot_maps rejected its arguments")
    return wp, rs


def write_slots(write_slot, k_new, v_new, k_cache, v_cache, *, private_begin):
    """Returns (new k_cache bytes, new v_cache bytes, flags); caches are copied, not modified."""
    ws = _i32(write_slot)
    B, R = ws.shape
    kn, vn = _bytes(k_new), _bytes(v_new)
    kc, vc = _bytes(k_cache).copy(), _bytes(v_cache).copy()
    Hkv, d = k_new.shape[2], k_new.shape[3]
    es = k_new.element_size()
    num_slots = k_cache.shape[0]
    flags = _load().ref_write_slots(B, R, Hkv, d, es, _p(ws), _p(kn), _p(vn), _p(kc), _p(vc),
                                    num_slots, private_begin)
    return kc, vc, flags


def gather_slots(read_slot, k_cache, v_cache):
    rs = _i32(read_slot)
    B, T = rs.shape
    num_slots, Hkv, d = k_cache.shape
    es = k_cache.element_size()
    kc, vc = _bytes(k_cache), _bytes(v_cache)
    ko = np.zeros(B * T * Hkv * d * es, np.uint8)
    vo = np.zeros_like(ko)
    flags = _load().ref_gather_slots(B, T, Hkv, d, es, _p(rs), _p(kc), _p(vc), num_slots,
                                     _p(ko), _p(vo))
    return ko, vo, flags


def slot_attention(q, read_slot, k_cache, v_cache, *, scale, rows=None, drop_none=False):
    """Read-slot attention (Sec. 4.3); with drop_none, read_slot entries of -1 are discarded
    keys (DropNA, reading R7).  Returns float64 [B][nq][Hq][d]."""
    qa, dt = _raw(q)
    ka, _ = _raw(k_cache)
    va, _ = _raw(v_cache)
    B, nq, Hq, d = qa.shape
    num_slots, Hkv = ka.shape[0], ka.shape[1]
    rs = _i32(read_slot)
    T = rs.shape[1]
    rw = _i32(rows)
    out = np.zeros((B, nq, Hq, d), np.float64)
    rc = _load().ref_slot_attention(B, nq, T, Hq, Hkv, d, float(scale), dt, _p(qa), _p(rs),
                                    _p(ka), _p(va), num_slots, _p(rw),
                                    0 if rw is None else rw.shape[0], int(drop_none), _p(out))
    if rc != 0:
        raise ValueError("ref_slot_attention rejected its arguments")
    return out


def dense_attention(q, k, v, *, scale):
    qa, dt = _raw(q)
    ka, _ = _raw(k)
    va, _ = _raw(v)
    B, nq, Hq, d = qa.shape
    T, Hkv = ka.shape[1], ka.shape[2]
    out = np.zeros((B, nq, Hq, d), np.float64)
    rc = _load().ref_dense_attention(B, nq, T, Hq, Hkv, d, float(scale), dt, _p(qa), _p(ka),
                                     _p(va), _p(out))
    if rc != 0:
        raise ValueError("ref_dense_attention rejected its arguments")
    return out


def kv_deviation(k_shared, v_shared, k_full, v_full, scores=None):
    """App. B.5 high-KV-deviation scores of one layer (reading R6), float64 [B][L]; added onto
    ``scores`` if given.  k_shared/v_shared [L][Hkv][d]; k_full/v_full [B][L][Hkv][d]."""
    ks, dt = _raw(k_shared)
    vs, _ = _raw(v_shared)
    kf, dt2 = _raw(k_full)
    vf, _ = _raw(v_full)
    assert dt == dt2
    B, L, Hkv, d = kf.shape
    assert ks.shape == (L, Hkv, d)
    sc = np.zeros((B, L), np.float64) if scores is None else np.ascontiguousarray(scores, np.float64).copy()
    rc = _load().ref_kv_deviation(B, L, Hkv, d, dt, _p(ks), _p(vs), _p(kf), _p(vf), _p(sc))
    if rc != 0:
        raise ValueError("ref_kv_deviation rejected its arguments")
    return sc


def rerotate(k, delta, theta, interleaved=False):
    """Reading R8: keys k [rows][Hkv][d] carrying the rotary rotation of some position, moved
    by ``delta`` positions.  Returns float64 [rows][Hkv][d]."""
    ka, dt = _raw(k)
    rows, Hkv, d = ka.shape
    out = np.zeros((rows, Hkv, d), np.float64)
    rc = _load().ref_rerotate(rows, Hkv, d, dt, _p(ka), int(delta), float(theta), int(bool(interleaved)), _p(out))
    if rc != 0:
        raise ValueError("ref_rerotate rejected its arguments")
    return out
