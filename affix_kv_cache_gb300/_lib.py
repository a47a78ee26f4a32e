"""ctypes binding of libacache.so (include/acache.h).

Argument marshalling only: every function takes torch tensors (device memory) or plain
integers, passes their device pointers, sizes and the current CUDA stream to the C entry
point of the same name, and raises AcacheError on a non-zero status.  No step of the
path runs here, and there is no fallback: if the library is missing, importing this
module's functions fails loudly.
"""
from __future__ import annotations

import ctypes
import os

import torch

_PKG = os.path.dirname(os.path.abspath(__file__))
LIB_PATH = os.path.join(_PKG, "_build", "libacache.so")

ACACHE_OK = 0
ACACHE_ERR_INVALID_ARG = -1
ACACHE_ERR_UNSUPPORTED = -2
ACACHE_ERR_CUDA = -3
ACACHE_ERR_WORKSPACE = -4
ACACHE_ERR_TIMEOUT = -5
ACACHE_F32 = 0
ACACHE_BF16 = 1
ACACHE_PATH_RECOMPUTE = 0
ACACHE_PATH_BLOCK_DECODE = 1
ACACHE_PATH_CUDA_CORES = 2
ACACHE_PATH_RECOMPUTE_PERSISTENT = 3
SLOT_NONE = -1
DEV_BAD_SLOT, DEV_SHARED_WRITE, DEV_BAD_ROW, DEV_BAD_ANCHOR, DEV_NAN, DEV_TIMEOUT = 1, 2, 4, 8, 16, 32
DEV_BAD_LENGTH = 64

EXPORTS = ("acache_status_string", "acache_version", "acache_wait_budget", "acache_probe_workspace_bytes",
           "acache_probe_scores", "acache_probe_scores_layers", "acache_probe_scores_noalloc", "acache_topk_anchors", "acache_build_slot_maps",
           "acache_write_slots", "acache_slot_attention", "acache_gather_slots",
           "acache_kv_deviation_scores", "acache_slot_attention_dropna", "acache_slot_attention_varlen",
           "acache_slot_attention_path",
           "acache_store_attend", "acache_store_attend_layers", "acache_rerotate_keys", "acache_pool_create",
           "acache_pool_destroy",
           "acache_pool_register_affix", "acache_pool_release_affix", "acache_pool_alloc_private",
           "acache_pool_free_private", "acache_pool_stats")


class AcacheError(RuntimeError):
    def __init__(self, fn, status):
        super().__init__(f"{fn} returned {status} ({status_string(status)})")
        self.status = status


class AttnDesc(ctypes.Structure):
    _fields_ = [("num_q_heads", ctypes.c_int32), ("num_kv_heads", ctypes.c_int32),
                ("head_dim", ctypes.c_int32), ("scale", ctypes.c_float),
                ("dtype", ctypes.c_int32)]


def attn_desc(hq: int, hkv: int, d: int, scale: float, dtype) -> AttnDesc:
    if isinstance(dtype, torch.dtype):
        dtype = {torch.float32: ACACHE_F32, torch.bfloat16: ACACHE_BF16}[dtype]
    elif isinstance(dtype, str):
        dtype = {"f32": ACACHE_F32, "bf16": ACACHE_BF16}[dtype]
    return AttnDesc(hq, hkv, d, scale, dtype)


_lib = None


def lib() -> ctypes.CDLL:
    """Load libacache.so (built by __graft_entry__.build() or build.py)."""
    global _lib
    if _lib is None:
        if not os.path.exists(LIB_PATH):
            raise RuntimeError(f"libacache.so is not built ({LIB_PATH} missing); "
                               "run `python -c 'import __graft_entry__ as g; g.build()'`")
        L = ctypes.CDLL(LIB_PATH)
        P, I, I64, S = ctypes.c_void_p, ctypes.c_int, ctypes.c_int64, ctypes.c_size_t
        D = ctypes.POINTER(AttnDesc)
        sig = {
            "acache_status_string": (ctypes.c_char_p, [I]),
            "acache_version": (I, []),
            "acache_wait_budget": (I64, [I64]),
            "acache_probe_workspace_bytes": (S, [D, I, I, I, I]),
            "acache_probe_scores": (I, [D, I, I, I, I, P, I, P, P, P, P, P, P, P, P, S, P, P]),
            "acache_probe_scores_layers": (I, [D, I, I, I, I, I, P, I, P, P, P, P, P, P, P, P, S, P, P]),
            "acache_probe_scores_noalloc": (I, [D, I, I, I, I, P, I, P, P, P, P, P, P, P, P, P]),
            "acache_topk_anchors": (I, [P, I, I, I, P, P, P]),
            "acache_build_slot_maps": (I, [I, I, I, I, I, P, P, P, P, P, P, P]),
            "acache_write_slots": (I, [D, I, I, P, P, P, P, P, I64, I64, P, P]),
            "acache_slot_attention": (I, [D, I, I, P, I, P, P, P, I64, P, P, P]),
            "acache_slot_attention_path": (I, [D, I, I, I]),
            "acache_gather_slots": (I, [D, I, I, P, P, P, I64, P, P, P, P]),
            "acache_kv_deviation_scores": (I, [D, I, I, P, P, P, P, P, P]),
            "acache_slot_attention_dropna": (I, [D, I, I, P, I, P, P, P, I64, P, P, P]),
            "acache_slot_attention_varlen": (I, [D, I, P, I, I, P, P, I, P, P, P, I64, P, I, P, P]),
            "acache_store_attend": (I, [D, I, I, P, P, P, P, P, I64, I64, I, P, I, P, P, P, P]),
            "acache_store_attend_layers": (I, [D, I, I, I, P, P, P, P, P, I64, I64, I, P, I, P, P, P, P]),
            "acache_rerotate_keys": (I, [D, I64, P, P, ctypes.c_int32, ctypes.c_double, I, P]),
            "acache_pool_create": (I, [I64, I64, ctypes.c_int32, ctypes.POINTER(P)]),
            "acache_pool_destroy": (None, [P]),
            "acache_pool_register_affix": (I, [P, ctypes.c_uint64, ctypes.c_int32, ctypes.POINTER(ctypes.c_int32),
                                               ctypes.POINTER(ctypes.c_int32)]),
            "acache_pool_release_affix": (I, [P, ctypes.c_uint64]),
            "acache_pool_alloc_private": (I, [P, ctypes.c_int32, P, ctypes.POINTER(I64)]),
            "acache_pool_free_private": (I, [P, I64]),
            "acache_pool_stats": (I, [P, ctypes.POINTER(I64), ctypes.POINTER(I64), ctypes.POINTER(ctypes.c_int32),
                                      ctypes.POINTER(ctypes.c_int32)]),
        }
        for name, (res, args) in sig.items():
            f = getattr(L, name)
            f.restype, f.argtypes = res, args
        _lib = L
    return _lib


def status_string(status: int) -> str:
    return lib().acache_status_string(int(status)).decode()


def version() -> int:
    return int(lib().acache_version())


def _p(t):
    if t is None:
        return None
    if isinstance(t, int):
        return t or None
    return t.data_ptr() or None


def _stream(stream):
    if stream is None:
        return torch.cuda.current_stream().cuda_stream if torch.cuda.is_available() else None
    if isinstance(stream, torch.cuda.Stream):
        return stream.cuda_stream
    return stream


def _check(fn, status):
    if status != ACACHE_OK:
        raise AcacheError(fn, status)
    return status


def acache_wait_budget(cycles: int = 0) -> int:
    """Set (cycles > 0) or read (cycles <= 0) the SM-cycle budget of the kernels' bounded
    waits; returns the budget in force before the call (see include/acache.h)."""
    return int(lib().acache_wait_budget(int(cycles)))


def acache_probe_workspace_bytes(desc, batch, seq_len, affix_len, num_masked) -> int:
    return int(lib().acache_probe_workspace_bytes(ctypes.byref(desc), batch, seq_len, affix_len,
                                                  num_masked))


def acache_probe_scores(desc, batch, seq_len, affix_begin, affix_len, masked_rows, num_masked,
                        q, k_req, v_req, k_affix, v_affix, out, scores, workspace,
                        workspace_bytes=None, dev_status=None, stream=None, check=True):
    if workspace_bytes is None:
        workspace_bytes = 0 if workspace is None else workspace.numel() * workspace.element_size()
    st = lib().acache_probe_scores(ctypes.byref(desc), batch, seq_len, affix_begin, affix_len,
                                   _p(masked_rows), num_masked, _p(q), _p(k_req), _p(v_req),
                                   _p(k_affix), _p(v_affix), _p(out), _p(scores), _p(workspace),
                                   workspace_bytes, _p(dev_status), _stream(stream))
    return _check("acache_probe_scores", st) if check else st


def acache_probe_scores_layers(desc, batch, seq_len, affix_begin, affix_len, masked_rows, num_masked,
                               q, k_req, v_req, k_affix, v_affix, out, scores, workspace,
                               workspace_bytes=None, dev_status=None, stream=None, check=True):
    """The probe of every layer in one call (see include/acache.h): q, k_req, v_req, k_affix,
    v_affix and out are lists of tensors, one per layer (out, k_affix and v_affix may be None)."""
    layers = len(q)
    if workspace_bytes is None:
        workspace_bytes = 0 if workspace is None else workspace.numel() * workspace.element_size()
    keep = [_ptr_array(x, layers) for x in (q, k_req, v_req, k_affix, v_affix, out)]
    ptrs = [k[0] if k is not None else None for k in keep]
    st = lib().acache_probe_scores_layers(ctypes.byref(desc), layers, batch, seq_len, affix_begin, affix_len,
                                          _p(masked_rows), num_masked, ptrs[0], ptrs[1], ptrs[2], ptrs[3],
                                          ptrs[4], ptrs[5], _p(scores), _p(workspace), workspace_bytes,
                                          _p(dev_status), _stream(stream))
    del keep
    return _check("acache_probe_scores_layers", st) if check else st


def acache_probe_scores_noalloc(desc, batch, seq_len, affix_begin, affix_len, masked_rows,
                                num_masked, q, k_req, v_req, k_affix, v_affix, out, scores,
                                dev_status=None, stream=None, check=True):
    """acache_probe_scores without a workspace, for callers that cannot allocate device
    memory: the scratch is a fixed 16 MiB array inside the library (see include/acache.h)."""
    st = lib().acache_probe_scores_noalloc(ctypes.byref(desc), batch, seq_len, affix_begin,
                                           affix_len, _p(masked_rows), num_masked, _p(q),
                                           _p(k_req), _p(v_req), _p(k_affix), _p(v_affix),
                                           _p(out), _p(scores), _p(dev_status), _stream(stream))
    return _check("acache_probe_scores_noalloc", st) if check else st


def acache_topk_anchors(scores, batch, affix_len, k, anchors, dev_status=None, stream=None,
                        check=True):
    st = lib().acache_topk_anchors(_p(scores), batch, affix_len, k, _p(anchors), _p(dev_status),
                                   _stream(stream))
    return _check("acache_topk_anchors", st) if check else st


def acache_build_slot_maps(batch, seq_len, affix_begin, affix_len, k, anchors, shared_slot,
                           private_slots, write_pos, read_slot, dev_status=None, stream=None,
                           check=True):
    st = lib().acache_build_slot_maps(batch, seq_len, affix_begin, affix_len, k, _p(anchors),
                                      _p(shared_slot), _p(private_slots), _p(write_pos),
                                      _p(read_slot), _p(dev_status), _stream(stream))
    return _check("acache_build_slot_maps", st) if check else st


def acache_write_slots(desc, batch, rows, write_slot, k_new, v_new, k_cache, v_cache, num_slots,
                       private_begin, dev_status=None, stream=None, check=True):
    st = lib().acache_write_slots(ctypes.byref(desc), batch, rows, _p(write_slot), _p(k_new),
                                  _p(v_new), _p(k_cache), _p(v_cache), num_slots, private_begin,
                                  _p(dev_status), _stream(stream))
    return _check("acache_write_slots", st) if check else st


def acache_slot_attention(desc, batch, n_q, q, seq_len, read_slot, k_cache, v_cache, num_slots,
                          out, dev_status=None, stream=None, check=True):
    st = lib().acache_slot_attention(ctypes.byref(desc), batch, n_q, _p(q), seq_len, _p(read_slot),
                                     _p(k_cache), _p(v_cache), num_slots, _p(out), _p(dev_status),
                                     _stream(stream))
    return _check("acache_slot_attention", st) if check else st


def acache_gather_slots(desc, batch, seq_len, read_slot, k_cache, v_cache, num_slots, k_out,
                        v_out, dev_status=None, stream=None, check=True):
    st = lib().acache_gather_slots(ctypes.byref(desc), batch, seq_len, _p(read_slot), _p(k_cache),
                                   _p(v_cache), num_slots, _p(k_out), _p(v_out), _p(dev_status),
                                   _stream(stream))
    return _check("acache_gather_slots", st) if check else st


def acache_kv_deviation_scores(desc, batch, affix_len, k_shared, v_shared, k_full, v_full, scores,
                               stream=None, check=True):
    """High-KV-deviation (CacheBlend-style) scores of one layer, accumulated into `scores`."""
    st = lib().acache_kv_deviation_scores(ctypes.byref(desc), batch, affix_len, _p(k_shared),
                                          _p(v_shared), _p(k_full), _p(v_full), _p(scores),
                                          _stream(stream))
    return _check("acache_kv_deviation_scores", st) if check else st


def acache_slot_attention_dropna(desc, batch, n_q, q, seq_len, read_slot, k_cache, v_cache,
                                 num_slots, out, dev_status=None, stream=None, check=True):
    """Read-slot attention where read_slot entries equal to SLOT_NONE are discarded keys."""
    st = lib().acache_slot_attention_dropna(ctypes.byref(desc), batch, n_q, _p(q), seq_len,
                                            _p(read_slot), _p(k_cache), _p(v_cache), num_slots,
                                            _p(out), _p(dev_status), _stream(stream))
    return _check("acache_slot_attention_dropna", st) if check else st


def acache_slot_attention_path(desc, batch, n_q, seq_len) -> int:
    """The kernel acache_slot_attention runs for this geometry: ACACHE_PATH_RECOMPUTE,
    ACACHE_PATH_RECOMPUTE_PERSISTENT, ACACHE_PATH_BLOCK_DECODE or ACACHE_PATH_CUDA_CORES (see
    include/acache.h)."""
    st = int(lib().acache_slot_attention_path(ctypes.byref(desc), batch, n_q, seq_len))
    return _check("acache_slot_attention_path", st) if st < 0 else st


def acache_slot_attention_varlen(desc, batch, q_start, max_q_rows, total_q_rows, q, kv_start,
                                 max_seq_len, read_slot, k_cache, v_cache, num_slots, out,
                                 drop_none=False, dev_status=None, stream=None, check=True):
    """Read-slot attention over a ragged batch: q_start / kv_start are [B+1] int32 device
    offsets into the flattened query rows and read-slot entries."""
    st = lib().acache_slot_attention_varlen(ctypes.byref(desc), batch, _p(q_start), max_q_rows,
                                            total_q_rows, _p(q), _p(kv_start), max_seq_len,
                                            _p(read_slot), _p(k_cache), _p(v_cache), num_slots, _p(out),
                                            int(bool(drop_none)), _p(dev_status), _stream(stream))
    return _check("acache_slot_attention_varlen", st) if check else st


def _ptr_array(ts, n):
    """Host array of n device pointers (None when ts is None; a None entry is a null pointer)."""
    if ts is None:
        return None
    if len(ts) != n:
        raise ValueError(f"expected {n} per-layer tensors, got {len(ts)}")
    arr = (ctypes.c_void_p * n)(*[None if t is None else t.data_ptr() for t in ts])
    return ctypes.cast(arr, ctypes.c_void_p), arr


def acache_store_attend_layers(desc, batch, rows, write_slot, k_new, v_new, k_cache, v_cache, num_slots,
                               private_begin, n_q, q, seq_len, read_slot, out, dev_status=None, stream=None,
                               check=True):
    """Store-then-attend for every layer of a recompute point in one call (see include/acache.h);
    the per-layer arguments are lists of tensors, one per layer."""
    layers = len(k_cache)
    keep = [_ptr_array(x, layers) for x in (k_new, v_new, k_cache, v_cache, q, out)]
    ptrs = [k[0] if k is not None else None for k in keep]
    st = lib().acache_store_attend_layers(ctypes.byref(desc), layers, batch, rows, _p(write_slot), ptrs[0],
                                          ptrs[1], ptrs[2], ptrs[3], num_slots, private_begin, n_q, ptrs[4],
                                          seq_len, _p(read_slot), ptrs[5], _p(dev_status), _stream(stream))
    del keep
    return _check("acache_store_attend_layers", st) if check else st


def acache_store_attend(desc, batch, rows, write_slot, k_new, v_new, k_cache, v_cache, num_slots,
                        private_begin, n_q, q, seq_len, read_slot, out, dev_status=None, stream=None,
                        check=True):
    """Store step then read-slot attention of one layer in one call (see include/acache.h)."""
    st = lib().acache_store_attend(ctypes.byref(desc), batch, rows, _p(write_slot), _p(k_new), _p(v_new),
                                   _p(k_cache), _p(v_cache), num_slots, private_begin, n_q, _p(q),
                                   seq_len, _p(read_slot), _p(out), _p(dev_status), _stream(stream))
    return _check("acache_store_attend", st) if check else st


def acache_rerotate_keys(desc, rows, k_in, k_out, delta_pos, rope_theta, interleaved=False, stream=None,
                         check=True):
    """Move rotary-embedded keys [rows][Hkv][d] by delta_pos positions (see include/acache.h)."""
    st = lib().acache_rerotate_keys(ctypes.byref(desc), rows, _p(k_in), _p(k_out), int(delta_pos),
                                    float(rope_theta), int(bool(interleaved)), _stream(stream))
    return _check("acache_rerotate_keys", st) if check else st


class Pool:
    """Host-side admission runtime of one KV slot layout (include/acache.h, acache_pool_*):
    the shared-affix registry and the private-page allocator.  Marshalling only."""

    def __init__(self, num_slots, private_begin, page_slots):
        h = ctypes.c_void_p()
        _check("acache_pool_create", lib().acache_pool_create(num_slots, private_begin, page_slots,
                                                              ctypes.byref(h)))
        self._h = h

    def close(self):
        if self._h:
            lib().acache_pool_destroy(self._h)
            self._h = None

    def __del__(self):
        try:
            self.close()
        except Exception:
            pass

    def register_affix(self, key, affix_len):
        """Returns (shared_base, created)."""
        base, created = ctypes.c_int32(), ctypes.c_int32()
        _check("acache_pool_register_affix", lib().acache_pool_register_affix(
            self._h, ctypes.c_uint64(key & (2 ** 64 - 1)), affix_len, ctypes.byref(base), ctypes.byref(created)))
        return base.value, bool(created.value)

    def release_affix(self, key):
        _check("acache_pool_release_affix", lib().acache_pool_release_affix(self._h, ctypes.c_uint64(key & (2 ** 64 - 1))))

    def alloc_private(self, rows):
        """Returns (slots as a CPU int32 tensor [rows], request_id)."""
        slots = torch.empty(rows, dtype=torch.int32)
        rid = ctypes.c_int64()
        _check("acache_pool_alloc_private", lib().acache_pool_alloc_private(
            self._h, rows, ctypes.c_void_p(slots.data_ptr()) if rows else None, ctypes.byref(rid)))
        return slots, rid.value

    def free_private(self, request_id):
        _check("acache_pool_free_private", lib().acache_pool_free_private(self._h, request_id))

    def stats(self):
        fs, fp, na, nr = ctypes.c_int64(), ctypes.c_int64(), ctypes.c_int32(), ctypes.c_int32()
        _check("acache_pool_stats", lib().acache_pool_stats(self._h, ctypes.byref(fs), ctypes.byref(fp),
                                                            ctypes.byref(na), ctypes.byref(nr)))
        return {"free_shared": fs.value, "free_private": fp.value, "affixes": na.value, "requests": nr.value}
