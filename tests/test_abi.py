"""The C ABI on a host without a GPU: symbols, host-side validation, workspace sizing.

None of these calls reaches a kernel launch: every one is rejected (or is a no-op) by the
host-side argument checks before any CUDA call.
"""
import ctypes
import os
import re

import pytest

import affix_kv_cache_gb300 as ac
from affix_kv_cache_gb300 import _lib

HEADER = os.path.join(os.path.dirname(os.path.dirname(__file__)), "include", "acache.h")
BOGUS = 1 << 40          # a non-null pointer value that is never dereferenced here


def declared_functions():
    src = open(HEADER).read()
    return re.findall(r"ACACHE_API\s+[\w\s\*]+?\b(acache_\w+)\s*\(", src)


def test_library_exports_every_declared_symbol():
    names = declared_functions()
    assert set(names) == set(_lib.EXPORTS), names
    L = ac.lib()
    for n in names:
        assert getattr(L, n) is not None
    assert ac.version() == 200
    assert ac.status_string(0) == "ok"


def test_binding_constants_match_header():
    """Every ACACHE_* enumerator and #define of the header has the same value in the binding
    (status codes, dtypes, device-status bits, kernel paths, the discarded-key sentinel)."""
    src = open(HEADER).read()
    found = dict((n, int(v)) for n, v in re.findall(r"\b(ACACHE_[A-Z0-9_]+)\s*=\s*(-?\d+)", src))
    found.update((n, int(v)) for n, v in re.findall(r"#define\s+(ACACHE_[A-Z0-9_]+)\s+\((-?\d+)\)", src))
    assert len(found) >= 20, sorted(found)
    for name, value in found.items():
        py = name if hasattr(_lib, name) else name.replace("ACACHE_", "", 1)
        assert getattr(_lib, py) == value, (name, getattr(_lib, py), value)


def test_wait_budget_set_and_read_on_the_host():
    # host-side state only: no kernel is launched
    default = ac.acache_wait_budget()
    assert default == 1 << 31
    assert ac.acache_wait_budget(12345) == default
    assert ac.acache_wait_budget(0) == 12345          # <= 0 reads without setting
    assert ac.acache_wait_budget(-7) == 12345
    assert ac.acache_wait_budget(default) == 12345
    assert ac.acache_wait_budget() == default


def test_struct_layout_matches_header():
    assert ctypes.sizeof(_lib.AttnDesc) == 20


def desc(hq=4, hkv=2, d=128, dtype="bf16", scale=0.088):
    return ac.attn_desc(hq, hkv, d, scale, dtype)


def test_descriptor_validation():
    L = ac.lib()
    bad = [(ac.attn_desc(3, 2, 128, 0.1, "bf16"), _lib.ACACHE_ERR_INVALID_ARG),
           (ac.attn_desc(0, 1, 128, 0.1, "bf16"), _lib.ACACHE_ERR_INVALID_ARG),
           (ac.attn_desc(4, 2, 96, 0.1, "bf16"), _lib.ACACHE_ERR_UNSUPPORTED),
           (_lib.AttnDesc(4, 2, 128, 0.1, 7), _lib.ACACHE_ERR_UNSUPPORTED),
           (ac.attn_desc(4, 2, 128, float("nan"), "bf16"), _lib.ACACHE_ERR_INVALID_ARG)]
    for dsc, want in bad:
        st = L.acache_slot_attention(ctypes.byref(dsc), 1, 1, BOGUS, 4, BOGUS, BOGUS, BOGUS, 8,
                                     BOGUS, None, None)
        assert st == want
    assert L.acache_slot_attention(None, 1, 1, BOGUS, 4, BOGUS, BOGUS, BOGUS, 8, BOGUS, None,
                                   None) == _lib.ACACHE_ERR_INVALID_ARG


def test_empty_work_is_a_noop():
    L = ac.lib()
    d = desc()
    assert L.acache_slot_attention(ctypes.byref(d), 0, 5, None, 4, None, None, None, 0, None, None, None) == 0
    assert L.acache_slot_attention(ctypes.byref(d), 2, 0, None, 4, None, None, None, 0, None, None, None) == 0
    assert L.acache_write_slots(ctypes.byref(d), 2, 0, None, None, None, None, None, 0, 0, None, None) == 0
    assert L.acache_topk_anchors(None, 3, 10, 0, None, None, None) == 0
    assert L.acache_gather_slots(ctypes.byref(d), 0, 9, None, None, None, 0, None, None, None, None) == 0
    # a probe with no probe rows (the whole sequence is the affix) attends nothing
    assert L.acache_probe_scores(ctypes.byref(d), 2, 16, 0, 16, None, 0, None, None, None, None,
                                 None, None, None, None, 0, None, None) == 0


def test_scalar_validation():
    L = ac.lib()
    d = desc()
    E = _lib.ACACHE_ERR_INVALID_ARG
    assert L.acache_topk_anchors(BOGUS, 1, 10, 11, BOGUS, None, None) == E      # K > L
    assert L.acache_topk_anchors(BOGUS, 1, 10, -1, BOGUS, None, None) == E
    assert L.acache_topk_anchors(None, 1, 10, 3, BOGUS, None, None) == E
    assert L.acache_build_slot_maps(1, 10, 4, 7, 2, BOGUS, BOGUS, BOGUS, BOGUS, BOGUS, None, None) == E  # l+L > T
    assert L.acache_build_slot_maps(1, 10, 0, 7, 8, BOGUS, BOGUS, BOGUS, BOGUS, BOGUS, None, None) == E  # K > L
    assert L.acache_build_slot_maps(1, 10, 0, 7, 2, None, BOGUS, BOGUS, BOGUS, BOGUS, None, None) == E
    assert L.acache_write_slots(ctypes.byref(d), 1, 4, BOGUS, BOGUS, BOGUS, BOGUS, BOGUS, 10, 11, None, None) == E
    assert L.acache_write_slots(ctypes.byref(d), 1, 4, None, BOGUS, BOGUS, BOGUS, BOGUS, 10, 2, None, None) == E
    assert L.acache_write_slots(ctypes.byref(d), 1, 4, BOGUS, BOGUS + 8, BOGUS, BOGUS, BOGUS, 10, 2, None, None) == E  # misaligned
    assert L.acache_slot_attention(ctypes.byref(d), 1, 4, BOGUS, 0, BOGUS, BOGUS, BOGUS, 8, BOGUS, None, None) == E  # T = 0
    # probe: m > P, l + L > T, bad masked pointer
    assert L.acache_probe_scores(ctypes.byref(d), 1, 16, 0, 8, BOGUS, 9, BOGUS, BOGUS, BOGUS, BOGUS,
                                 BOGUS, None, BOGUS, BOGUS, 1 << 30, None, None) == E
    assert L.acache_probe_scores(ctypes.byref(d), 1, 16, 10, 8, BOGUS, 2, BOGUS, BOGUS, BOGUS, BOGUS,
                                 BOGUS, None, BOGUS, BOGUS, 1 << 30, None, None) == E
    assert L.acache_probe_scores(ctypes.byref(d), 1, 16, 0, 8, None, 2, BOGUS, BOGUS, BOGUS, BOGUS,
                                 BOGUS, None, BOGUS, BOGUS, 1 << 30, None, None) == E


def test_probe_workspace_sizing_and_check():
    L = ac.lib()
    d = desc(hq=32, hkv=32)
    B, T, Lf = 4, 1408, 1024
    need = ac.acache_probe_workspace_bytes(d, B, T, Lf, 256)
    P = T - Lf
    st = -(-(B * 32 * P * 4) // 256) * 256
    pa = -(-(B * 32 * Lf * 4) // 256) * 256
    assert need == 2 * st + pa
    st_code = L.acache_probe_scores(ctypes.byref(d), B, T, 0, Lf, BOGUS, 256, BOGUS, BOGUS, BOGUS,
                                    BOGUS, BOGUS, None, BOGUS, BOGUS, need - 1, None, None)
    assert st_code == _lib.ACACHE_ERR_WORKSPACE
    st_code = L.acache_probe_scores(ctypes.byref(d), B, T, 0, Lf, BOGUS, 256, BOGUS, BOGUS, BOGUS,
                                    BOGUS, BOGUS, None, BOGUS, None, need, None, None)
    assert st_code == _lib.ACACHE_ERR_WORKSPACE


def test_binding_raises_on_error():
    with pytest.raises(ac.AcacheError) as e:
        ac.acache_topk_anchors(None, 1, 10, 3, None)
    assert e.value.status == _lib.ACACHE_ERR_INVALID_ARG


def test_slot_attention_path_choice():
    """Host-only: which kernel the read-slot attention picks for a geometry."""
    path = lambda hq, hkv, B, n_q, T, dt="bf16", d=128: ac.acache_slot_attention_path(  # noqa: E731
        ac.attn_desc(hq, hkv, d, d ** -0.5, dt), B, n_q, T)
    # a recompute point: 384 blocks of 256 query rows (more than SMs) of 11-20 key tiles run
    # persistent; 96 blocks, or 1,536 blocks of 35 key tiles, do not
    assert path(32, 32, 4, 589, 1408) == _lib.ACACHE_PATH_RECOMPUTE_PERSISTENT
    assert path(32, 32, 1, 589, 1408) == _lib.ACACHE_PATH_RECOMPUTE
    assert path(32, 32, 16, 1204, 4480) == _lib.ACACHE_PATH_RECOMPUTE
    assert path(32, 32, 16, 32, 4480) == _lib.ACACHE_PATH_RECOMPUTE_PERSISTENT   # 512 one-tile blocks
    assert path(32, 32, 16, 129, 4480) == _lib.ACACHE_PATH_RECOMPUTE
    assert path(32, 32, 4, 589, 2560) == _lib.ACACHE_PATH_RECOMPUTE_PERSISTENT
    assert path(32, 32, 4, 589, 2561) == _lib.ACACHE_PATH_RECOMPUTE
    assert path(32, 32, 4, 32, 1408) == _lib.ACACHE_PATH_RECOMPUTE       # decode, 128 streams
    assert path(32, 32, 1, 32, 1408) == _lib.ACACHE_PATH_BLOCK_DECODE    # decode, 32 streams
    assert path(28, 4, 16, 32, 2624) == _lib.ACACHE_PATH_BLOCK_DECODE    # GQA group shares a stream
    assert path(2, 2, 1, 32, 100, "f32", 64) == _lib.ACACHE_PATH_CUDA_CORES
    assert path(8, 8, 1, 32, 100, "bf16", 64) == _lib.ACACHE_PATH_CUDA_CORES
    with pytest.raises(ac.AcacheError):
        path(3, 2, 1, 32, 100)                                            # Hq % Hkv != 0


def test_probe_layers_host_validation():
    """Host-only checks of acache_probe_scores_layers: nothing is launched on bad input."""
    L = ac.lib()
    d = desc(hq=4, hkv=2)
    E, W = _lib.ACACHE_ERR_INVALID_ARG, _lib.ACACHE_ERR_WORKSPACE
    arr = (ctypes.c_void_p * 3)(BOGUS, BOGUS, BOGUS)
    bad = (ctypes.c_void_p * 3)(BOGUS, BOGUS + 8, BOGUS)        # layer 1's pointer misaligned
    nul = (ctypes.c_void_p * 3)(BOGUS, None, BOGUS)             # layer 1's pointer missing
    args = lambda q, n=3, ws=1 << 30: (ctypes.byref(d), n, 2, 64, 0, 32, BOGUS, 16, q, arr, arr, arr, arr,  # noqa: E731
                                       None, BOGUS, BOGUS, ws, None, None)
    assert L.acache_probe_scores_layers(*args(arr, n=-1)) == E
    assert L.acache_probe_scores_layers(*args(arr, n=0)) == _lib.ACACHE_OK     # nothing to do
    assert L.acache_probe_scores_layers(*args(None)) == E                      # no query array
    assert L.acache_probe_scores_layers(*args(bad)) == E
    assert L.acache_probe_scores_layers(*args(nul)) == E
    assert L.acache_probe_scores_layers(*args(arr, ws=16)) == W
