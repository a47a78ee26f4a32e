"""affix_kv_cache_gb300 -- the affix-cache attention hot path on GB300 (sm_103a).

The compute path lives in libacache.so (hand-written CUDA, C ABI in include/acache.h);
``_lib`` is its ctypes binding, ``workloads`` the seeded synthetic-input generator.
Importing the package loads nothing; the library is loaded on first use and a missing
library is an error.
"""
from ._lib import (AcacheError, AttnDesc, attn_desc, acache_build_slot_maps,  # noqa: F401
                   acache_gather_slots, acache_kv_deviation_scores, acache_probe_scores,
                   acache_probe_scores_layers, acache_probe_scores_noalloc,
                   acache_probe_workspace_bytes,
                   acache_slot_attention, acache_slot_attention_dropna, acache_slot_attention_path,
                   acache_slot_attention_varlen,
                   acache_rerotate_keys, acache_store_attend, acache_store_attend_layers, acache_topk_anchors, Pool,
                   acache_wait_budget, acache_write_slots, lib,
                   status_string, version)
