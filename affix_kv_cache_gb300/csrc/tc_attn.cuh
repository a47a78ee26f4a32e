// tc_attn.cuh -- tensor-core (tcgen05 + TMEM) attention kernels for bf16, head_dim 128.
#pragma once

#include <cuda.h>

#include "attn.cuh"

namespace acache {

// bf16 tensor of `rank` dims (innermost first, dims[0] = head_dim), contiguous, 128-byte
// swizzle, box `box` (box[0] = 64: one 128-byte swizzle span); out-of-range elements read as
// zero.  False when the driver entry point is missing or the encoding is rejected.
bool make_map_box(CUtensorMap* m, const void* ptr, int rank, const uint64_t* dims, const uint32_t* box);
// The same with box {64, 1, ..., box_rows at dimension row_dim, 1, ...}.
bool make_map(CUtensorMap* m, const void* ptr, int rank, const uint64_t* dims, int row_dim,
              uint32_t box_rows);

// True when the tcgen05 kernels cover this geometry (bf16, head_dim 128).
bool tc_supported(const AttnArgs& a);
// True when launch_tc_slot_attention (no discarded keys) runs the persistent kernel: more
// 256-row query blocks of a (request, head) than SMs, and short units (at most 20 key tiles) or
// one query tile per unit (at most 128 query rows).
bool tc_slot_persistent(const AttnArgs& a, int B, int n_q, int T_len);

// drop_none: read-slot entries equal to ACACHE_SLOT_NONE are discarded keys (DropNA).
int launch_tc_slot_attention(const AttnArgs& a, int B, int n_q, const void* q, int T_len,
                             const int32_t* read_slot, const void* k_cache, const void* v_cache,
                             int64_t num_slots, void* out, int32_t* dev_status,
                             cudaStream_t stream, bool drop_none = false, bool pdl = false,
                             bool chained = false);
// Ragged batches: request b's query rows are [q_start[b], q_start[b+1]) of q / out
// ([total_q][Hq][d]) and its logical keys read_slot[kv_start[b] .. kv_start[b+1]); max_q and
// max_T bound the per-request counts (a request outside them is skipped and flagged).
int launch_tc_slot_attention_varlen(const AttnArgs& a, int B, const int32_t* q_start, int max_q,
                                    int total_q, const void* q, const int32_t* kv_start, int max_T,
                                    const int32_t* read_slot, const void* k_cache, const void* v_cache,
                                    int64_t num_slots, void* out, int32_t* dev_status,
                                    cudaStream_t stream, bool drop_none);
// Block-decode form of the read-slot attention (few query rows per KV head): true when it
// streams fewer K/V tiles than the recompute-point kernel for this geometry, or as many and
// the streams would leave most SMs idle (its cluster split of the keys fills them).
bool tc_decode_preferred(const AttnArgs& a, int B, int n_q, int T_len);
int launch_tc_decode_attention(const AttnArgs& a, int B, int n_q, const void* q, int T_len,
                               const int32_t* read_slot, const void* k_cache, const void* v_cache,
                               int64_t num_slots, void* out, int32_t* dev_status, cudaStream_t stream,
                               bool drop_none = false, bool pdl = false);
int launch_tc_probe_pass_a(const AttnArgs& a, int B, int T_len, int l, int L, const void* q,
                           const void* k_req, const void* v_req, const void* k_aff,
                           const void* v_aff, void* out, float* stat_m, float* stat_l,
                           int32_t* dev_status, cudaStream_t stream, bool chained = false);
int launch_tc_probe_pass_b(const AttnArgs& a, int B, int T_len, int L, const int32_t* masked_rows,
                           int m, const void* q, const void* k_aff, const float* stat_m,
                           const float* stat_l, float* partial, int32_t* dev_status,
                           cudaStream_t stream);

}  // namespace acache
