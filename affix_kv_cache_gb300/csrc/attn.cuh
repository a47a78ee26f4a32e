// attn.cuh -- key sources and launch declarations shared by the attention kernels.
#pragma once

#include "common.cuh"

namespace acache {

struct AttnArgs {
    int hq, hkv, d, dtype;
    float scale;
};

// Keys of the read-slot attention: logical key t of request b lives in physical slot
// read_slot[b][t] of the layer's pool (Sec. 4.1, App. C.1).  An out-of-range slot reads
// as a zero row and is flagged.  With drop_none, an entry equal to ACACHE_SLOT_NONE is a
// discarded key (the DropNA ablation, Sec. 5.3): it takes no part in the softmax.
template <typename T>
struct SlotKeys {
    const T* k_cache;
    const T* v_cache;
    const int32_t* read_slot;
    int64_t num_slots;
    int T_len;
    int hkv;
    int d;
    bool drop_none;
    const int32_t* kv_start;   // ragged batches: [B+1] offsets of each request's entries, or null
    ACACHE_DEVFN int64_t base(int b) const { return kv_start ? (int64_t)kv_start[b] : (int64_t)b * T_len; }
    ACACHE_DEVFN int len(int b) const { return kv_start ? kv_start[b + 1] - kv_start[b] : T_len; }
    ACACHE_DEVFN bool dropped(int b, int t) const {
        return drop_none && read_slot[base(b) + t] == ACACHE_SLOT_NONE;
    }
    ACACHE_DEVFN bool rows(int b, int t, int hk, const T*& kr, const T*& vr,
                           int32_t* dev_status) const {
        const int64_t s = read_slot[base(b) + t];
        if (s < 0 || s >= num_slots) {
            flag(dev_status, ACACHE_DEV_BAD_SLOT);
            return false;
        }
        const int64_t off = (s * hkv + hk) * d;
        kr = k_cache + off;
        vr = v_cache + off;
        return true;
    }
    // Element offset of key t's row (same for K and V) in source `src`, or -1 (zero row).
    ACACHE_DEVFN int64_t locate(int b, int t, int hk, int& src, int32_t* dev_status) const {
        src = 0;
        const int64_t s = read_slot[base(b) + t];
        if (s < 0 || s >= num_slots) {
            flag(dev_status, ACACHE_DEV_BAD_SLOT);
            return -1;
        }
        return (s * hkv + hk) * d;
    }
    ACACHE_DEVFN const T* kbase(int) const { return k_cache; }
    ACACHE_DEVFN const T* vbase(int) const { return v_cache; }
};

// Keys of the probe: logical key t is the shared affix row t - l for t in F = [l, l+L),
// otherwise the request's own row (non-affix rows in ascending logical order) (Sec. 3.2).
template <typename T>
struct ProbeKeys {
    const T* k_req;
    const T* v_req;
    const T* k_aff;
    const T* v_aff;
    int l, L, P, hkv, d;
    ACACHE_DEVFN bool dropped(int, int) const { return false; }
    ACACHE_DEVFN int len(int) const { return P + L; }
    ACACHE_DEVFN bool rows(int b, int t, int hk, const T*& kr, const T*& vr, int32_t*) const {
        if (t >= l && t < l + L) {
            const int64_t off = ((int64_t)(t - l) * hkv + hk) * d;
            kr = k_aff + off;
            vr = v_aff + off;
        } else {
            const int pr = t < l ? t : t - L;
            const int64_t off = (((int64_t)b * P + pr) * hkv + hk) * d;
            kr = k_req + off;
            vr = v_req + off;
        }
        return true;
    }
    // source 0 = the shared affix cache, 1 = the request's own rows
    ACACHE_DEVFN int64_t locate(int b, int t, int hk, int& src, int32_t*) const {
        if (t >= l && t < l + L) {
            src = 0;
            return ((int64_t)(t - l) * hkv + hk) * d;
        }
        src = 1;
        const int pr = t < l ? t : t - L;
        return (((int64_t)b * P + pr) * hkv + hk) * d;
    }
    ACACHE_DEVFN const T* kbase(int src) const { return src ? k_req : k_aff; }
    ACACHE_DEVFN const T* vbase(int src) const { return src ? v_req : v_aff; }
};

// ---- the probe of one layer, shared by the entry points that differ only in where the
// scratch lives (a caller's workspace, or the library's fixed array) ------------------------
struct ProbeCall {
    AttnArgs a;
    int B, T, l, L, m;
    const int32_t* masked;
    const void *q, *k_req, *v_req, *k_aff, *v_aff;
    void* out;
    float* scores;
    bool chained = false;   // a later layer of acache_probe_scores_layers (programmatic launch)
};
// Validates a probe call's arguments (errors as acache_probe_scores); on ACACHE_OK, *empty
// says there is nothing to launch, else *c holds the call.
int probe_check(const acache_attn_desc* desc, int batch, int seq_len, int affix_begin, int affix_len,
                const int32_t* masked_rows, int num_masked, const void* q, const void* k_req,
                const void* v_req, const void* k_affix, const void* v_affix, void* out, float* scores,
                ProbeCall* c, bool* empty);
// Scratch bytes of the call: row maximum and row sum [B][Hq][P] and per-head column sums
// [B][Hq][L], float32, each part 256-byte aligned.
size_t probe_scratch_bytes(const ProbeCall& c);
// Launches the probe forward, the masked-to-affix mass and the head sum into c.scores, with the
// scratch at `scratch` (256-byte aligned, probe_scratch_bytes(c) bytes).
int probe_launch(const ProbeCall& c, void* scratch, int32_t* dev_status, cudaStream_t stream);

// ---- launchers (host) ---------------------------------------------------------------
int launch_simt_slot_attention(const AttnArgs& a, int B, int n_q, const void* q, int T_len,
                               const int32_t* read_slot, const void* k_cache, const void* v_cache,
                               int64_t num_slots, void* out, int32_t* dev_status,
                               cudaStream_t stream, bool drop_none = false);
// Ragged batches (see launch_tc_slot_attention_varlen).
int launch_simt_slot_attention_varlen(const AttnArgs& a, int B, const int32_t* q_start, int max_q,
                                      const void* q, const int32_t* kv_start, int max_T,
                                      const int32_t* read_slot, const void* k_cache, const void* v_cache,
                                      int64_t num_slots, void* out, int32_t* dev_status,
                                      cudaStream_t stream, bool drop_none);
int launch_simt_probe_pass_a(const AttnArgs& a, int B, int T_len, int l, int L, const void* q,
                             const void* k_req, const void* v_req, const void* k_aff,
                             const void* v_aff, void* out, float* stat_m, float* stat_l,
                             cudaStream_t stream);
int launch_simt_probe_pass_b(const AttnArgs& a, int B, int T_len, int L, const int32_t* masked_rows,
                             int m, const void* q, const void* k_aff, const float* stat_m,
                             const float* stat_l, float* partial, int32_t* dev_status,
                             cudaStream_t stream);
int launch_score_reduce(int B, int Hq, int L, const float* partial, float* scores,
                        cudaStream_t stream);

int launch_write_slots(int batch, int rows, const int32_t* write_slot, const void* k_new,
                       const void* v_new, void* k_cache, void* v_cache, int64_t row_bytes,
                       int64_t num_slots, int64_t private_begin, int32_t* dev_status,
                       cudaStream_t stream, bool pdl = false);
int launch_gather_slots(int batch, int seq_len, const int32_t* read_slot, const void* k_cache,
                        const void* v_cache, int64_t row_bytes, int64_t num_slots, void* k_out,
                        void* v_out, int32_t* dev_status, cudaStream_t stream);
int launch_build_maps(int batch, int T, int l, int L, int K, const int32_t* anchors,
                      const int32_t* shared_slot, const int32_t* private_slots,
                      int32_t* write_pos, int32_t* read_slot, int32_t* dev_status,
                      cudaStream_t stream);
int launch_topk(const float* scores, int batch, int L, int K, int32_t* anchors,
                int32_t* dev_status, cudaStream_t stream);
int launch_rerotate(int dtype, int64_t rows, int hkv, int d, const void* k_in, void* k_out, int32_t delta,
                    double theta, int interleaved, cudaStream_t stream);
int launch_kv_deviation(int dtype, int B, int L, int Hkv, int d, const void* k_sh, const void* v_sh,
                        const void* k_full, const void* v_full, float* scores, cudaStream_t stream);

}  // namespace acache
