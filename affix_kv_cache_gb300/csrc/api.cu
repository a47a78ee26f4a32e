// api.cu -- the C ABI of libacache.so: argument validation, workspace carving and kernel
// dispatch.  Every entry point is declared and documented in include/acache.h.
#include <math.h>

#include <atomic>
#include <vector>

#include "attn.cuh"
#include "ptx.cuh"
#include "tc_attn.cuh"

namespace acache {

int sm_count() {
    static int cache[64] = {0};
    int dev = 0;
    if (cudaGetDevice(&dev) != cudaSuccess || dev < 0 || dev >= 64) return 148;
    if (!cache[dev]) {
        int n = 0;
        if (cudaDeviceGetAttribute(&n, cudaDevAttrMultiProcessorCount, dev) != cudaSuccess || n <= 0)
            n = 148;
        cache[dev] = n;
    }
    return cache[dev];
}

int launch_status() {
    const cudaError_t e = cudaGetLastError();
    return e == cudaSuccess ? ACACHE_OK : ACACHE_ERR_CUDA;
}

namespace {
constexpr long long kDefaultWaitBudget = 1LL << 31;   // SM clock cycles: about 1 s at 2.07 GHz
std::atomic<long long> g_wait_budget{kDefaultWaitBudget};
}  // namespace

long long wait_budget() { return g_wait_budget.load(std::memory_order_relaxed); }

namespace {

constexpr size_t kAlign = 256;
size_t align_up(size_t x) { return (x + kAlign - 1) / kAlign * kAlign; }

bool aligned16(const void* p) { return ((uintptr_t)p & 15u) == 0; }

// Validates the attention descriptor; fills `out`.
int check_desc(const acache_attn_desc* a, AttnArgs* out) {
    if (!a) return ACACHE_ERR_INVALID_ARG;
    if (a->num_q_heads <= 0 || a->num_kv_heads <= 0 || a->num_q_heads % a->num_kv_heads)
        return ACACHE_ERR_INVALID_ARG;
    if (!(a->scale == a->scale) || isinf(a->scale)) return ACACHE_ERR_INVALID_ARG;
    if (a->dtype != ACACHE_F32 && a->dtype != ACACHE_BF16) return ACACHE_ERR_UNSUPPORTED;
    if (a->head_dim != 64 && a->head_dim != 128) return ACACHE_ERR_UNSUPPORTED;
    *out = AttnArgs{a->num_q_heads, a->num_kv_heads, a->head_dim, a->dtype, a->scale};
    return ACACHE_OK;
}

size_t elem_bytes(int dtype) { return dtype == ACACHE_F32 ? 4 : 2; }

struct ProbeWorkspace {
    float* stat_m;
    float* stat_l;
    float* partial;
    size_t bytes;
};

ProbeWorkspace carve_probe_ws(void* base, int64_t B, int64_t Hq, int64_t P, int64_t L) {
    ProbeWorkspace w{};
    const size_t st = align_up((size_t)(B * Hq * P) * sizeof(float));
    const size_t pa = align_up((size_t)(B * Hq * L) * sizeof(float));
    char* p = (char*)base;
    w.stat_m = (float*)p;
    w.stat_l = (float*)(p + st);
    w.partial = (float*)(p + 2 * st);
    w.bytes = 2 * st + pa;
    return w;
}

// scores[b][j] += sum over heads h (ascending) of partial[b][h][j].  Launched behind the mass
// pass (programmatic dependent launch): it waits for it before reading the partial sums, and
// lets the next layer's probe forward start at once.
__global__ void score_reduce_kernel(int B, int Hq, int L, const float* __restrict__ partial,
                                    float* __restrict__ scores) {
    ptx::grid_launch_dependents();
    ptx::grid_dependency_wait();
    const int64_t gid = (int64_t)blockIdx.x * blockDim.x + threadIdx.x;
    if (gid >= (int64_t)B * L) return;
    const int64_t b = gid / L, j = gid % L;
    float acc = scores[gid];
    for (int h = 0; h < Hq; ++h) acc += partial[(b * Hq + h) * L + j];
    scores[gid] = acc;
}

}  // namespace

int launch_score_reduce(int B, int Hq, int L, const float* partial, float* scores,
                        cudaStream_t stream) {
    const int64_t n = (int64_t)B * L;
    if (n == 0) return ACACHE_OK;
    cudaLaunchConfig_t cfg = {};
    cfg.gridDim = dim3((unsigned)((n + 255) / 256));
    cfg.blockDim = dim3(256);
    cfg.stream = stream;
    cudaLaunchAttribute attr[1];
    attr[0].id = cudaLaunchAttributeProgrammaticStreamSerialization;
    attr[0].val.programmaticStreamSerializationAllowed = 1;
    cfg.attrs = attr;
    cfg.numAttrs = 1;
    if (cudaLaunchKernelEx(&cfg, score_reduce_kernel, B, Hq, L, partial, scores) != cudaSuccess) {
        (void)cudaGetLastError();
        return ACACHE_ERR_CUDA;
    }
    return launch_status();
}

}  // namespace acache

namespace acache {
namespace {
int slot_attention(const acache_attn_desc* desc, int batch, int n_q, const void* q, int seq_len,
                   const int32_t* read_slot, const void* k_cache, const void* v_cache,
                   int64_t num_slots, void* out, int32_t* dev_status, void* stream_, bool drop_none,
                   bool after_store = false) {
    AttnArgs a;
    if (int rc = check_desc(desc, &a)) return rc;
    if (batch < 0 || n_q < 0 || seq_len < 0 || num_slots < 0) return ACACHE_ERR_INVALID_ARG;
    if (batch == 0 || n_q == 0) return ACACHE_OK;
    if (seq_len == 0) return ACACHE_ERR_INVALID_ARG;       // a softmax over no keys
    if (!q || !read_slot || !k_cache || !v_cache || !out) return ACACHE_ERR_INVALID_ARG;
    if (!aligned16(q) || !aligned16(k_cache) || !aligned16(v_cache) || !aligned16(out))
        return ACACHE_ERR_INVALID_ARG;
    cudaStream_t stream = (cudaStream_t)stream_;
    if (tc_supported(a)) {
        // few query rows per KV head (the block-decode step): the kernel that packs a GQA
        // group's heads into one K/V stream and splits the keys over a cluster
        if (tc_decode_preferred(a, batch, n_q, seq_len))
            return launch_tc_decode_attention(a, batch, n_q, q, seq_len, read_slot, k_cache, v_cache,
                                              num_slots, out, dev_status, stream, drop_none, after_store);
        return launch_tc_slot_attention(a, batch, n_q, q, seq_len, read_slot, k_cache, v_cache,
                                        num_slots, out, dev_status, stream, drop_none, after_store);
    }
    return launch_simt_slot_attention(a, batch, n_q, q, seq_len, read_slot, k_cache, v_cache,
                                      num_slots, out, dev_status, stream, drop_none);
}
}  // namespace
}  // namespace acache

namespace acache {

int probe_check(const acache_attn_desc* desc, int batch, int seq_len, int affix_begin, int affix_len,
                const int32_t* masked_rows, int num_masked, const void* q, const void* k_req,
                const void* v_req, const void* k_affix, const void* v_affix, void* out, float* scores,
                ProbeCall* c, bool* empty) {
    AttnArgs a;
    if (int rc = check_desc(desc, &a)) return rc;
    const int T = seq_len, l = affix_begin, L = affix_len, m = num_masked;
    if (batch < 0 || T < 0 || l < 0 || L < 0 || (int64_t)l + L > T || m < 0 || m > T - L)
        return ACACHE_ERR_INVALID_ARG;
    *empty = batch == 0 || T == L;      // no probe rows: nothing attends
    if (*empty) return ACACHE_OK;
    if (!q || !k_req || !v_req || (L > 0 && (!k_affix || !v_affix)) || (m > 0 && !masked_rows) ||
        (L > 0 && !scores))
        return ACACHE_ERR_INVALID_ARG;
    if (!aligned16(q) || !aligned16(k_req) || !aligned16(v_req) || !aligned16(k_affix) ||
        !aligned16(v_affix) || !aligned16(out))
        return ACACHE_ERR_INVALID_ARG;
    *c = ProbeCall{a, batch, T, l, L, m, masked_rows, q, k_req, v_req, k_affix, v_affix, out, scores};
    return ACACHE_OK;
}

size_t probe_scratch_bytes(const ProbeCall& c) {
    return carve_probe_ws(nullptr, c.B, c.a.hq, c.T - c.L, c.L).bytes;
}

int probe_launch(const ProbeCall& c, void* scratch, int32_t* dev_status, cudaStream_t stream) {
    const AttnArgs& a = c.a;
    const ProbeWorkspace ws = carve_probe_ws(scratch, c.B, a.hq, c.T - c.L, c.L);
    int rc;
    if (tc_supported(a)) {
        rc = launch_tc_probe_pass_a(a, c.B, c.T, c.l, c.L, c.q, c.k_req, c.v_req, c.k_aff, c.v_aff, c.out,
                                    ws.stat_m, ws.stat_l, dev_status, stream, c.chained);
    } else {
        rc = launch_simt_probe_pass_a(a, c.B, c.T, c.l, c.L, c.q, c.k_req, c.v_req, c.k_aff, c.v_aff, c.out,
                                      ws.stat_m, ws.stat_l, stream);
    }
    if (rc) return rc;
    if (c.L == 0) return ACACHE_OK;
    if (tc_supported(a)) {
        rc = launch_tc_probe_pass_b(a, c.B, c.T, c.L, c.masked, c.m, c.q, c.k_aff, ws.stat_m, ws.stat_l,
                                    ws.partial, dev_status, stream);
    } else {
        rc = launch_simt_probe_pass_b(a, c.B, c.T, c.L, c.masked, c.m, c.q, c.k_aff, ws.stat_m, ws.stat_l,
                                      ws.partial, dev_status, stream);
    }
    if (rc) return rc;
    return launch_score_reduce(c.B, a.hq, c.L, ws.partial, c.scores, stream);
}

}  // namespace acache

using namespace acache;

extern "C" {

const char* acache_status_string(int status) {
    switch (status) {
        case ACACHE_OK: return "ok";
        case ACACHE_ERR_INVALID_ARG: return "invalid argument";
        case ACACHE_ERR_UNSUPPORTED: return "unsupported dtype/head_dim";
        case ACACHE_ERR_CUDA: return "CUDA launch error";
        case ACACHE_ERR_WORKSPACE: return "workspace too small";
        case ACACHE_ERR_TIMEOUT: return "bounded wait timed out";
        default: return "unknown status";
    }
}

int acache_version(void) { return 200; }   // 0.2.0

int64_t acache_wait_budget(int64_t cycles) {
    if (cycles > 0) return g_wait_budget.exchange(cycles);
    return g_wait_budget.load();
}

size_t acache_probe_workspace_bytes(const acache_attn_desc* a, int batch, int seq_len,
                                    int affix_len, int num_masked) {
    (void)num_masked;
    if (!a || batch < 0 || affix_len < 0 || seq_len < affix_len || a->num_q_heads <= 0) return 0;
    return carve_probe_ws(nullptr, batch, a->num_q_heads, seq_len - affix_len, affix_len).bytes;
}

int acache_probe_scores(const acache_attn_desc* desc, int batch, int seq_len, int affix_begin,
                        int affix_len, const int32_t* masked_rows, int num_masked,
                        const void* q, const void* k_req, const void* v_req,
                        const void* k_affix, const void* v_affix, void* out, float* scores,
                        void* workspace, size_t workspace_bytes, int32_t* dev_status,
                        void* stream_) {
    ProbeCall c;
    bool empty = false;
    if (int rc = probe_check(desc, batch, seq_len, affix_begin, affix_len, masked_rows, num_masked, q, k_req,
                             v_req, k_affix, v_affix, out, scores, &c, &empty))
        return rc;
    if (empty) return ACACHE_OK;
    if (!workspace || workspace_bytes < probe_scratch_bytes(c)) return ACACHE_ERR_WORKSPACE;
    if ((uintptr_t)workspace & 255u) return ACACHE_ERR_INVALID_ARG;
    return probe_launch(c, workspace, dev_status, (cudaStream_t)stream_);
}

int acache_probe_scores_layers(const acache_attn_desc* desc, int layers, int batch, int seq_len,
                               int affix_begin, int affix_len, const int32_t* masked_rows, int num_masked,
                               const void* const* q, const void* const* k_req, const void* const* v_req,
                               const void* const* k_affix, const void* const* v_affix, void* const* out,
                               float* scores, void* workspace, size_t workspace_bytes, int32_t* dev_status,
                               void* stream_) {
    if (layers < 0) return ACACHE_ERR_INVALID_ARG;
    if (layers == 0) return ACACHE_OK;
    if (!q || !k_req || !v_req || (affix_len > 0 && (!k_affix || !v_affix))) return ACACHE_ERR_INVALID_ARG;
    // every layer's arguments are checked before anything is launched
    std::vector<ProbeCall> calls((size_t)layers);
    bool empty = false;
    for (int n = 0; n < layers; ++n)
        if (int rc = probe_check(desc, batch, seq_len, affix_begin, affix_len, masked_rows, num_masked, q[n],
                                 k_req[n], v_req[n], k_affix ? k_affix[n] : nullptr,
                                 v_affix ? v_affix[n] : nullptr, out ? out[n] : nullptr, scores,
                                 &calls[(size_t)n], &empty))
            return rc;
    if (empty) return ACACHE_OK;
    const ProbeCall& c0 = calls[0];
    if (!workspace || workspace_bytes < probe_scratch_bytes(c0)) return ACACHE_ERR_WORKSPACE;
    if ((uintptr_t)workspace & 255u) return ACACHE_ERR_INVALID_ARG;
    // A chained forward reads its layer's inputs before the grids ahead of it are complete:
    // chain only when nothing the call writes (any layer's output, the scores, the workspace)
    // meets any layer's inputs.
    const int64_t eb = elem_bytes(c0.a.dtype), P = c0.T - c0.L;
    const int64_t qo_bytes = (int64_t)c0.B * P * c0.a.hq * c0.a.d * eb;
    const int64_t req_bytes = (int64_t)c0.B * P * c0.a.hkv * c0.a.d * eb;
    const int64_t aff_bytes = (int64_t)c0.L * c0.a.hkv * c0.a.d * eb;
    struct Range {
        uintptr_t lo, hi;
    };
    auto span = [](const void* ptr, int64_t bytes) {
        return Range{(uintptr_t)ptr, ptr ? (uintptr_t)ptr + (uintptr_t)bytes : (uintptr_t)ptr};
    };
    std::vector<Range> written = {span(scores, (int64_t)c0.B * c0.L * 4),
                                  span(workspace, (int64_t)probe_scratch_bytes(c0))};
    for (const ProbeCall& c : calls) written.push_back(span(c.out, qo_bytes));
    bool disjoint = true;
    for (const ProbeCall& c : calls) {
        const Range read[5] = {span(c.q, qo_bytes), span(c.k_req, req_bytes), span(c.v_req, req_bytes),
                               span(c.k_aff, aff_bytes), span(c.v_aff, aff_bytes)};
        for (const Range& x : written)
            for (const Range& y : read)
                if (x.lo < x.hi && y.lo < y.hi && x.lo < y.hi && y.lo < x.hi) disjoint = false;
    }
    cudaStream_t st = (cudaStream_t)stream_;
    for (int n = 0; n < layers; ++n) {
        ProbeCall& c = calls[(size_t)n];
        c.chained = disjoint && n > 0;
        if (int rc = probe_launch(c, workspace, dev_status, st)) return rc;
    }
    return ACACHE_OK;
}

int acache_slot_attention_path(const acache_attn_desc* desc, int batch, int n_q, int seq_len) {
    AttnArgs a;
    if (int rc = check_desc(desc, &a)) return rc;
    if (batch < 0 || n_q < 0 || seq_len < 0) return ACACHE_ERR_INVALID_ARG;
    if (!tc_supported(a)) return ACACHE_PATH_CUDA_CORES;
    if (tc_decode_preferred(a, batch, n_q, seq_len)) return ACACHE_PATH_BLOCK_DECODE;
    return tc_slot_persistent(a, batch, n_q, seq_len) ? ACACHE_PATH_RECOMPUTE_PERSISTENT : ACACHE_PATH_RECOMPUTE;
}

int acache_topk_anchors(const float* scores, int batch, int affix_len, int k, int32_t* anchors,
                        int32_t* dev_status, void* stream) {
    if (batch < 0 || affix_len < 0 || k < 0 || k > affix_len) return ACACHE_ERR_INVALID_ARG;
    if (batch == 0 || k == 0) return ACACHE_OK;
    if (!scores || !anchors) return ACACHE_ERR_INVALID_ARG;
    return launch_topk(scores, batch, affix_len, k, anchors, dev_status, (cudaStream_t)stream);
}

int acache_kv_deviation_scores(const acache_attn_desc* desc, int batch, int affix_len,
                               const void* k_shared, const void* v_shared, const void* k_full,
                               const void* v_full, float* scores, void* stream) {
    AttnArgs a;
    if (int rc = check_desc(desc, &a)) return rc;
    if (batch < 0 || affix_len < 0) return ACACHE_ERR_INVALID_ARG;
    if (batch == 0 || affix_len == 0) return ACACHE_OK;
    if (!k_shared || !v_shared || !k_full || !v_full || !scores) return ACACHE_ERR_INVALID_ARG;
    if (!aligned16(k_shared) || !aligned16(v_shared) || !aligned16(k_full) || !aligned16(v_full))
        return ACACHE_ERR_INVALID_ARG;
    return launch_kv_deviation(a.dtype, batch, affix_len, a.hkv, a.d, k_shared, v_shared, k_full,
                               v_full, scores, (cudaStream_t)stream);
}

int acache_rerotate_keys(const acache_attn_desc* desc, int64_t rows, const void* k_in, void* k_out,
                         int32_t delta_pos, double rope_theta, int interleaved, void* stream) {
    AttnArgs a;
    if (int rc = check_desc(desc, &a)) return rc;
    if (rows < 0 || !(rope_theta > 0.0) || isinf(rope_theta)) return ACACHE_ERR_INVALID_ARG;
    if (rows == 0) return ACACHE_OK;
    if (!k_in || !k_out || !aligned16(k_in) || !aligned16(k_out)) return ACACHE_ERR_INVALID_ARG;
    return launch_rerotate(a.dtype, rows, a.hkv, a.d, k_in, k_out, delta_pos, rope_theta, interleaved != 0,
                           (cudaStream_t)stream);
}

int acache_build_slot_maps(int batch, int seq_len, int affix_begin, int affix_len, int k,
                           const int32_t* anchors, const int32_t* shared_slot,
                           const int32_t* private_slots, int32_t* write_pos, int32_t* read_slot,
                           int32_t* dev_status, void* stream) {
    const int T = seq_len, l = affix_begin, L = affix_len;
    if (batch < 0 || T < 0 || l < 0 || L < 0 || (int64_t)l + L > T || k < 0 || k > L)
        return ACACHE_ERR_INVALID_ARG;
    if (batch == 0 || T == 0) return ACACHE_OK;
    const int R = k + T - L;
    if ((k > 0 && !anchors) || (L > k && !shared_slot) || (R > 0 && (!private_slots || !write_pos)) ||
        !read_slot)
        return ACACHE_ERR_INVALID_ARG;
    return launch_build_maps(batch, T, l, L, k, anchors, shared_slot, private_slots, write_pos,
                             read_slot, dev_status, (cudaStream_t)stream);
}

int acache_store_attend(const acache_attn_desc* desc, int batch, int rows, const int32_t* write_slot,
                        const void* k_new, const void* v_new, void* k_cache, void* v_cache,
                        int64_t num_slots, int64_t private_begin, int n_q, const void* q, int seq_len,
                        const int32_t* read_slot, void* out, int32_t* dev_status, void* stream) {
    AttnArgs a;
    if (int rc = check_desc(desc, &a)) return rc;
    // validate both halves before launching either
    if (batch < 0 || rows < 0 || n_q < 0 || seq_len < 0 || num_slots < 0 || private_begin < 0 ||
        private_begin > num_slots)
        return ACACHE_ERR_INVALID_ARG;
    if (batch == 0) return ACACHE_OK;
    const bool store = rows > 0, attend = n_q > 0;
    if (store && (!write_slot || !k_new || !v_new || !aligned16(k_new) || !aligned16(v_new)))
        return ACACHE_ERR_INVALID_ARG;
    if (attend && (seq_len == 0 || !q || !read_slot || !out || !aligned16(q) || !aligned16(out)))
        return ACACHE_ERR_INVALID_ARG;
    if ((store || attend) && (!k_cache || !v_cache || !aligned16(k_cache) || !aligned16(v_cache)))
        return ACACHE_ERR_INVALID_ARG;
    if (store) {
        const int64_t row_bytes = (int64_t)a.hkv * a.d * elem_bytes(a.dtype);
        if (int rc = launch_write_slots(batch, rows, write_slot, k_new, v_new, k_cache, v_cache, row_bytes,
                                        num_slots, private_begin, dev_status, (cudaStream_t)stream))
            return rc;
    }
    if (!attend) return ACACHE_OK;
    // the tensor-core attention starts its prologue while the store drains (programmatic
    // dependent launch); its producers wait for the store before reading the pool
    return slot_attention(desc, batch, n_q, q, seq_len, read_slot, k_cache, v_cache, num_slots, out,
                          dev_status, stream, false, store && tc_supported(a));
}

int acache_store_attend_layers(const acache_attn_desc* desc, int layers, int batch, int rows,
                               const int32_t* write_slot, const void* const* k_new, const void* const* v_new,
                               void* const* k_cache, void* const* v_cache, int64_t num_slots,
                               int64_t private_begin, int n_q, const void* const* q, int seq_len,
                               const int32_t* read_slot, void* const* out, int32_t* dev_status,
                               void* stream) {
    AttnArgs a;
    if (int rc = check_desc(desc, &a)) return rc;
    if (layers < 0 || batch < 0 || rows < 0 || n_q < 0 || seq_len < 0 || num_slots < 0 ||
        private_begin < 0 || private_begin > num_slots)
        return ACACHE_ERR_INVALID_ARG;
    if (layers == 0 || batch == 0) return ACACHE_OK;
    const bool store = rows > 0, attend = n_q > 0;
    if (!k_cache || !v_cache || (store && (!k_new || !v_new || !write_slot)) ||
        (attend && (!q || !out || !read_slot || seq_len == 0)))
        return ACACHE_ERR_INVALID_ARG;
    // every layer's arguments are checked before anything is launched
    for (int l = 0; l < layers; ++l) {
        if (!k_cache[l] || !v_cache[l] || !aligned16(k_cache[l]) || !aligned16(v_cache[l]))
            return ACACHE_ERR_INVALID_ARG;
        if (store && (!k_new[l] || !v_new[l] || !aligned16(k_new[l]) || !aligned16(v_new[l])))
            return ACACHE_ERR_INVALID_ARG;
        if (attend && (!q[l] || !out[l] || !aligned16(q[l]) || !aligned16(out[l])))
            return ACACHE_ERR_INVALID_ARG;
    }
    cudaStream_t st = (cudaStream_t)stream;
    const int64_t eb = elem_bytes(a.dtype);
    const int64_t row_bytes = (int64_t)a.hkv * a.d * eb;
    // Byte ranges of each layer's buffers; a layer's written ranges (its pools, its output) must
    // meet no range of another layer for their grids to overlap.
    struct Range {
        uintptr_t lo, hi;
        bool written;
    };
    auto span = [](const void* ptr, int64_t bytes, bool written) {
        return Range{(uintptr_t)ptr, (uintptr_t)ptr + (uintptr_t)bytes, written};
    };
    const int64_t pool_bytes = num_slots * row_bytes;
    const int64_t new_bytes = (int64_t)batch * rows * row_bytes;
    const int64_t qo_bytes = (int64_t)batch * n_q * a.hq * a.d * eb;
    bool disjoint = true;
    for (int i = 0; i < layers && disjoint; ++i) {
        Range wi[3] = {span(k_cache[i], pool_bytes, true), span(v_cache[i], pool_bytes, true),
                       span(attend ? out[i] : nullptr, attend ? qo_bytes : 0, true)};
        for (int j = 0; j < layers && disjoint; ++j) {
            if (i == j) continue;
            Range rj[6] = {span(k_cache[j], pool_bytes, true), span(v_cache[j], pool_bytes, true),
                           span(attend ? out[j] : nullptr, attend ? qo_bytes : 0, true),
                           span(attend ? q[j] : nullptr, attend ? qo_bytes : 0, false),
                           span(store ? k_new[j] : nullptr, store ? new_bytes : 0, false),
                           span(store ? v_new[j] : nullptr, store ? new_bytes : 0, false)};
            for (const Range& x : wi)
                for (const Range& y : rj)
                    if (x.lo < x.hi && y.lo < y.hi && x.lo < y.hi && y.lo < x.hi) disjoint = false;
        }
    }
    const bool chain = disjoint && layers > 1 && (!attend || (tc_supported(a) && !tc_decode_preferred(a, batch, n_q, seq_len)));
    if (!chain) {
        for (int l = 0; l < layers; ++l)
            if (int rc = acache_store_attend(desc, batch, rows, write_slot, store ? k_new[l] : nullptr,
                                             store ? v_new[l] : nullptr, k_cache[l], v_cache[l], num_slots,
                                             private_begin, n_q, attend ? q[l] : nullptr, seq_len, read_slot,
                                             attend ? out[l] : nullptr, dev_status, stream))
                return rc;
        return ACACHE_OK;
    }
    // Chained: the stores of every layer back to back, then the attentions; each grid may start
    // on the SMs its predecessor's last wave leaves idle.  The first attention is an ordinary
    // launch, so it starts after every store of the call (and every earlier grid) is complete;
    // the attentions chained after it start only once all of its CTAs have started reading.
    if (store)
        for (int l = 0; l < layers; ++l)
            if (int rc = launch_write_slots(batch, rows, write_slot, k_new[l], v_new[l], k_cache[l], v_cache[l],
                                            row_bytes, num_slots, private_begin, dev_status, st, l > 0))
                return rc;
    if (attend)
        for (int l = 0; l < layers; ++l)
            if (int rc = launch_tc_slot_attention(a, batch, n_q, q[l], seq_len, read_slot, k_cache[l], v_cache[l],
                                                  num_slots, out[l], dev_status, st, false, false, l > 0))
                return rc;
    return ACACHE_OK;
}

int acache_write_slots(const acache_attn_desc* desc, int batch, int rows,
                       const int32_t* write_slot, const void* k_new, const void* v_new,
                       void* k_cache, void* v_cache, int64_t num_slots, int64_t private_begin,
                       int32_t* dev_status, void* stream) {
    AttnArgs a;
    if (int rc = check_desc(desc, &a)) return rc;
    if (batch < 0 || rows < 0 || num_slots < 0 || private_begin < 0 || private_begin > num_slots)
        return ACACHE_ERR_INVALID_ARG;
    if (batch == 0 || rows == 0) return ACACHE_OK;
    if (!write_slot || !k_new || !v_new || !k_cache || !v_cache) return ACACHE_ERR_INVALID_ARG;
    if (!aligned16(k_new) || !aligned16(v_new) || !aligned16(k_cache) || !aligned16(v_cache))
        return ACACHE_ERR_INVALID_ARG;
    const int64_t row_bytes = (int64_t)a.hkv * a.d * elem_bytes(a.dtype);
    return launch_write_slots(batch, rows, write_slot, k_new, v_new, k_cache, v_cache, row_bytes,
                              num_slots, private_begin, dev_status, (cudaStream_t)stream);
}


int acache_slot_attention(const acache_attn_desc* desc, int batch, int n_q, const void* q,
                          int seq_len, const int32_t* read_slot, const void* k_cache,
                          const void* v_cache, int64_t num_slots, void* out,
                          int32_t* dev_status, void* stream) {
    return slot_attention(desc, batch, n_q, q, seq_len, read_slot, k_cache, v_cache, num_slots, out,
                          dev_status, stream, false);
}

int acache_slot_attention_varlen(const acache_attn_desc* desc, int batch, const int32_t* q_start,
                                 int max_q_rows, int total_q_rows, const void* q, const int32_t* kv_start,
                                 int max_seq_len, const int32_t* read_slot, const void* k_cache,
                                 const void* v_cache, int64_t num_slots, void* out, int drop_none,
                                 int32_t* dev_status, void* stream_) {
    AttnArgs a;
    if (int rc = check_desc(desc, &a)) return rc;
    if (batch < 0 || max_q_rows < 0 || total_q_rows < 0 || max_seq_len < 0 || num_slots < 0)
        return ACACHE_ERR_INVALID_ARG;
    if (batch == 0 || max_q_rows == 0 || total_q_rows == 0) return ACACHE_OK;
    if (max_seq_len == 0) return ACACHE_ERR_INVALID_ARG;   // a softmax over no keys
    if (!q_start || !kv_start || !q || !read_slot || !k_cache || !v_cache || !out)
        return ACACHE_ERR_INVALID_ARG;
    if (!aligned16(q) || !aligned16(k_cache) || !aligned16(v_cache) || !aligned16(out))
        return ACACHE_ERR_INVALID_ARG;
    cudaStream_t stream = (cudaStream_t)stream_;
    if (tc_supported(a))
        return launch_tc_slot_attention_varlen(a, batch, q_start, max_q_rows, total_q_rows, q, kv_start,
                                               max_seq_len, read_slot, k_cache, v_cache, num_slots, out,
                                               dev_status, stream, drop_none != 0);
    return launch_simt_slot_attention_varlen(a, batch, q_start, max_q_rows, q, kv_start, max_seq_len,
                                             read_slot, k_cache, v_cache, num_slots, out, dev_status,
                                             stream, drop_none != 0);
}

int acache_slot_attention_dropna(const acache_attn_desc* desc, int batch, int n_q, const void* q,
                                 int seq_len, const int32_t* read_slot, const void* k_cache,
                                 const void* v_cache, int64_t num_slots, void* out,
                                 int32_t* dev_status, void* stream) {
    return slot_attention(desc, batch, n_q, q, seq_len, read_slot, k_cache, v_cache, num_slots, out,
                          dev_status, stream, true);
}

int acache_gather_slots(const acache_attn_desc* desc, int batch, int seq_len,
                        const int32_t* read_slot, const void* k_cache, const void* v_cache,
                        int64_t num_slots, void* k_out, void* v_out, int32_t* dev_status,
                        void* stream) {
    AttnArgs a;
    if (int rc = check_desc(desc, &a)) return rc;
    if (batch < 0 || seq_len < 0 || num_slots < 0) return ACACHE_ERR_INVALID_ARG;
    if (batch == 0 || seq_len == 0) return ACACHE_OK;
    if (!read_slot || !k_cache || !v_cache || !k_out || !v_out) return ACACHE_ERR_INVALID_ARG;
    if (!aligned16(k_cache) || !aligned16(v_cache) || !aligned16(k_out) || !aligned16(v_out))
        return ACACHE_ERR_INVALID_ARG;
    const int64_t row_bytes = (int64_t)a.hkv * a.d * elem_bytes(a.dtype);
    return launch_gather_slots(batch, seq_len, read_slot, k_cache, v_cache, row_bytes, num_slots,
                               k_out, v_out, dev_status, (cudaStream_t)stream);
}

}  // extern "C"
