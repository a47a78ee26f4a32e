// probe_noalloc.cu -- acache_probe_scores_noalloc: the anchor probe of one layer with no
// workspace argument and no device allocation.
//
// Some callers cannot allocate device memory at the point where they probe: an engine that
// hands the library only the tensors it already owns (a fixed memory budget carved up at
// start-up, a custom allocator the library cannot reach, or code that must not call into the
// CUDA allocator at all).  For them this entry point keeps the probe's scratch -- the per-row
// maximum and sum of the forward pass and the per-head column sums of the masked-to-affix
// mass -- in one file-scope device array of fixed size instead of a caller-provided
// workspace.  The caller still passes every input and output.
//
// Properties of the static scratch (see include/acache.h):
//  - kStaticScratchBytes (16 MiB) per GPU, reserved on every GPU that loads this library and
//    held until the process exits;
//  - a call whose scratch need exceeds it returns ACACHE_ERR_WORKSPACE before any launch;
//  - every call shares it and it keeps the previous call's contents; nothing in it has to
//    start at zero (each call writes every byte it reads), but calls whose kernels overlap
//    on the GPU (different streams, no ordering between them) race on it;
//  - the first call on a device looks up the array's device address (once per device, with
//    that device current); make that first call before any stream capture begins.
#include <mutex>

#include "attn.cuh"
#include "tc_attn.cuh"

namespace acache {
namespace {

constexpr size_t kStaticScratchBytes = size_t(16) << 20;
constexpr size_t kScratchAlign = 256;

// In host code this name is only a host-side stand-in for the device array: kernels get the
// device address looked up below, never the name itself.
__device__ __align__(256) unsigned char g_probe_scratch[kStaticScratchBytes];

size_t round_up(size_t x) { return (x + kScratchAlign - 1) / kScratchAlign * kScratchAlign; }

constexpr int kMaxDevices = 64;
std::mutex g_scratch_mutex;
void* g_scratch_addr[kMaxDevices] = {};

// Device address of g_probe_scratch on the current device (looked up once per device).
int scratch_address(void** out) {
    int dev = 0;
    if (cudaGetDevice(&dev) != cudaSuccess || dev < 0 || dev >= kMaxDevices) {
        (void)cudaGetLastError();
        return ACACHE_ERR_CUDA;
    }
    std::lock_guard<std::mutex> lock(g_scratch_mutex);
    if (!g_scratch_addr[dev]) {
        void* ptr = nullptr;
        const cudaError_t e = cudaGetSymbolAddress(&ptr, g_probe_scratch);
        if (e != cudaSuccess || !ptr) {
            (void)cudaGetLastError();
            return ACACHE_ERR_CUDA;
        }
        g_scratch_addr[dev] = ptr;
    }
    *out = g_scratch_addr[dev];
    return ACACHE_OK;
}

}  // namespace
}  // namespace acache

using namespace acache;

extern "C" int acache_probe_scores_noalloc(const acache_attn_desc* desc, int batch, int seq_len,
                                           int affix_begin, int affix_len,
                                           const int32_t* masked_rows, int num_masked,
                                           const void* q, const void* k_req, const void* v_req,
                                           const void* k_affix, const void* v_affix, void* out,
                                           float* scores, int32_t* dev_status, void* stream_) {
    if (!desc || desc->num_q_heads <= 0 || desc->num_kv_heads <= 0 ||
        desc->num_q_heads % desc->num_kv_heads || !(desc->scale == desc->scale) ||
        isinf(desc->scale))
        return ACACHE_ERR_INVALID_ARG;
    if (desc->dtype != ACACHE_F32 && desc->dtype != ACACHE_BF16) return ACACHE_ERR_UNSUPPORTED;
    if (desc->head_dim != 64 && desc->head_dim != 128) return ACACHE_ERR_UNSUPPORTED;
    const AttnArgs a{desc->num_q_heads, desc->num_kv_heads, desc->head_dim, desc->dtype, desc->scale};
    const int T = seq_len, l = affix_begin, L = affix_len, m = num_masked;
    if (batch < 0 || T < 0 || l < 0 || L < 0 || (int64_t)l + L > T || m < 0 || m > T - L)
        return ACACHE_ERR_INVALID_ARG;
    const int P = T - L;
    if (batch == 0 || P == 0) return ACACHE_OK;
    if (!q || !k_req || !v_req || (L > 0 && (!k_affix || !v_affix)) || (m > 0 && !masked_rows) ||
        (L > 0 && !scores))
        return ACACHE_ERR_INVALID_ARG;
    auto a16 = [](const void* p) { return ((uintptr_t)p & 15u) == 0; };
    if (!a16(q) || !a16(k_req) || !a16(v_req) || !a16(k_affix) || !a16(v_affix) || !a16(out))
        return ACACHE_ERR_INVALID_ARG;
    // scratch: row max, row sum [B][Hq][P] and column sums [B][Hq][L], 256-byte aligned parts
    const size_t st = round_up((size_t)batch * a.hq * P * sizeof(float));
    const size_t pa = round_up((size_t)batch * a.hq * L * sizeof(float));
    if (2 * st + pa > kStaticScratchBytes) return ACACHE_ERR_WORKSPACE;
    void* base = nullptr;
    if (int rc = scratch_address(&base)) return rc;
    float* stat_m = (float*)base;
    float* stat_l = (float*)((char*)base + st);
    float* partial = (float*)((char*)base + 2 * st);
    cudaStream_t stream = (cudaStream_t)stream_;
    int rc;
    if (tc_supported(a))
        rc = launch_tc_probe_pass_a(a, batch, T, l, L, q, k_req, v_req, k_affix, v_affix, out,
                                    stat_m, stat_l, dev_status, stream);
    else
        rc = launch_simt_probe_pass_a(a, batch, T, l, L, q, k_req, v_req, k_affix, v_affix, out,
                                      stat_m, stat_l, stream);
    if (rc) return rc;
    if (L == 0) return ACACHE_OK;
    if (tc_supported(a))
        rc = launch_tc_probe_pass_b(a, batch, T, L, masked_rows, m, q, k_affix, stat_m, stat_l,
                                    partial, dev_status, stream);
    else
        rc = launch_simt_probe_pass_b(a, batch, T, L, masked_rows, m, q, k_affix, stat_m, stat_l,
                                      partial, dev_status, stream);
    if (rc) return rc;
    return launch_score_reduce(batch, a.hq, L, partial, scores, stream);
}
