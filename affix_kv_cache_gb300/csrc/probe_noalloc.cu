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
//  - the array's device address is looked up on every call made while the stream is not
//    capturing (so a device reset, which reloads the library's device code, is followed);
//    a call made during stream capture uses the address of the device's last earlier call,
//    so the first call on a device must come before any capture.
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

constexpr int kMaxDevices = 64;
std::mutex g_scratch_mutex;
void* g_scratch_addr[kMaxDevices] = {};

// Device address of g_probe_scratch on the current device.  Outside stream capture it is looked
// up afresh (after a device reset the array may sit elsewhere); during capture the address the
// device's last earlier call found is used.
int scratch_address(cudaStream_t stream, void** out) {
    int dev = 0;
    if (cudaGetDevice(&dev) != cudaSuccess || dev < 0 || dev >= kMaxDevices) {
        (void)cudaGetLastError();
        return ACACHE_ERR_CUDA;
    }
    cudaStreamCaptureStatus cap = cudaStreamCaptureStatusNone;
    if (cudaStreamIsCapturing(stream, &cap) != cudaSuccess) {
        (void)cudaGetLastError();
        return ACACHE_ERR_CUDA;
    }
    std::lock_guard<std::mutex> lock(g_scratch_mutex);
    if (cap == cudaStreamCaptureStatusNone) {
        void* ptr = nullptr;
        const cudaError_t e = cudaGetSymbolAddress(&ptr, g_probe_scratch);
        if (e != cudaSuccess || !ptr) {
            (void)cudaGetLastError();
            return ACACHE_ERR_CUDA;
        }
        g_scratch_addr[dev] = ptr;
    } else if (!g_scratch_addr[dev]) {
        return ACACHE_ERR_CUDA;     // never called on this device before the capture began
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
    ProbeCall c;
    bool empty = false;
    if (int rc = probe_check(desc, batch, seq_len, affix_begin, affix_len, masked_rows, num_masked, q, k_req,
                             v_req, k_affix, v_affix, out, scores, &c, &empty))
        return rc;
    if (empty) return ACACHE_OK;
    static_assert(kStaticScratchBytes % kScratchAlign == 0, "whole aligned parts");
    if (probe_scratch_bytes(c) > kStaticScratchBytes) return ACACHE_ERR_WORKSPACE;
    cudaStream_t stream = (cudaStream_t)stream_;
    void* base = nullptr;
    if (int rc = scratch_address(stream, &base)) return rc;
    return probe_launch(c, base, dev_status, stream);
}
