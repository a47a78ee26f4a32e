// slots.cu -- the store step, the logical-KV gather and the admission-time maps.
//
// Page: "Affix Cache for Diffusion Large Language Models", Sec. 4.1 (write-side
// recomputation map, per-request read-slot map), Sec. 4.2 (maps recorded at admission),
// Sec. 4.3 and App. C.1 (store-then-attend).
//
// The copies are HBM-bound: every thread moves 16-byte vectors, keeps kUnroll
// independent loads in flight before its stores, and the grid is a multiple of the SM
// count.  Slot indices are read once per 16-byte chunk (they hit L1: all chunks of a
// row share one index).
#include "common.cuh"
#include "ptx.cuh"

namespace acache {
namespace {

constexpr int kCopyThreads = 256;
constexpr int kUnroll = 4;

// Row copy through an index table.  Rows are `cpr` 16-byte chunks long.
//   scatter = true : dst[idx[r]] = src[r]   (store step, idx = write slots)
//   scatter = false: dst[r] = src[idx[r]]   (gather through the read-slot map)
template <bool kScatter>
__global__ void __launch_bounds__(kCopyThreads)
indexed_row_copy(const int32_t* __restrict__ idx, int64_t nrows, int64_t cpr,
                 const uint4* __restrict__ src_k, const uint4* __restrict__ src_v,
                 uint4* __restrict__ dst_k, uint4* __restrict__ dst_v,
                 int64_t num_slots, int64_t private_begin, int32_t* dev_status) {
    // a grid that waits on this copy (store-then-attend) may start its prologue now; it
    // reads nothing this copy writes before its own grid-dependency wait
    ptx::grid_launch_dependents();
    const int64_t total = nrows * cpr;                   // chunks per tensor (K or V)
    const int64_t stride = (int64_t)gridDim.x * blockDim.x;
    for (int64_t base = (int64_t)blockIdx.x * blockDim.x + threadIdx.x; base < 2 * total;
         base += stride * kUnroll) {
        uint4 val[kUnroll];
        uint4* dst[kUnroll];
#pragma unroll
        for (int u = 0; u < kUnroll; ++u) {
            const int64_t c = base + u * stride;
            dst[u] = nullptr;
            if (c < 2 * total) {
                const bool is_v = c >= total;
                const int64_t cc = is_v ? c - total : c;
                const int64_t r = cc / cpr, w = cc - r * cpr;
                const int64_t slot = idx[r];
                bool good = slot >= 0 && slot < num_slots;
                if (!good) {
                    if (w == 0 && !is_v) flag(dev_status, ACACHE_DEV_BAD_SLOT);
                } else if (kScatter && slot < private_begin) {
                    good = false;
                    if (w == 0 && !is_v) flag(dev_status, ACACHE_DEV_SHARED_WRITE);
                }
                if (good) {
                    const int64_t s_off = kScatter ? r * cpr + w : slot * cpr + w;
                    const int64_t d_off = kScatter ? slot * cpr + w : r * cpr + w;
                    val[u] = __ldcs((is_v ? src_v : src_k) + s_off);   // streamed once
                    dst[u] = (is_v ? dst_v : dst_k) + d_off;
                }
            }
        }
#pragma unroll
        for (int u = 0; u < kUnroll; ++u)
            if (dst[u]) __stcs(dst[u], val[u]);
    }
}

// Admission-time maps, one CTA per request (see acache.h).  The recomputed positions in
// ascending order are: [0, l) (non-affix), then the anchors l + A_b, then [l+L, T).  So
// the write index of a position has a closed form and no scan is needed:
//   t <  l          : i = t
//   t in F, anchor  : i = l + (number of anchors below t - l)
//   t >= l + L      : i = l + K + (t - l - L)
__global__ void __launch_bounds__(1024)
build_maps_kernel(int T, int l, int L, int K, const int32_t* __restrict__ anchors,
                  const int32_t* __restrict__ shared_slot,
                  const int32_t* __restrict__ private_slots, int32_t* __restrict__ write_pos,
                  int32_t* __restrict__ read_slot, int32_t* dev_status) {
    const int b = blockIdx.x;
    const int R = K + (T - L);
    const int32_t* A = anchors + (int64_t)b * K;
    // anchors must be strictly ascending offsets in [0, L)
    int bad = 0;
    for (int i = threadIdx.x; i < K; i += blockDim.x) {
        const int a = A[i];
        bad |= (a < 0 || a >= L || (i > 0 && a <= A[i - 1]));
    }
    if (__syncthreads_or(bad)) {
        if (threadIdx.x == 0) flag(dev_status, ACACHE_DEV_BAD_ANCHOR);
        return;
    }
    const int32_t* priv = private_slots + (int64_t)b * R;
    for (int t = threadIdx.x; t < T; t += blockDim.x) {
        int i = -1;
        if (t < l) {
            i = t;
        } else if (t >= l + L) {
            i = l + K + (t - l - L);
        } else {
            const int j = t - l;
            int lo = 0, hi = K;                 // lower_bound(A, j)
            while (lo < hi) {
                const int mid = (lo + hi) >> 1;
                if (A[mid] < j) lo = mid + 1; else hi = mid;
            }
            if (lo < K && A[lo] == j) i = l + lo;
        }
        if (i >= 0) {
            write_pos[(int64_t)b * R + i] = t;
            read_slot[(int64_t)b * T + t] = priv[i];
        } else {
            read_slot[(int64_t)b * T + t] = shared_slot[t - l];
        }
    }
}

int copy_grid(int64_t chunks) {
    const int64_t per_cta = (int64_t)kCopyThreads * kUnroll;
    int64_t want = (chunks + per_cta - 1) / per_cta;
    const int64_t cap = (int64_t)sm_count() * 8;     // 8 resident CTAs of 256 threads per SM
    if (want > cap) want = cap;
    if (want < 1) want = 1;
    return (int)want;
}

}  // namespace

int launch_write_slots(int batch, int rows, const int32_t* write_slot, const void* k_new,
                       const void* v_new, void* k_cache, void* v_cache, int64_t row_bytes,
                       int64_t num_slots, int64_t private_begin, int32_t* dev_status,
                       cudaStream_t stream) {
    const int64_t nrows = (int64_t)batch * rows, cpr = row_bytes / 16;
    if (nrows == 0) return ACACHE_OK;
    indexed_row_copy<true><<<copy_grid(2 * nrows * cpr), kCopyThreads, 0, stream>>>(
        write_slot, nrows, cpr, (const uint4*)k_new, (const uint4*)v_new, (uint4*)k_cache,
        (uint4*)v_cache, num_slots, private_begin, dev_status);
    return launch_status();
}

int launch_gather_slots(int batch, int seq_len, const int32_t* read_slot, const void* k_cache,
                        const void* v_cache, int64_t row_bytes, int64_t num_slots, void* k_out,
                        void* v_out, int32_t* dev_status, cudaStream_t stream) {
    const int64_t nrows = (int64_t)batch * seq_len, cpr = row_bytes / 16;
    if (nrows == 0) return ACACHE_OK;
    indexed_row_copy<false><<<copy_grid(2 * nrows * cpr), kCopyThreads, 0, stream>>>(
        read_slot, nrows, cpr, (const uint4*)k_cache, (const uint4*)v_cache, (uint4*)k_out,
        (uint4*)v_out, num_slots, 0, dev_status);
    return launch_status();
}

int launch_build_maps(int batch, int T, int l, int L, int K, const int32_t* anchors,
                      const int32_t* shared_slot, const int32_t* private_slots,
                      int32_t* write_pos, int32_t* read_slot, int32_t* dev_status,
                      cudaStream_t stream) {
    if (batch == 0 || T == 0) return ACACHE_OK;
    build_maps_kernel<<<batch, 1024, 0, stream>>>(T, l, L, K, anchors, shared_slot,
                                                  private_slots, write_pos, read_slot,
                                                  dev_status);
    return launch_status();
}

}  // namespace acache
