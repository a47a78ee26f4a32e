// slots.cu -- the store step, the logical-KV gather and the admission-time maps.
//
// Page: "Affix Cache for Diffusion Large Language Models", Sec. 4.1 (write-side
// recomputation map, per-request read-slot map), Sec. 4.2 (maps recorded at admission),
// Sec. 4.3 and App. C.1 (store-then-attend).
//
// The copies are HBM-bound: every thread moves 16-byte vectors and keeps kUnroll
// independent loads in flight before its stores; a warp copies one row, reading its slot
// index once; the grid is capped at 8 CTAs per SM.
#include "common.cuh"
#include "ptx.cuh"

namespace acache {
namespace {

constexpr int kCopyThreads = 256;
constexpr int kUnroll = 8;

// Row copy through an index table, one warp per part of a row of K or of V (2 * nrows rows,
// `parts` parts of `per_part` 16-byte chunks each -- several warps per row when rows are few):
// the row's index is read once and the lanes stride over the part's chunks, kUnroll loads in
// flight each, with no per-chunk index arithmetic.
//   scatter = true : dst[idx[r]] = src[r]   (store step, idx = write slots)
//   scatter = false: dst[r] = src[idx[r]]   (gather through the read-slot map)
template <bool kScatter>
__global__ void __launch_bounds__(kCopyThreads)
indexed_row_copy(const int32_t* __restrict__ idx, int64_t nrows, int64_t cpr,
                 int parts, int64_t per_part,
                 const uint4* __restrict__ src_k, const uint4* __restrict__ src_v,
                 uint4* __restrict__ dst_k, uint4* __restrict__ dst_v,
                 int64_t num_slots, int64_t private_begin, int32_t* dev_status) {
    // a grid that waits on this copy (store-then-attend) may start its prologue now; it
    // reads nothing this copy writes before its own grid-dependency wait
    ptx::grid_launch_dependents();
    constexpr int kWarps = kCopyThreads / 32;
    const int lane = threadIdx.x & 31;
    const int64_t n_warps = (int64_t)gridDim.x * kWarps;
    for (int64_t w = (int64_t)blockIdx.x * kWarps + (threadIdx.x >> 5); w < 2 * nrows * parts; w += n_warps) {
        const int64_t wr = w / parts;                    // row of K (< nrows) or of V
        const int part = (int)(w - wr * parts);
        const bool is_v = wr >= nrows;
        const int64_t r = is_v ? wr - nrows : wr;
        const int64_t slot = idx[r];
        if (slot < 0 || slot >= num_slots) {
            if (!is_v && part == 0 && lane == 0) flag(dev_status, ACACHE_DEV_BAD_SLOT);
            continue;
        }
        if (kScatter && slot < private_begin) {
            if (!is_v && part == 0 && lane == 0) flag(dev_status, ACACHE_DEV_SHARED_WRITE);
            continue;
        }
        const int64_t c_end = (part + 1) * per_part < cpr ? (part + 1) * per_part : cpr;
        const uint4* src = (is_v ? src_v : src_k) + (kScatter ? r : slot) * cpr;
        uint4* dst = (is_v ? dst_v : dst_k) + (kScatter ? slot : r) * cpr;
        for (int64_t c0 = part * per_part + lane; c0 < c_end; c0 += 32 * kUnroll) {
            uint4 val[kUnroll];
#pragma unroll
            for (int u = 0; u < kUnroll; ++u)
                if (c0 + 32 * u < c_end) val[u] = __ldcs(src + c0 + 32 * u);   // streamed once
#pragma unroll
            for (int u = 0; u < kUnroll; ++u)
                if (c0 + 32 * u < c_end) __stcs(dst + c0 + 32 * u, val[u]);
        }
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

// Parts per row: enough warps to cover the SMs' memory latency (16 per SM) when rows are few,
// but at least 32 * kUnroll chunks per part.
struct CopyShape {
    int parts;
    int64_t per_part;
};
CopyShape copy_shape(int64_t rows, int64_t cpr) {      // rows: of K and V together
    const int64_t want_warps = (int64_t)sm_count() * 16;
    int64_t parts = (want_warps + rows - 1) / rows;
    const int64_t max_parts = cpr / (32 * kUnroll) > 1 ? cpr / (32 * kUnroll) : 1;
    if (parts > max_parts) parts = max_parts;
    if (parts < 1) parts = 1;
    int64_t per_part = (cpr + parts - 1) / parts;
    per_part = (per_part + 31) / 32 * 32;
    return {(int)parts, per_part};
}

int copy_grid(int64_t items) {                      // one warp per part of a row of K or V
    const int64_t per_cta = kCopyThreads / 32;
    int64_t want = (items + per_cta - 1) / per_cta;
    const int64_t cap = (int64_t)sm_count() * 8;     // 8 resident CTAs of 256 threads per SM
    if (want > cap) want = cap;
    if (want < 1) want = 1;
    return (int)want;
}

}  // namespace

// pdl: launched with programmatic stream serialisation after a grid that touches none of this
// store's memory (the store of another layer): it may run alongside that grid.
int launch_write_slots(int batch, int rows, const int32_t* write_slot, const void* k_new,
                       const void* v_new, void* k_cache, void* v_cache, int64_t row_bytes,
                       int64_t num_slots, int64_t private_begin, int32_t* dev_status,
                       cudaStream_t stream, bool pdl) {
    const int64_t nrows = (int64_t)batch * rows, cpr = row_bytes / 16;
    if (nrows == 0) return ACACHE_OK;
    const CopyShape cs = copy_shape(2 * nrows, cpr);
    const unsigned grid = (unsigned)copy_grid(2 * nrows * cs.parts);
    if (!pdl) {
        indexed_row_copy<true><<<grid, kCopyThreads, 0, stream>>>(
            write_slot, nrows, cpr, cs.parts, cs.per_part, (const uint4*)k_new, (const uint4*)v_new,
            (uint4*)k_cache, (uint4*)v_cache, num_slots, private_begin, dev_status);
        return launch_status();
    }
    cudaLaunchConfig_t cfg = {};
    cfg.gridDim = dim3(grid);
    cfg.blockDim = dim3(kCopyThreads);
    cfg.stream = stream;
    cudaLaunchAttribute attr[1];
    attr[0].id = cudaLaunchAttributeProgrammaticStreamSerialization;
    attr[0].val.programmaticStreamSerializationAllowed = 1;
    cfg.attrs = attr;
    cfg.numAttrs = 1;
    if (cudaLaunchKernelEx(&cfg, indexed_row_copy<true>, write_slot, nrows, cpr, cs.parts, cs.per_part,
                           (const uint4*)k_new, (const uint4*)v_new, (uint4*)k_cache, (uint4*)v_cache,
                           num_slots, private_begin, dev_status) != cudaSuccess) {
        (void)cudaGetLastError();
        return ACACHE_ERR_CUDA;
    }
    return launch_status();
}

int launch_gather_slots(int batch, int seq_len, const int32_t* read_slot, const void* k_cache,
                        const void* v_cache, int64_t row_bytes, int64_t num_slots, void* k_out,
                        void* v_out, int32_t* dev_status, cudaStream_t stream) {
    const int64_t nrows = (int64_t)batch * seq_len, cpr = row_bytes / 16;
    if (nrows == 0) return ACACHE_OK;
    const CopyShape cs = copy_shape(2 * nrows, cpr);
    indexed_row_copy<false><<<copy_grid(2 * nrows * cs.parts), kCopyThreads, 0, stream>>>(
        read_slot, nrows, cpr, cs.parts, cs.per_part, (const uint4*)k_cache, (const uint4*)v_cache, (uint4*)k_out,
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
