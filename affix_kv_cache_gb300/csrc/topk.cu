// topk.cu -- anchor selection A = TopK({s_j}, K) with ties toward the lower offset.
//
// Page: "Affix Cache for Diffusion Large Language Models", Sec. 3.2, Eq. 6 (cost
// O(L log K) there; here one CTA per request does a 4-pass radix select, O(L)).
//
// Each score maps to an order-preserving 32-bit key (larger float -> larger key; -0.0 is
// folded onto +0.0; NaN maps below every number and is flagged).  A most-significant-
// digit-first radix select (4 passes of 8 bits, histograms in shared memory) finds the
// K-th largest key u* and how many keys equal to u* still have to be taken.  A final
// ordered pass takes every key above u* plus the lowest-offset keys equal to u*, and
// writes the chosen offsets in ascending order with a block-wide prefix sum.  All counts
// are integers, so the result is exact and deterministic.  The scores are re-read from
// global memory on every pass (L <= a few 10^4 floats, L1/L2 resident).
#include "common.cuh"

namespace acache {
namespace {

constexpr int kTopkThreads = 1024;
constexpr int kWarps = kTopkThreads / 32;

ACACHE_DEVFN uint32_t order_key(float f, bool& is_nan) {
    uint32_t u = __float_as_uint(f);
    is_nan = (u & 0x7fffffffu) > 0x7f800000u;
    if (is_nan) return 0u;
    if (u == 0x80000000u) u = 0u;                      // -0.0 -> +0.0
    return (u & 0x80000000u) ? ~u : (u | 0x80000000u);
}

// Exclusive prefix sum over the block; returns this thread's offset, total in *total.
ACACHE_DEVFN int block_exclusive_scan(int v, int* warp_sums, int* total) {
    const int lane = threadIdx.x & 31, warp = threadIdx.x >> 5;
    int x = v;
#pragma unroll
    for (int o = 1; o < 32; o <<= 1) {
        const int y = __shfl_up_sync(0xffffffffu, x, o);
        if (lane >= o) x += y;
    }
    if (lane == 31) warp_sums[warp] = x;
    __syncthreads();
    if (warp == 0) {
        int w = lane < kWarps ? warp_sums[lane] : 0;
#pragma unroll
        for (int o = 1; o < 32; o <<= 1) {
            const int y = __shfl_up_sync(0xffffffffu, w, o);
            if (lane >= o) w += y;
        }
        warp_sums[lane] = w;                           // inclusive over warps
    }
    __syncthreads();
    const int before = (warp > 0 ? warp_sums[warp - 1] : 0) + x - v;
    *total = warp_sums[kWarps - 1];
    __syncthreads();
    return before;
}

__global__ void __launch_bounds__(kTopkThreads)
topk_kernel(const float* __restrict__ scores, int L, int K, int32_t* __restrict__ anchors,
            int32_t* dev_status) {
    __shared__ int hist[256];
    __shared__ int warp_sums[32];
    __shared__ uint32_t s_prefix;
    __shared__ int s_need;
    const int b = blockIdx.x;
    const float* s = scores + (int64_t)b * L;
    int32_t* out = anchors + (int64_t)b * K;
    if (K == 0) return;

    // ---- radix select of the K-th largest key --------------------------------------
    uint32_t prefix = 0, prefix_mask = 0;
    int need = K;                                      // keys still to take at/below prefix
    bool any_nan = false;
    for (int shift = 24; shift >= 0; shift -= 8) {
        for (int i = threadIdx.x; i < 256; i += blockDim.x) hist[i] = 0;
        __syncthreads();
        for (int j = threadIdx.x; j < L; j += blockDim.x) {
            bool nan;
            const uint32_t u = order_key(s[j], nan);
            any_nan |= nan;
            if ((u & prefix_mask) == prefix) atomicAdd(&hist[(u >> shift) & 0xffu], 1);
        }
        __syncthreads();
        if (threadIdx.x == 0) {
            int above = 0, digit = 255;
            for (; digit > 0; --digit) {
                if (above + hist[digit] >= need) break;
                above += hist[digit];
            }
            s_prefix = prefix | ((uint32_t)digit << shift);
            s_need = need - above;
        }
        __syncthreads();
        prefix = s_prefix;
        need = s_need;
        prefix_mask |= 0xffu << shift;
        __syncthreads();
    }
    if (any_nan) flag(dev_status, ACACHE_DEV_NAN);
    const uint32_t kth = prefix;                       // the K-th largest key
    // ---- ordered compaction ---------------------------------------------------------
    int taken = 0, equal_seen = 0;
    for (int j0 = 0; j0 < L; j0 += blockDim.x) {
        const int j = j0 + threadIdx.x;
        uint32_t u = 0;
        if (j < L) {
            bool nan;
            u = order_key(s[j], nan);
        }
        const int is_eq = (j < L && u == kth) ? 1 : 0;
        int eq_total;
        const int eq_before = equal_seen + block_exclusive_scan(is_eq, warp_sums, &eq_total);
        const int take = (j < L) && (u > kth || (is_eq && eq_before < need));
        int take_total;
        const int pos = taken + block_exclusive_scan(take, warp_sums, &take_total);
        if (take) out[pos] = j;
        taken += take_total;
        equal_seen += eq_total;
    }
}

}  // namespace

int launch_topk(const float* scores, int batch, int L, int K, int32_t* anchors,
                int32_t* dev_status, cudaStream_t stream) {
    if (batch == 0 || K == 0) return ACACHE_OK;
    topk_kernel<<<batch, kTopkThreads, 0, stream>>>(scores, L, K, anchors, dev_status);
    return launch_status();
}

}  // namespace acache
