// rope.cu -- position-aware affix registration: move cached, already rotated keys to another
// offset.
//
// Page: "Affix Cache for Diffusion Large Language Models", Sec. 4 (opening) and Limitations:
// the prototype stores the cache after the positional rotation, so reusing an affix at
// another offset (infix / suffix reuse) needs the span registered with its position.
// Rotary embeddings rotate each frequency pair of a key by (position x frequency), and
// rotations compose, so a key computed at position p is moved to position p + delta by one more rotation by
// (delta x frequency) -- no access to the unrotated keys is needed.  Values carry no rotation.
//
// Pair i of a head (frequency theta^(-2i/d)) is (x_i, x_{i+d/2}) in the half-split layout
// (the rotate-half convention) or (x_{2i}, x_{2i+1}) in the interleaved layout.  The cos/sin
// table is computed on the host in double precision; the rotation is two float32 FMAs per
// element, rounded once to the storage type.  HBM-bound and off the online path (it runs at
// affix registration), so a plain element-pair-per-thread kernel.
#include <math.h>

#include "common.cuh"

namespace acache {
namespace {

constexpr int kRopeThreads = 256;

struct RopeTable {
    float c[64];
    float s[64];
};

template <typename T>
__global__ void __launch_bounds__(kRopeThreads)
rerotate_kernel(int64_t n_pairs, int d, int interleaved, const T* __restrict__ k_in, T* __restrict__ k_out,
                const __grid_constant__ RopeTable tab) {
    const int64_t idx = (int64_t)blockIdx.x * kRopeThreads + threadIdx.x;
    if (idx >= n_pairs) return;
    const int half = d / 2;
    const int64_t head = idx / half;        // (row, kv head)
    const int i = (int)(idx % half);
    const int64_t o0 = head * d + (interleaved ? 2 * i : i);
    const int64_t o1 = o0 + (interleaved ? 1 : half);
    const float x0 = to_f32(k_in[o0]), x1 = to_f32(k_in[o1]);
    const float c = tab.c[i], s = tab.s[i];
    k_out[o0] = from_f32<T>(fmaf(x0, c, -x1 * s));
    k_out[o1] = from_f32<T>(fmaf(x0, s, x1 * c));
}

}  // namespace

int launch_rerotate(int dtype, int64_t rows, int hkv, int d, const void* k_in, void* k_out, int32_t delta,
                    double theta, int interleaved, cudaStream_t stream) {
    const int64_t n_pairs = rows * hkv * (d / 2);
    if (n_pairs == 0) return ACACHE_OK;
    RopeTable tab{};
    for (int i = 0; i < d / 2; ++i) {
        const double freq = pow(theta, -2.0 * i / d);
        const double ang = (double)delta * freq;
        tab.c[i] = (float)cos(ang);
        tab.s[i] = (float)sin(ang);
    }
    const int64_t blocks = (n_pairs + kRopeThreads - 1) / kRopeThreads;
    if (blocks > 0x7fffffffLL) return ACACHE_ERR_INVALID_ARG;
    if (dtype == ACACHE_BF16)
        rerotate_kernel<__nv_bfloat16><<<(unsigned)blocks, kRopeThreads, 0, stream>>>(
            n_pairs, d, interleaved, (const __nv_bfloat16*)k_in, (__nv_bfloat16*)k_out, tab);
    else
        rerotate_kernel<float><<<(unsigned)blocks, kRopeThreads, 0, stream>>>(
            n_pairs, d, interleaved, (const float*)k_in, (float*)k_out, tab);
    return launch_status();
}

}  // namespace acache
