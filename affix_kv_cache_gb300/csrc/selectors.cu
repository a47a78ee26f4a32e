// selectors.cu -- the alternative anchor selector the page compares ACache against.
//
// Page: "Affix Cache for Diffusion Large Language Models", App. B.5 (CacheBlend-style
// anchor selection): affix tokens are ranked by the deviation between the affix-only KV
// cache and the KV the affix tokens get inside the full prompt, instead of by
// masked-to-affix attention.  The ranking itself reuses the Top-K of Eq. 6.
//
// Deviation of affix token j in one layer (reading: the L2 norm of the difference per
// KV head, K and V, summed over KV heads):
//     dev_j = sum_{hk ascending} ( ||K_full[j,hk] - K_shared[j,hk]||_2 + ||V_full[j,hk] - V_shared[j,hk]||_2 )
// and scores[b][j] += dev_j layer after layer, like the probe's Eq. 5 sum.
//
// HBM-bound: one warp per (request, affix token); every lane reads 8 consecutive elements
// (16 bytes of bf16) of the four rows per step, the squares are summed in float32 and
// reduced inside each head's group of lanes with a fixed xor tree, and lane 0 adds the
// heads in ascending order -- so the result is bit-reproducible and needs no atomics.
#include "common.cuh"

namespace acache {
namespace {

constexpr int kDevWarps = 8;

template <typename T>
ACACHE_DEVFN void load8(const T* p, float (&x)[8]);
template <>
ACACHE_DEVFN void load8<__nv_bfloat16>(const __nv_bfloat16* p, float (&x)[8]) {
    const uint4 u = __ldcs(reinterpret_cast<const uint4*>(p));
    const uint32_t w[4] = {u.x, u.y, u.z, u.w};
#pragma unroll
    for (int i = 0; i < 4; ++i) {
        x[2 * i] = __uint_as_float(w[i] << 16);
        x[2 * i + 1] = __uint_as_float(w[i] & 0xffff0000u);
    }
}
template <>
ACACHE_DEVFN void load8<float>(const float* p, float (&x)[8]) {
    const float4 a = __ldcs(reinterpret_cast<const float4*>(p));
    const float4 b = __ldcs(reinterpret_cast<const float4*>(p) + 1);
    x[0] = a.x; x[1] = a.y; x[2] = a.z; x[3] = a.w;
    x[4] = b.x; x[5] = b.y; x[6] = b.z; x[7] = b.w;
}

template <typename T>
__global__ void __launch_bounds__(kDevWarps * 32)
kv_deviation_kernel(int64_t n_tok, int L, int Hkv, int d, const T* __restrict__ k_sh,
                    const T* __restrict__ v_sh, const T* __restrict__ k_full,
                    const T* __restrict__ v_full, float* __restrict__ scores) {
    const int64_t tok = (int64_t)blockIdx.x * kDevWarps + (threadIdx.x >> 5);
    if (tok >= n_tok) return;
    const int lane = threadIdx.x & 31;
    const int j = (int)(tok % L);
    const int64_t E = (int64_t)Hkv * d;          // elements of one token row (all KV heads)
    const T* ks = k_sh + (int64_t)j * E;
    const T* vs = v_sh + (int64_t)j * E;
    const T* kf = k_full + tok * E;
    const T* vf = v_full + tok * E;
    const int G = d / 8;                         // lanes per head within one 256-element step
    float acc = 0.f;
    for (int64_t e0 = 0; e0 < E; e0 += 256) {
        const int64_t e = e0 + 8 * lane;
        float sk = 0.f, sv = 0.f;
        if (e < E) {
            float a[8], c[8];
            load8<T>(kf + e, a);
            load8<T>(ks + e, c);
#pragma unroll
            for (int i = 0; i < 8; ++i) {
                const float t = a[i] - c[i];
                sk = fmaf(t, t, sk);
            }
            load8<T>(vf + e, a);
            load8<T>(vs + e, c);
#pragma unroll
            for (int i = 0; i < 8; ++i) {
                const float t = a[i] - c[i];
                sv = fmaf(t, t, sv);
            }
        }
        for (int o = G / 2; o >= 1; o >>= 1) {
            sk += __shfl_xor_sync(0xffffffffu, sk, o);
            sv += __shfl_xor_sync(0xffffffffu, sv, o);
        }
        // lane gi*G now holds the squared norms of head (e0 + gi*G*8) / d
        for (int gi = 0; gi < 32 / G; ++gi) {
            const float hk2 = __shfl_sync(0xffffffffu, sk, gi * G);
            const float hv2 = __shfl_sync(0xffffffffu, sv, gi * G);
            if (e0 + (int64_t)gi * G * 8 < E) acc += sqrtf(hk2) + sqrtf(hv2);
        }
    }
    if (lane == 0) scores[tok] += acc;
}

}  // namespace

int launch_kv_deviation(int dtype, int B, int L, int Hkv, int d, const void* k_sh, const void* v_sh,
                        const void* k_full, const void* v_full, float* scores, cudaStream_t stream) {
    const int64_t n_tok = (int64_t)B * L;
    if (n_tok == 0) return ACACHE_OK;
    const int64_t blocks = (n_tok + kDevWarps - 1) / kDevWarps;
    if (blocks > 0x7fffffffLL) return ACACHE_ERR_INVALID_ARG;
    if (dtype == ACACHE_BF16)
        kv_deviation_kernel<__nv_bfloat16><<<(unsigned)blocks, kDevWarps * 32, 0, stream>>>(
            n_tok, L, Hkv, d, (const __nv_bfloat16*)k_sh, (const __nv_bfloat16*)v_sh,
            (const __nv_bfloat16*)k_full, (const __nv_bfloat16*)v_full, scores);
    else
        kv_deviation_kernel<float><<<(unsigned)blocks, kDevWarps * 32, 0, stream>>>(
            n_tok, L, Hkv, d, (const float*)k_sh, (const float*)v_sh, (const float*)k_full,
            (const float*)v_full, scores);
    return launch_status();
}

}  // namespace acache
