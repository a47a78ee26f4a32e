// simt_attn.cu -- CUDA-core (FFMA) attention kernels for float32 inputs and for shapes
// the tensor-core kernels do not cover.
//
// Page: "Affix Cache for Diffusion Large Language Models", Sec. 3.2 (probe, Eq. 4-5) and
// Sec. 4.3 / App. C.1 (read-slot attention).  Tensor cores have no float32 mode that keeps
// the float32 inputs' precision, so the float32 path runs here.
//
// Layout of work: one warp per (request, query head, query row).  Lanes take 32 keys at a
// time (one key each: a full d-long dot product against the query row held in shared
// memory), then the warp runs an online softmax over the chunk in the base-2 domain, and
// every lane accumulates d/32 output columns with coalesced value-row loads.
//
// The probe's second pass recomputes the masked-to-affix logits with one thread per
// (request, head, affix offset) and sums fully normalised probabilities over the masked
// rows in ascending order; a last kernel adds the heads in ascending order into scores.
#include "common.cuh"
#include "attn.cuh"

namespace acache {
namespace {

constexpr int kWarpsPerBlock = 4;

template <typename T, int D, typename Keys>
__global__ void __launch_bounds__(kWarpsPerBlock * 32)
simt_attention_kernel(Keys keys, const T* __restrict__ q, T* __restrict__ out, int B, int n_rows,
                      int Hq, int Hkv, int T_len, float scale_log2, float* __restrict__ stat_m,
                      float* __restrict__ stat_l, int32_t* dev_status,
                      const int32_t* __restrict__ q_start) {
    static_assert(D % 32 == 0, "head dim must be a multiple of 32");
    constexpr int kPer = D / 32;
    __shared__ float qs[kWarpsPerBlock][D];
    const int warp = threadIdx.x >> 5, lane = threadIdx.x & 31;
    const int64_t gw = (int64_t)blockIdx.x * kWarpsPerBlock + warp;
    if (gw >= (int64_t)B * Hq * n_rows) return;
    const int i = (int)(gw % n_rows);
    const int h = (int)((gw / n_rows) % Hq);
    const int b = (int)(gw / ((int64_t)n_rows * Hq));
    const int hk = h / (Hq / Hkv);
    // ragged batches: request b owns query rows [q_start[b], q_start[b+1]) and keys.len(b)
    // logical keys; n_rows and T_len are then the largest per-request counts
    int64_t qrow = (int64_t)b * n_rows + i;
    if (q_start) {
        const int nb = q_start[b + 1] - q_start[b], tb = keys.len(b);
        if (nb != 0 && (nb < 0 || nb > n_rows || tb < 1 || tb > T_len)) {
            if (i == 0 && h == 0 && lane == 0) flag(dev_status, ACACHE_DEV_BAD_LENGTH);
            return;
        }
        if (i >= nb) return;
        qrow = q_start[b] + i;
        T_len = tb;
    }
    const int64_t qoff = (qrow * Hq + h) * D;
    for (int c = lane; c < D; c += 32) qs[warp][c] = to_f32(q[qoff + c]);
    __syncwarp();

    float m = -INFINITY, l = 0.f, acc[kPer];
#pragma unroll
    for (int x = 0; x < kPer; ++x) acc[x] = 0.f;
    for (int t0 = 0; t0 < T_len; t0 += 32) {
        const int t = t0 + lane;
        float s = -INFINITY;
        if (t < T_len && !keys.dropped(b, t)) {
            const T *kr, *vr;
            s = 0.f;
            if (keys.rows(b, t, hk, kr, vr, dev_status)) {
                float dot = 0.f;
#pragma unroll 8
                for (int c = 0; c < D; ++c) dot = fmaf(qs[warp][c], to_f32(kr[c]), dot);
                s = dot * scale_log2;
            }
        }
        const float m_new = fmaxf(m, warp_max(s));
        // while every key so far was discarded (m_new = -inf) exponentiate against 0
        const float m_ref = m_new == -INFINITY ? 0.f : m_new;
        const float alpha = fast_exp2(m - m_ref);        // m = -inf on the first chunk -> 0
        const float p = fast_exp2(s - m_ref);
        l = l * alpha + warp_sum(p);
#pragma unroll
        for (int x = 0; x < kPer; ++x) acc[x] *= alpha;
        const int nvalid = min(32, T_len - t0);
        for (int u = 0; u < nvalid; ++u) {
            const float pu = __shfl_sync(0xffffffffu, p, u);
            const T *kr, *vr;
            if (keys.dropped(b, t0 + u) || !keys.rows(b, t0 + u, hk, kr, vr, nullptr))
                continue;   // a discarded key or a zero value row
#pragma unroll
            for (int x = 0; x < kPer; ++x) acc[x] = fmaf(pu, to_f32(vr[lane + 32 * x]), acc[x]);
        }
        m = m_new;
    }
    const float inv_l = l > 0.f ? 1.f / l : 0.f;   // no key left: zeros
    if (out) {
#pragma unroll
        for (int x = 0; x < kPer; ++x) out[qoff + lane + 32 * x] = from_f32<T>(acc[x] * inv_l);
    }
    if (stat_m && lane == 0) {
        const int64_t so = ((int64_t)b * Hq + h) * n_rows + i;
        stat_m[so] = m;
        stat_l[so] = l;
    }
}

// Second probe pass: partial[b][h][j] = sum over masked rows k (ascending) of
// 2^(logit2(k, j) - m_k) / l_k, with the row statistics of the first pass.
template <typename T, int D>
__global__ void __launch_bounds__(128)
simt_probe_colsum_kernel(const T* __restrict__ q, const T* __restrict__ k_aff,
                         const int32_t* __restrict__ masked_rows, int B, int P, int L, int m,
                         int Hq, int Hkv, float scale_log2, const float* __restrict__ stat_m,
                         const float* __restrict__ stat_l, float* __restrict__ partial,
                         int32_t* dev_status) {
    const int64_t gid = (int64_t)blockIdx.x * blockDim.x + threadIdx.x;
    if (gid >= (int64_t)B * Hq * L) return;
    const int j = (int)(gid % L);
    const int h = (int)((gid / L) % Hq);
    const int b = (int)(gid / ((int64_t)L * Hq));
    const int hk = h / (Hq / Hkv);
    const T* kr = k_aff + ((int64_t)j * Hkv + hk) * D;
    float kf[D];
#pragma unroll
    for (int c = 0; c < D; ++c) kf[c] = to_f32(kr[c]);
    float acc = 0.f;
    for (int x = 0; x < m; ++x) {
        const int p = masked_rows[(int64_t)b * m + x];
        if (p < 0 || p >= P) {
            if (j == 0) flag(dev_status, ACACHE_DEV_BAD_ROW);
            continue;
        }
        const T* qr = q + (((int64_t)b * P + p) * Hq + h) * D;
        float dot = 0.f;
#pragma unroll
        for (int c = 0; c < D; ++c) dot = fmaf(to_f32(qr[c]), kf[c], dot);
        const int64_t so = ((int64_t)b * Hq + h) * P + p;
        acc += fast_exp2(dot * scale_log2 - stat_m[so]) / stat_l[so];
    }
    partial[((int64_t)b * Hq + h) * L + j] = acc;
}

template <typename T, int D, typename Keys>
int launch_simt(Keys keys, const void* q, void* out, int B, int n_rows, int Hq, int Hkv, int T_len,
                float scale_log2, float* stat_m, float* stat_l, int32_t* dev_status,
                cudaStream_t stream, const int32_t* q_start = nullptr) {
    const int64_t warps = (int64_t)B * Hq * n_rows;
    if (warps == 0) return ACACHE_OK;
    const int64_t blocks = (warps + kWarpsPerBlock - 1) / kWarpsPerBlock;
    simt_attention_kernel<T, D, Keys><<<(unsigned)blocks, kWarpsPerBlock * 32, 0, stream>>>(
        keys, (const T*)q, (T*)out, B, n_rows, Hq, Hkv, T_len, scale_log2, stat_m, stat_l,
        dev_status, q_start);
    return launch_status();
}

}  // namespace

// ---- entry points used by api.cu ------------------------------------------------------
#define ACACHE_DISPATCH_TD(dtype, d, ...)                                                   \
    do {                                                                                    \
        if ((dtype) == ACACHE_F32 && (d) == 64) { using T = float; constexpr int D = 64; __VA_ARGS__; } \
        else if ((dtype) == ACACHE_F32 && (d) == 128) { using T = float; constexpr int D = 128; __VA_ARGS__; } \
        else if ((dtype) == ACACHE_BF16 && (d) == 64) { using T = __nv_bfloat16; constexpr int D = 64; __VA_ARGS__; } \
        else if ((dtype) == ACACHE_BF16 && (d) == 128) { using T = __nv_bfloat16; constexpr int D = 128; __VA_ARGS__; } \
        else return ACACHE_ERR_UNSUPPORTED;                                                 \
    } while (0)

int launch_simt_slot_attention(const AttnArgs& a, int B, int n_q, const void* q, int T_len,
                               const int32_t* read_slot, const void* k_cache, const void* v_cache,
                               int64_t num_slots, void* out, int32_t* dev_status,
                               cudaStream_t stream, bool drop_none) {
    ACACHE_DISPATCH_TD(a.dtype, a.d, {
        SlotKeys<T> keys{(const T*)k_cache, (const T*)v_cache, read_slot, num_slots, T_len, a.hkv, D,
                         drop_none, nullptr};
        return launch_simt<T, D>(keys, q, out, B, n_q, a.hq, a.hkv, T_len, a.scale * kLog2e,
                                 nullptr, nullptr, dev_status, stream);
    });
}

int launch_simt_slot_attention_varlen(const AttnArgs& a, int B, const int32_t* q_start, int max_q,
                                      const void* q, const int32_t* kv_start, int max_T,
                                      const int32_t* read_slot, const void* k_cache, const void* v_cache,
                                      int64_t num_slots, void* out, int32_t* dev_status,
                                      cudaStream_t stream, bool drop_none) {
    ACACHE_DISPATCH_TD(a.dtype, a.d, {
        SlotKeys<T> keys{(const T*)k_cache, (const T*)v_cache, read_slot, num_slots, max_T, a.hkv, D,
                         drop_none, kv_start};
        return launch_simt<T, D>(keys, q, out, B, max_q, a.hq, a.hkv, max_T, a.scale * kLog2e,
                                 nullptr, nullptr, dev_status, stream, q_start);
    });
}

int launch_simt_probe_pass_a(const AttnArgs& a, int B, int T_len, int l, int L, const void* q,
                             const void* k_req, const void* v_req, const void* k_aff,
                             const void* v_aff, void* out, float* stat_m, float* stat_l,
                             cudaStream_t stream) {
    ACACHE_DISPATCH_TD(a.dtype, a.d, {
        ProbeKeys<T> keys{(const T*)k_req, (const T*)v_req, (const T*)k_aff, (const T*)v_aff,
                          l, L, T_len - L, a.hkv, D};
        return launch_simt<T, D>(keys, q, out, B, T_len - L, a.hq, a.hkv, T_len,
                                 a.scale * kLog2e, stat_m, stat_l, nullptr, stream);
    });
}

int launch_simt_probe_pass_b(const AttnArgs& a, int B, int T_len, int L, const int32_t* masked_rows,
                             int m, const void* q, const void* k_aff, const float* stat_m,
                             const float* stat_l, float* partial, int32_t* dev_status,
                             cudaStream_t stream) {
    const int64_t n = (int64_t)B * a.hq * L;
    if (n == 0) return ACACHE_OK;
    ACACHE_DISPATCH_TD(a.dtype, a.d, {
        simt_probe_colsum_kernel<T, D><<<(unsigned)((n + 127) / 128), 128, 0, stream>>>(
            (const T*)q, (const T*)k_aff, masked_rows, B, T_len - L, L, m, a.hq, a.hkv,
            a.scale * kLog2e, stat_m, stat_l, partial, dev_status);
        return launch_status();
    });
}

}  // namespace acache
