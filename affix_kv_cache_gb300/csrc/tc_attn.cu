// tc_attn.cu -- tensor-core (tcgen05 + TMEM) attention kernels for bf16, head_dim 128.
//
// Page: "Affix Cache for Diffusion Large Language Models" -- Sec. 3.2 (the one-shot probe,
// Eq. 4-5) and Sec. 4.3 / App. C.1 (attention that reads every logical key through the
// per-request read-slot map).  The page's prototype is a Triton kernel on A100; this is a
// GB300-first design:
//
// tc_attn_kernel  (probe forward and read-slot attention; one CTA per 128 query rows of one
//                  (request, query head); 256 threads, 1 CTA per SM)
//   warps 0-3  softmax + epilogue: thread r owns query row r (= TMEM lane r)
//   warp  4    TMEM allocation and the single MMA-issuing thread
//   warps 5-7  producers: warp 5+s gathers key tiles j = s, s+3, ... (128 keys x 256 B for
//              K and for V) with 16-byte cp.async through the key source (the read-slot
//              map, or the affix / own-row split of the probe) straight into the 128-byte-
//              swizzled K-major layout tcgen05.mma reads; warp 5 also loads the Q tile.
//   TMEM (512 columns): S double buffer [0,128) [128,256) (fp32), O [256,384) (fp32).
//   Per key tile j:  S_j = Q K_j^T (SS MMA, M=N=128, K=128)  ->  softmax threads read S_j,
//   exponentiate in base 2 against a lazily raised row maximum (the maximum only moves
//   when it grows by more than 2^8, then O and the row sum are rescaled in place), and
//   write P_j as packed bf16 back over S_j's columns  ->  O += P_j V_j (TS MMA, P from
//   TMEM, V from shared memory as an MN-major operand).  S_{j+1} is issued before PV_j, so
//   the tensor core works on the next tile while the softmax threads exponentiate.
//   The kernel emits O / row-sum and, for the probe, the row statistics (max, sum) that
//   the second probe pass needs to normalise probabilities exactly.
//
// tc_colsum_kernel  (second probe pass: masked-to-affix attention mass; one CTA per
//                    (request, query head, 128 affix keys))
//   D = K_affix_tile Q_masked_chunk^T (SS MMA, M = 128 affix keys, N = 128 masked rows);
//   thread r owns affix key r and sums 2^(logit - m_k) / l_k over the masked rows k in
//   ascending order -- a per-thread serial sum, so the result is deterministic and no
//   cross-thread reduction is needed.
//
// Every mbarrier wait is bounded (about a second); a wait that gives up raises a CTA-wide
// abort flag and ACACHE_DEV_TIMEOUT, every role leaves its loop, in-flight copies and MMAs
// are drained with bounded waits, and TMEM is freed before the CTA exits.
#include "tc_attn.cuh"
#include "ptx.cuh"

namespace acache {
namespace {

using namespace ptx;
using bf16 = __nv_bfloat16;

constexpr int kD = 128;                     // head dim
constexpr int kBM = 128;                    // query rows per CTA
constexpr int kBN = 128;                    // keys per tile
constexpr int kStages = 3;                  // K+V stages (= producer warps)
constexpr int kMmaWarp = 4;
constexpr int kProdWarp0 = 5;
constexpr int kThreads = (kProdWarp0 + kStages) * 32;
constexpr uint32_t kTileBytes = kBN * kD * 2;     // 32 KB: one 128 x 128 bf16 tile
constexpr uint32_t kRegion = kBN * 128;           // 16 KB: 64 columns of a 128-row tile
constexpr uint32_t kSmemBytes = kTileBytes * (1 + 2 * kStages) + 1024;
constexpr uint32_t kTmemCols = 512;
constexpr uint32_t kColS = 0, kColO = 256;
constexpr float kRescaleThreshold = 8.0f;         // log2 units: P values stay below 2^8
constexpr long long kBudget = 1LL << 31;          // cycles (~1 s) before a wait gives up

struct AttnCtl {
    uint64_t q_full;
    uint64_t kv_full[kStages];
    uint64_t kv_empty[kStages];
    uint64_t s_full[2];
    uint64_t p_full[2];
    uint64_t o_done;
    uint64_t drain;
    uint32_t tmem_base;
    int abort;
};

// Bounded wait that also leaves early once another role has aborted.
ACACHE_DEVFN bool wait_bar(uint64_t* bar, uint32_t parity, volatile int* abort_flag,
                           int32_t* dev_status) {
    if (mbar_try_wait(bar, parity)) return true;
    const long long t0 = clock64();
    while (true) {
        if (mbar_try_wait(bar, parity)) return true;
        if (*abort_flag) return false;
        if (clock64() - t0 > kBudget) {
            *abort_flag = 1;
            flag(dev_status, ACACHE_DEV_TIMEOUT);
            return false;
        }
    }
}

// Copy one 128-row x 128-column bf16 tile into the 128-byte-swizzled K-major layout.  Lane
// l holds the location (source, element offset; offset -1 = zero row) of rows l, l+32,
// l+64 and l+96, resolved up front with independent loads; every copy instruction moves two
// whole 256-byte rows (lanes 0-15 one row, 16-31 the next) and takes the row's location
// from its owner lane by shuffle.
template <typename BaseFn>
ACACHE_DEVFN void warp_copy_tile(uint32_t dst, int lane, const int64_t (&off)[4], const int (&src)[4],
                                 BaseFn base_of, const bf16* fallback) {
    const int ch = lane & 15;
#pragma unroll
    for (int u = 0; u < 4; ++u) {
#pragma unroll 4
        for (int i = 0; i < 16; ++i) {
            const int owner = i * 2 + (lane >> 4);
            const long long o = __shfl_sync(0xffffffffu, (long long)off[u], owner);
            const int s = __shfl_sync(0xffffffffu, src[u], owner);
            const bf16* p = o >= 0 ? base_of(s) + o + ch * 8 : fallback;
            cp_async16(dst + sw128_offset(u * 32 + owner, ch, kBN), p, o >= 0 ? 16u : 0u);
        }
    }
}

template <typename Keys>
__global__ void __launch_bounds__(kThreads, 1)
tc_attn_kernel(Keys keys, const bf16* __restrict__ q, bf16* __restrict__ out, int n_rows, int Hq,
               int Hkv, int T_len, float scale_log2, float* __restrict__ stat_m,
               float* __restrict__ stat_l, int32_t* dev_status) {
    extern __shared__ uint8_t dsm[];
    __shared__ AttnCtl ctl;
    const uint32_t base = (smem_u32(dsm) + 1023u) & ~1023u;
    const uint32_t sQ = base;
    const int n_qt = (n_rows + kBM - 1) / kBM;
    const int qt = blockIdx.x % n_qt;
    const int h = (blockIdx.x / n_qt) % Hq;
    const int b = blockIdx.x / (n_qt * Hq);
    const int hk = h / (Hq / Hkv);
    const int q0 = qt * kBM;
    const int n_kv = (T_len + kBN - 1) / kBN;
    const int warp = threadIdx.x >> 5, lane = threadIdx.x & 31;
    volatile int* abort_flag = &ctl.abort;

    if (threadIdx.x == 0) {
        mbar_init(&ctl.q_full, 32);
        for (int s = 0; s < kStages; ++s) {
            mbar_init(&ctl.kv_full[s], 32);
            mbar_init(&ctl.kv_empty[s], 1);
        }
        for (int i = 0; i < 2; ++i) {
            mbar_init(&ctl.s_full[i], 1);
            mbar_init(&ctl.p_full[i], 128);
        }
        mbar_init(&ctl.o_done, 1);
        mbar_init(&ctl.drain, 1);
        ctl.abort = 0;
        fence_mbar_init();
    }
    if (warp == kMmaWarp) {
        tmem_alloc(&ctl.tmem_base, kTmemCols);
        tmem_relinquish();
    }
    tc_fence_before();
    __syncthreads();
    tc_fence_after();
    const uint32_t tmem = ctl.tmem_base;

    if (warp >= kProdWarp0) {
        // ------------------------------------------------------------------ producers
        const int pw = warp - kProdWarp0;
        if (pw == 0) {
            int64_t off[4];
            int src[4];
#pragma unroll
            for (int u = 0; u < 4; ++u) {
                const int i = q0 + u * 32 + lane;
                src[u] = 0;
                off[u] = i < n_rows ? (((int64_t)b * n_rows + i) * Hq + h) * kD : -1;
            }
            warp_copy_tile(sQ, lane, off, src, [&](int) { return q; }, q);
            cp_async_commit();
            cp_async_wait<0>();
            fence_proxy_async_smem();
            mbar_arrive(&ctl.q_full);
        }
        const uint32_t sK = base + kTileBytes * (1 + 2 * pw);
        const uint32_t sV = sK + kTileBytes;
        const bf16* fallback = q;
        for (int j = pw; j < n_kv; j += kStages) {
            // resolve the tile's 128 key rows first (independent loads), then wait for the stage
            const int t0 = j * kBN;
            int64_t off[4];
            int src[4];
#pragma unroll
            for (int u = 0; u < 4; ++u) {
                const int t = t0 + u * 32 + lane;
                src[u] = 0;
                off[u] = t < T_len ? keys.locate(b, t, hk, src[u], dev_status) : -1;
            }
            if (j >= kStages &&
                !wait_bar(&ctl.kv_empty[pw], ((j / kStages) - 1) & 1, abort_flag, dev_status))
                break;
            warp_copy_tile(sK, lane, off, src, [&](int s) { return keys.kbase(s); }, fallback);
            warp_copy_tile(sV, lane, off, src, [&](int s) { return keys.vbase(s); }, fallback);
            cp_async_commit();
            cp_async_wait<0>();
            fence_proxy_async_smem();
            mbar_arrive(&ctl.kv_full[pw]);
        }
        cp_async_wait<0>();
    } else if (warp == kMmaWarp) {
        // ------------------------------------------------------------------ MMA issuer
        if (lane == 0) {
            const uint32_t idS = idesc_bf16(kBM, kBN, false, false);
            const uint32_t idO = idesc_bf16(kBM, kD, false, true);
            auto issue_s = [&](int j) {
                const uint32_t sK = base + kTileBytes * (1 + 2 * (j % kStages));
                const uint32_t d = tmem + kColS + (uint32_t)(j & 1) * kBN;
#pragma unroll
                for (int k = 0; k < kD / 16; ++k) {
                    const uint32_t ko = (uint32_t)(k >> 2) * kRegion + (uint32_t)(k & 3) * 32u;
                    umma_ss(d, sdesc_sw128(sQ + ko, 16, 1024), sdesc_sw128(sK + ko, 16, 1024), idS,
                            k > 0);
                }
                umma_commit(&ctl.s_full[j & 1]);
            };
            bool ok = wait_bar(&ctl.q_full, 0, abort_flag, dev_status) &&
                      wait_bar(&ctl.kv_full[0], 0, abort_flag, dev_status);
            if (ok) {
                tc_fence_after();
                issue_s(0);
            }
            for (int j = 0; ok && j < n_kv; ++j) {
                if (j + 1 < n_kv) {
                    ok = wait_bar(&ctl.kv_full[(j + 1) % kStages], ((j + 1) / kStages) & 1,
                                  abort_flag, dev_status);
                    if (!ok) break;
                    tc_fence_after();
                    issue_s(j + 1);
                }
                ok = wait_bar(&ctl.p_full[j & 1], (j >> 1) & 1, abort_flag, dev_status);
                if (!ok) break;
                tc_fence_after();
                const uint32_t sV = base + kTileBytes * (2 + 2 * (j % kStages));
                const uint32_t p_tmem = tmem + kColS + (uint32_t)(j & 1) * kBN;
#pragma unroll
                for (int k = 0; k < kBN / 16; ++k)
                    umma_ts(tmem + kColO, p_tmem + k * 8, sdesc_sw128(sV + k * 2048, kRegion, 1024),
                            idO, (j > 0 || k > 0));
                umma_commit(&ctl.o_done);
                umma_commit(&ctl.kv_empty[j % kStages]);
            }
            // no MMA may still run when TMEM is released
            umma_commit(&ctl.drain);
            mbar_wait(&ctl.drain, 0, kBudget);
        }
        __syncwarp();
    } else {
        // ------------------------------------------------------------------ softmax + epilogue
        const int r = threadIdx.x;                         // query row in the tile
        const uint32_t lane_base = tmem + ((uint32_t)(warp * 32) << 16);
        float m_used = -INFINITY, l_sum = 0.f;
        bool ok = true;
        for (int j = 0; j < n_kv; ++j) {
            const int bs = j & 1;
            ok = __all_sync(0xffffffffu, wait_bar(&ctl.s_full[bs], (j >> 1) & 1, abort_flag, dev_status));
            if (!ok) break;
            tc_fence_after();
            uint32_t v[4][32];
#pragma unroll
            for (int c = 0; c < 4; ++c) tmem_ld32(lane_base + kColS + bs * kBN + c * 32, v[c]);
            tmem_ld_wait();
            const int valid = min(kBN, T_len - j * kBN);
            float mt = -INFINITY;
#pragma unroll
            for (int c = 0; c < 4; ++c)
#pragma unroll
                for (int i = 0; i < 32; ++i) {
                    const float x = (c * 32 + i < valid) ? __uint_as_float(v[c][i]) * scale_log2 : -INFINITY;
                    v[c][i] = __float_as_uint(x);
                    mt = fmaxf(mt, x);
                }
            float alpha = 1.f;
            bool resc = false;
            if (j == 0) {
                m_used = mt;
            } else if (mt > m_used + kRescaleThreshold) {
                alpha = fast_exp2(m_used - mt);
                m_used = mt;
                resc = true;
            }
            if (__any_sync(0xffffffffu, resc)) {
                // O holds PV_0..PV_{j-1}: wait for the last one, rescale in place
                ok = __all_sync(0xffffffffu, wait_bar(&ctl.o_done, (j - 1) & 1, abort_flag, dev_status));
                if (!ok) break;
                tc_fence_after();
#pragma unroll
                for (int c = 0; c < 4; ++c) {
                    uint32_t o[32];
                    tmem_ld32(lane_base + kColO + c * 32, o);
                    tmem_ld_wait();
#pragma unroll
                    for (int i = 0; i < 32; ++i) o[i] = __float_as_uint(__uint_as_float(o[i]) * alpha);
                    tmem_st32(lane_base + kColO + c * 32, o);
                }
                tmem_st_wait();
            }
            l_sum *= alpha;
            uint32_t pk[2][32];
#pragma unroll
            for (int c = 0; c < 4; ++c)
#pragma unroll
                for (int i = 0; i < 32; i += 2) {
                    const float p0 = fast_exp2(__uint_as_float(v[c][i]) - m_used);
                    const float p1 = fast_exp2(__uint_as_float(v[c][i + 1]) - m_used);
                    l_sum += p0 + p1;
                    __nv_bfloat162 two = __floats2bfloat162_rn(p0, p1);   // low half = lower key
                    pk[c >> 1][(c & 1) * 16 + (i >> 1)] = *reinterpret_cast<uint32_t*>(&two);
                }
            // P_j (bf16 pairs, 64 columns) overwrites the first half of S_j's columns
            tmem_st32(lane_base + kColS + bs * kBN, pk[0]);
            tmem_st32(lane_base + kColS + bs * kBN + 32, pk[1]);
            tmem_st_wait();
            tc_fence_before();
            mbar_arrive(&ctl.p_full[bs]);
        }
        // `drain` is committed after the last PV; a parity wait on o_done could be fooled here,
        // because PV_{n-2} may still be running when the last P is handed over
        if (ok) ok = __all_sync(0xffffffffu, wait_bar(&ctl.drain, 0, abort_flag, dev_status));
        if (ok) {
            tc_fence_after();
            const int i = q0 + r;
            const float inv_l = 1.f / l_sum;
            bf16* orow = out ? out + (((int64_t)b * n_rows + i) * Hq + h) * kD : nullptr;
#pragma unroll
            for (int c = 0; c < 4; ++c) {
                uint32_t o[32];
                tmem_ld32(lane_base + kColO + c * 32, o);
                tmem_ld_wait();
                if (orow && i < n_rows) {
                    uint32_t pkd[16];
#pragma unroll
                    for (int x = 0; x < 16; ++x) {
                        __nv_bfloat162 two = __floats2bfloat162_rn(__uint_as_float(o[2 * x]) * inv_l,
                                                                   __uint_as_float(o[2 * x + 1]) * inv_l);
                        pkd[x] = *reinterpret_cast<uint32_t*>(&two);
                    }
                    uint4* dst = reinterpret_cast<uint4*>(orow + c * 32);
#pragma unroll
                    for (int x = 0; x < 4; ++x)
                        dst[x] = make_uint4(pkd[4 * x], pkd[4 * x + 1], pkd[4 * x + 2], pkd[4 * x + 3]);
                }
            }
            if (stat_m && i < n_rows) {
                const int64_t so = ((int64_t)b * Hq + h) * n_rows + i;
                stat_m[so] = m_used;
                stat_l[so] = l_sum;
            }
        }
    }
    tc_fence_before();
    __syncthreads();
    tc_fence_after();
    if (warp == kMmaWarp) tmem_dealloc(tmem, kTmemCols);
}

// ------------------------------------------------------------------------------------------
// Second probe pass.
constexpr int kCsStages = 2;
constexpr int kCsThreads = (kProdWarp0 + kCsStages) * 32;
constexpr uint32_t kCsSmemBytes = kTileBytes * (1 + kCsStages) + 1024;
constexpr uint32_t kCsTmemCols = 256;

struct ColsumCtl {
    uint64_t a_full;
    uint64_t b_full[kCsStages];
    uint64_t b_empty[kCsStages];      // MMA finished reading the Q chunk of the stage
    uint64_t d_full[2];
    uint64_t cons_done[2];            // consumers finished with D buffer and stats of a stage
    uint64_t drain;
    uint32_t tmem_base;
    int abort;
    float st_m[kCsStages][kBN];       // row maximum (log2 domain) of each masked row; +inf = skip
    float st_il[kCsStages][kBN];      // 1 / row sum; 0 = skip
};

__global__ void __launch_bounds__(kCsThreads, 1)
tc_colsum_kernel(const bf16* __restrict__ q, const bf16* __restrict__ k_aff,
                 const int32_t* __restrict__ masked, int P, int L, int m, int Hq, int Hkv,
                 float scale_log2, const float* __restrict__ stat_m,
                 const float* __restrict__ stat_l, float* __restrict__ partial,
                 int32_t* dev_status) {
    extern __shared__ uint8_t dsm[];
    __shared__ ColsumCtl ctl;
    const uint32_t base = (smem_u32(dsm) + 1023u) & ~1023u;
    const uint32_t sA = base;
    const int n_jt = (L + kBN - 1) / kBN;
    const int jt = blockIdx.x % n_jt;
    const int h = (blockIdx.x / n_jt) % Hq;
    const int b = blockIdx.x / (n_jt * Hq);
    const int hk = h / (Hq / Hkv);
    const int j0 = jt * kBN;
    const int n_ch = (m + kBN - 1) / kBN;
    const int warp = threadIdx.x >> 5, lane = threadIdx.x & 31;
    volatile int* abort_flag = &ctl.abort;

    if (threadIdx.x == 0) {
        mbar_init(&ctl.a_full, 32);
        for (int s = 0; s < kCsStages; ++s) {
            mbar_init(&ctl.b_full[s], 32);
            mbar_init(&ctl.b_empty[s], 1);
        }
        for (int i = 0; i < 2; ++i) {
            mbar_init(&ctl.d_full[i], 1);
            mbar_init(&ctl.cons_done[i], 128);
        }
        mbar_init(&ctl.drain, 1);
        ctl.abort = 0;
        fence_mbar_init();
    }
    if (warp == kMmaWarp) {
        tmem_alloc(&ctl.tmem_base, kCsTmemCols);
        tmem_relinquish();
    }
    tc_fence_before();
    __syncthreads();
    tc_fence_after();
    const uint32_t tmem = ctl.tmem_base;
    const float* sm_row = stat_m + ((int64_t)b * Hq + h) * P;
    const float* sl_row = stat_l + ((int64_t)b * Hq + h) * P;
    const int32_t* mrow = masked + (int64_t)b * m;

    if (warp >= kProdWarp0) {
        const int pw = warp - kProdWarp0;
        if (pw == 0) {
            int64_t off[4];
            int src[4];
#pragma unroll
            for (int u = 0; u < 4; ++u) {
                const int j = j0 + u * 32 + lane;
                src[u] = 0;
                off[u] = j < L ? ((int64_t)j * Hkv + hk) * kD : -1;
            }
            warp_copy_tile(sA, lane, off, src, [&](int) { return k_aff; }, k_aff);
            cp_async_commit();
            cp_async_wait<0>();
            fence_proxy_async_smem();
            mbar_arrive(&ctl.a_full);
        }
        const uint32_t sB = base + kTileBytes * (1 + pw);
        for (int c = pw; c < n_ch; c += kCsStages) {
            if (c >= kCsStages) {
                const uint32_t par = ((c / kCsStages) - 1) & 1;
                if (!wait_bar(&ctl.b_empty[pw], par, abort_flag, dev_status)) break;
                if (!wait_bar(&ctl.cons_done[pw], par, abort_flag, dev_status)) break;
            }
            const int k0 = c * kBN;
            int64_t off[4];
            int src[4];
#pragma unroll
            for (int u = 0; u < 4; ++u) {
                const int row = u * 32 + lane;
                const int k = k0 + row;
                const int p = k < m ? mrow[k] : -1;
                const bool good = p >= 0 && p < P;
                if (k < m && !good) flag(dev_status, ACACHE_DEV_BAD_ROW);
                src[u] = 0;
                off[u] = good ? (((int64_t)b * P + p) * Hq + h) * kD : -1;
                ctl.st_m[pw][row] = good ? sm_row[p] : INFINITY;
                ctl.st_il[pw][row] = good ? 1.f / sl_row[p] : 0.f;
            }
            warp_copy_tile(sB, lane, off, src, [&](int) { return q; }, q);
            cp_async_commit();
            cp_async_wait<0>();
            fence_proxy_async_smem();
            mbar_arrive(&ctl.b_full[pw]);
        }
        cp_async_wait<0>();
    } else if (warp == kMmaWarp) {
        if (lane == 0) {
            const uint32_t id = idesc_bf16(kBN, kBN, false, false);
            bool ok = wait_bar(&ctl.a_full, 0, abort_flag, dev_status);
            for (int c = 0; ok && c < n_ch; ++c) {
                const int s = c % kCsStages, db = c & 1;
                ok = wait_bar(&ctl.b_full[s], (c / kCsStages) & 1, abort_flag, dev_status);
                if (ok && c >= 2) ok = wait_bar(&ctl.cons_done[db], ((c >> 1) - 1) & 1, abort_flag, dev_status);
                if (!ok) break;
                tc_fence_after();
                const uint32_t sB = base + kTileBytes * (1 + s);
#pragma unroll
                for (int k = 0; k < kD / 16; ++k) {
                    const uint32_t ko = (uint32_t)(k >> 2) * kRegion + (uint32_t)(k & 3) * 32u;
                    umma_ss(tmem + db * kBN, sdesc_sw128(sA + ko, 16, 1024),
                            sdesc_sw128(sB + ko, 16, 1024), id, k > 0);
                }
                umma_commit(&ctl.d_full[db]);
                umma_commit(&ctl.b_empty[s]);
            }
            umma_commit(&ctl.drain);
            mbar_wait(&ctl.drain, 0, kBudget);
        }
        __syncwarp();
    } else {
        const int r = threadIdx.x;                         // affix key j0 + r
        const uint32_t lane_base = tmem + ((uint32_t)(warp * 32) << 16);
        float acc = 0.f;
        bool ok = true;
        for (int c = 0; c < n_ch; ++c) {
            const int s = c % kCsStages, db = c & 1;
            // the stats of this chunk were published with b_full; D with d_full
            ok = __all_sync(0xffffffffu,
                            wait_bar(&ctl.b_full[s], (c / kCsStages) & 1, abort_flag, dev_status) &&
                            wait_bar(&ctl.d_full[db], (c >> 1) & 1, abort_flag, dev_status));
            if (!ok) break;
            tc_fence_after();
#pragma unroll
            for (int cc = 0; cc < 4; ++cc) {
                uint32_t v[32];
                tmem_ld32(lane_base + db * kBN + cc * 32, v);
                tmem_ld_wait();
#pragma unroll
                for (int i = 0; i < 32; ++i) {
                    const int k = cc * 32 + i;
                    acc += fast_exp2(__uint_as_float(v[i]) * scale_log2 - ctl.st_m[s][k]) * ctl.st_il[s][k];
                }
            }
            tc_fence_before();
            mbar_arrive(&ctl.cons_done[db]);
        }
        if (ok && j0 + r < L) partial[((int64_t)b * Hq + h) * L + j0 + r] = acc;
    }
    tc_fence_before();
    __syncthreads();
    tc_fence_after();
    if (warp == kMmaWarp) tmem_dealloc(tmem, kCsTmemCols);
}

template <typename Keys>
int launch_attn(Keys keys, const void* q, void* out, int B, int n_rows, int Hq, int Hkv, int T_len,
                float scale_log2, float* stat_m, float* stat_l, int32_t* dev_status,
                cudaStream_t stream) {
    const int64_t ctas = (int64_t)B * Hq * ((n_rows + kBM - 1) / kBM);
    if (ctas == 0) return ACACHE_OK;
    if (ctas > 0x7fffffff) return ACACHE_ERR_INVALID_ARG;
    auto kern = tc_attn_kernel<Keys>;
    if (cudaFuncSetAttribute(kern, cudaFuncAttributeMaxDynamicSharedMemorySize, kSmemBytes) != cudaSuccess) {
        (void)cudaGetLastError();
        return ACACHE_ERR_CUDA;
    }
    kern<<<(unsigned)ctas, kThreads, kSmemBytes, stream>>>(keys, (const bf16*)q, (bf16*)out, n_rows, Hq,
                                                         Hkv, T_len, scale_log2, stat_m, stat_l,
                                                         dev_status);
    return launch_status();
}

}  // namespace

bool tc_supported(const AttnArgs& a) { return a.dtype == ACACHE_BF16 && a.d == kD; }

int launch_tc_slot_attention(const AttnArgs& a, int B, int n_q, const void* q, int T_len,
                             const int32_t* read_slot, const void* k_cache, const void* v_cache,
                             int64_t num_slots, void* out, int32_t* dev_status,
                             cudaStream_t stream) {
    SlotKeys<bf16> keys{(const bf16*)k_cache, (const bf16*)v_cache, read_slot, num_slots, T_len,
                        a.hkv, kD};
    return launch_attn(keys, q, out, B, n_q, a.hq, a.hkv, T_len, a.scale * kLog2e, nullptr, nullptr,
                       dev_status, stream);
}

int launch_tc_probe_pass_a(const AttnArgs& a, int B, int T_len, int l, int L, const void* q,
                           const void* k_req, const void* v_req, const void* k_aff,
                           const void* v_aff, void* out, float* stat_m, float* stat_l,
                           int32_t* dev_status, cudaStream_t stream) {
    ProbeKeys<bf16> keys{(const bf16*)k_req, (const bf16*)v_req, (const bf16*)k_aff,
                         (const bf16*)v_aff, l, L, T_len - L, a.hkv, kD};
    return launch_attn(keys, q, out, B, T_len - L, a.hq, a.hkv, T_len, a.scale * kLog2e, stat_m,
                       stat_l, dev_status, stream);
}

int launch_tc_probe_pass_b(const AttnArgs& a, int B, int T_len, int L, const int32_t* masked_rows,
                           int m, const void* q, const void* k_aff, const float* stat_m,
                           const float* stat_l, float* partial, int32_t* dev_status,
                           cudaStream_t stream) {
    const int64_t ctas = (int64_t)B * a.hq * ((L + kBN - 1) / kBN);
    if (ctas == 0) return ACACHE_OK;
    if (m == 0) {   // no masked rows: every affix key receives zero mass
        if (cudaMemsetAsync(partial, 0, (size_t)B * a.hq * L * sizeof(float), stream) != cudaSuccess)
            return ACACHE_ERR_CUDA;
        return ACACHE_OK;
    }
    if (cudaFuncSetAttribute(tc_colsum_kernel, cudaFuncAttributeMaxDynamicSharedMemorySize,
                             kCsSmemBytes) != cudaSuccess) {
        (void)cudaGetLastError();
        return ACACHE_ERR_CUDA;
    }
    tc_colsum_kernel<<<(unsigned)ctas, kCsThreads, kCsSmemBytes, stream>>>(
        (const bf16*)q, (const bf16*)k_aff, masked_rows, T_len - L, L, m, a.hq, a.hkv,
        a.scale * kLog2e, stat_m, stat_l, partial, dev_status);
    return launch_status();
}

}  // namespace acache
