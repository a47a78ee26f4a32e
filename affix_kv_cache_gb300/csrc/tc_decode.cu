// tc_decode.cu -- read-slot attention for few query rows per (request, KV head): the
// block-decode step, where the current block's queries attend over every logical key of the
// request through the read-slot map.
//
// Page: "Affix Cache for Diffusion Large Language Models" -- Sec. 4.3 and App. C.1 (attention
// that gathers K/V through the read map; the decode loop attends with the current block's
// queries) and Sec. 5 (block length 32).  bf16, head_dim 128, tcgen05 + TMEM, TMA-fed.
//
// With 32 queries per request the work per (request, head) is one Q tile against a long key
// stream: memory-bound for multi-head attention.  The design follows from that:
//   * Rows are (query, head-in-group) pairs of one KV head, so all query heads of a GQA group
//     share one gathered K/V stream (a CTA row block holds whole queries: qpb queries x g heads).
//   * A row block of at most 32 (64) rows is replicated 4 (2) times across the 128 TMEM lanes
//     and each replica takes a quarter (half) of every key tile, so the four softmax warps
//     share the exponentials of a tile instead of one warp doing all of them.  Each replica
//     writes its P columns into a TMEM buffer whose other columns stay zero, so one
//     M = 128 PV MMA adds every replica's keys into its own O rows.
//   * S is double-buffered in TMEM: S(j+2) is computed while the softmax of tile j+1 runs.
//   * The key range of a (request, KV head, row block) is split across a thread-block cluster
//     of cs CTAs when that fills the SMs better; every CTA leaves its partial (row maximum,
//     row sum, unnormalised O) per replica in shared memory and the cluster combines them
//     through distributed shared memory -- no workspace and no second launch.
//
// Warp roles (384 threads, 1 CTA per SM):
//   warps 0-3   softmax + epilogue: thread r owns TMEM lane r
//   warp 4      TMEM allocation; lane 0 issues every MMA
//   warps 6-11  TMA producers: warps 6-8 gather K tiles, 9-11 V tiles (a tile's 64
//               `tile::gather4` loads of 4 pool rows x 64 columns, 21-22 per warp: a gather4
//               costs its warp tens of cycles of issue, so more warps gather faster); warp 6
//               lane 0 loads Q
// TMEM (512 columns): S0 [0,128)  S1 [128,256)  O [256,384)  P0 [384,448)  P1 [448,512).
//
// Every mbarrier wait is bounded; a wait that gives up raises a CTA-wide abort flag and
// ACACHE_DEV_TIMEOUT, roles leave their loops, in-flight MMAs are drained with a bounded wait,
// TMA loads issued before the abort get a bounded ~30 us to land, and TMEM is freed before the
// CTA exits; the cluster barriers are reached on every path.
#include <cuda.h>

#include <algorithm>
#include <atomic>

#include "tc_attn.cuh"
#include "ptx.cuh"

namespace acache {
namespace {

using namespace ptx;
using bf16 = __nv_bfloat16;

constexpr int kD = 128;
constexpr int kBM = 128;                  // TMEM lanes / rows of the Q tile
constexpr int kBN = 128;                  // keys per tile
constexpr int kStages = 3;                // K ring and V ring depth
constexpr int kMmaWarp = 4;
constexpr int kProdWarp = 6;              // first TMA producer warp
constexpr int kPerRing = 3;               // producer warps per ring: K warps 6-8, V 9-11
constexpr int kThreads = 12 * 32;
static_assert(kThreads == (kProdWarp + 2 * kPerRing) * 32, "warp roles");
constexpr int kMaxCluster = 4;
// Registers: 384 threads x 168 at launch = 64512; the softmax warpgroup grows to 232, the
// other two shrink to 136: 128*232 + 256*136 = 64512.
constexpr int kLaunchRegs = 168, kRegSoftmax = 232, kRegOther = 136;
static_assert(128 * kRegSoftmax + 256 * kRegOther <= kThreads * kLaunchRegs, "register split");
constexpr uint32_t kTileBytes = kBN * kD * 2;          // 32 KB
constexpr uint32_t kRegion = kBN * 128;                // 16 KB: 64 columns of a 128-row tile
constexpr uint32_t kSmemBytes = kTileBytes * (1 + 2 * kStages) + 1024;
constexpr uint32_t kTmemCols = 512;
constexpr uint32_t kColS0 = 0, kColO = 256, kColP0 = 384;
constexpr float kRescaleThreshold = 8.0f;
constexpr long long kDrainBudget = 1LL << 31;   // cycles: MMAs issued before an abort
constexpr long long kLandBudget = 1LL << 21;    // cycles (~1 ms): TMA loads issued before an abort

struct DecParams {
    CUtensorMap tm_q;     // 4-D [B][n_q][Hq][d], box {64, g, qpb, 1}
    CUtensorMap tm_k;     // 2-D pool rows [num_slots*Hkv][d], box {64, 1} (gather4)
    CUtensorMap tm_v;
    const int32_t* read_slot;
    bf16* out;
    int32_t* dev_status;
    int64_t num_slots;
    int n_q, Hq, Hkv, g, T_len;
    int qpb;              // queries per row block
    int n_rb;             // row blocks per (request, KV head)
    int cs;               // CTAs per cluster (key-range split)
    float scale_log2;
    long long budget;     // cycles a pipeline wait may take before it gives up
};

struct DecCtl {
    uint64_t q_full;
    uint64_t k_full[kStages], k_empty[kStages];
    uint64_t v_full[kStages], v_empty[kStages];
    uint64_t s_full[2];
    uint64_t p_full[2];
    uint64_t pv_done;     // phase j completes when PV(j) has completed
    uint64_t drain;
    uint32_t tmem_base;
    int abort;
    int unlanded;         // abort path: some TMA load issued before the abort may not have landed
    float part_m[kBM];    // per TMEM lane: row maximum (log2 units) of the replica's keys
    float part_l[kBM];    // per TMEM lane: row sum
};

ACACHE_DEVFN bool wait_bar(uint64_t* bar, uint32_t parity, volatile int* abort_flag, int32_t* dev_status,
                           long long budget) {
    if (mbar_try_wait(bar, parity)) return true;
    const long long t0 = clock64();
    while (true) {
        if (mbar_try_wait(bar, parity)) return true;
        if (*abort_flag) return false;
        if (clock64() - t0 > budget) {
            *abort_flag = 1;
            flag(dev_status, ACACHE_DEV_TIMEOUT);
            return false;
        }
    }
}

// Float4 slot q of lane row r in the partial-O area (512-byte rows; the XOR spreads the 32
// lanes of a warp over the banks).
ACACHE_DEVFN uint32_t part_off(int r, int q) { return (uint32_t)r * 512u + (uint32_t)((q ^ (r & 31)) << 4); }

// kDrop: a read-slot entry equal to ACACHE_SLOT_NONE marks a discarded key (the page's
// DropNA ablation, Sec. 5.3): it takes no part in the softmax.
template <int REP, bool kDrop>
__global__ void __launch_bounds__(kThreads, 1)
tc_decode_kernel(const __grid_constant__ DecParams p) {
    extern __shared__ uint8_t dsm[];
    __shared__ DecCtl ctl;
    const uint32_t base = (smem_u32(dsm) + 1023u) & ~1023u;
    uint8_t* base_ptr = dsm + (base - smem_u32(dsm));
    const uint32_t sQ = base;
    auto sK = [&](int s) { return base + kTileBytes * (uint32_t)(1 + s); };
    auto sV = [&](int s) { return base + kTileBytes * (uint32_t)(1 + kStages + s); };
    constexpr int G = kBM / REP;                    // lanes per replica
    const int cs = p.cs;
    const int cr = (int)(blockIdx.x % (unsigned)cs);     // rank in the cluster = key-range part
    const int unit = (int)(blockIdx.x / (unsigned)cs);
    const int rb = unit % p.n_rb;
    const int hk = (unit / p.n_rb) % p.Hkv;
    const int b = unit / (p.n_rb * p.Hkv);
    const int q0 = rb * p.qpb;
    const int rows_valid = min(p.qpb, p.n_q - q0) * p.g;   // packed rows of this block (<= G)
    const int n_all = (p.T_len + kBN - 1) / kBN;
    const int kt0 = (int)((int64_t)cr * n_all / cs);
    const int n_kv = (int)((int64_t)(cr + 1) * n_all / cs) - kt0;   // >= 1 (cs <= n_all)
    const int warp = threadIdx.x >> 5, lane = threadIdx.x & 31, wg = warp >> 2;
    volatile int* abort_flag = &ctl.abort;
    int32_t* dev_status = p.dev_status;
    const long long budget = p.budget;

    if (threadIdx.x == 0) {
        mbar_init(&ctl.q_full, 1);
        for (int s = 0; s < kStages; ++s) {
            mbar_init(&ctl.k_full[s], 1);
            mbar_init(&ctl.k_empty[s], 1);
            mbar_init(&ctl.v_full[s], 1);
            mbar_init(&ctl.v_empty[s], 1);
        }
        for (int t = 0; t < 2; ++t) {
            mbar_init(&ctl.s_full[t], 1);
            mbar_init(&ctl.p_full[t], 128);
        }
        mbar_init(&ctl.pv_done, 1);
        mbar_init(&ctl.drain, 1);
        ctl.abort = 0;
        ctl.unlanded = 0;
        fence_mbar_init();
    }
    // Q rows the TMA does not write (past the block's packed rows) must be finite: zero the
    // whole Q tile first (generic-proxy writes, made visible to the async proxy)
    for (uint32_t o = threadIdx.x * 16u; o < kTileBytes; o += kThreads * 16u)
        *reinterpret_cast<uint4*>(base_ptr + o) = make_uint4(0u, 0u, 0u, 0u);
    fence_proxy_async_smem();
    if (warp == kMmaWarp) {
        tmem_alloc(&ctl.tmem_base, kTmemCols);
        tmem_relinquish();
    }
    tc_fence_before();
    __syncthreads();
    tc_fence_after();
    const uint32_t tmem = ctl.tmem_base;
    bool ok = true;

    if (wg >= 1) {
        setmaxnreg_dec<kRegOther>();
        if (warp >= kProdWarp) {
            // -------------------------------------------------------------- TMA producers
            const int pw = warp - kProdWarp;
            if (pw == 0 && lane == 0) {
                tma_prefetch_desc(&p.tm_q);
                tma_prefetch_desc(&p.tm_k);
                tma_prefetch_desc(&p.tm_v);
                // replica w of the row block lands at lanes [w*G, w*G + qpb*g)
                mbar_arrive_expect_tx(&ctl.q_full, (uint32_t)(REP * 2 * 128 * p.g * p.qpb));
                for (int w = 0; w < REP; ++w) {
                    tma_load_4d(sQ + (uint32_t)(w * G) * 128u, &p.tm_q, 0, hk * p.g, q0, b, &ctl.q_full);
                    tma_load_4d(sQ + kRegion + (uint32_t)(w * G) * 128u, &p.tm_q, 64, hk * p.g, q0, b, &ctl.q_full);
                }
            }
            const bool is_v = pw >= kPerRing;
            const int pi = pw - (is_v ? kPerRing : 0);    // place among the ring's warps
            uint64_t* full = is_v ? ctl.v_full : ctl.k_full;
            uint64_t* empty = is_v ? ctl.v_empty : ctl.k_empty;
            const CUtensorMap* tm = is_v ? &p.tm_v : &p.tm_k;
            const bool leader = pi == 0 && lane == 0;
            const int oob_row = (int)(p.num_slots * p.Hkv);
            // this lane's gather x = 4-row group x / 2 of the tile, column half x % 2; lanes with
            // x >= 64 have none (every warp of the ring still has some in every tile)
            const int x = kPerRing * lane + pi;
            const bool gathers = x < 64;
            const int gi = x >> 1, half = x & 1;
            const int32_t* rs = p.read_slot + (int64_t)b * p.T_len;
            auto resolve = [&](int j, int (&rows)[4]) {
    #pragma unroll
                for (int u = 0; u < 4; ++u) {
                    const int t = (kt0 + j) * kBN + 4 * gi + u;
                    rows[u] = oob_row;
                    if (gathers && j < n_kv && t < p.T_len) {
                        const int64_t slot = rs[t];
                        if (slot >= 0 && slot < p.num_slots)
                            rows[u] = (int)(slot * p.Hkv + hk);
                        else if (!is_v && half == 0 && !(kDrop && slot == ACACHE_SLOT_NONE))
                            flag(dev_status, ACACHE_DEV_BAD_SLOT);
                    }
                }
            };
            int next[4];
            resolve(0, next);
            // store-then-attend: wait for the preceding store grid before reading the pool
            grid_dependency_wait();
            int armed = -1;                               // last entry this warp loaded into
            for (int j = 0; j < n_kv; ++j) {
                const int s = j % kStages;
                int rows[4] = {next[0], next[1], next[2], next[3]};
                resolve(j + 1, next);
                if (j >= kStages &&
                    !__all_sync(0xffffffffu, wait_bar(&empty[s], ((j / kStages) - 1) & 1, abort_flag, dev_status, budget)))
                    break;
                if (leader) mbar_arrive_expect_tx(&full[s], kTileBytes);
                armed = j;
                __syncwarp();
                if (gathers)
                    tma_gather4((is_v ? sV(s) : sK(s)) + (uint32_t)half * kRegion + (uint32_t)gi * 512u, tm,
                                half * 64, rows[0], rows[1], rows[2], rows[3], &full[s]);
            }
            // Abort: the loads this warp issued land before the CTA exits.  Only the last entry
            // of each stage can still have loads in flight, so wait, bounded, for those phases
            // (and for the query rows); a phase that another warp of the ring never loaded
            // into cannot complete, and then the CTA holds for a fixed time instead.
            if (*abort_flag) {
                bool landed = is_v || pi != 0 || mbar_wait(&ctl.q_full, 0, kLandBudget);
                for (int e = max(0, armed - kStages + 1); e <= armed; ++e)
                    landed = mbar_wait(&full[e % kStages], (uint32_t)(e / kStages) & 1u, kLandBudget) && landed;
                if (!__all_sync(0xffffffffu, landed) && lane == 0) ctl.unlanded = 1;
            }
        } else {
            // ------------------------------------------------------------------ MMA issuer
            // Order: S(0), S(1), then per tile j: PV(j) once P(j) is in TMEM, then S(j+2) into
            // the buffer P(j)'s scores came from.  MMAs of one thread run in issue order, so the
            // completion of S(j+2) implies that of PV(j): the softmax of tile j+2 may then
            // overwrite P buffer j % 2.
            if (warp == kMmaWarp && lane == 0) {
                const uint32_t idS = idesc_bf16(kBM, kBN, false, false);
                const uint32_t idO = idesc_bf16(kBM, kD, false, true);
                const uint64_t dq = sdesc_sw128(sQ, 16, 1024);
                auto issue_s = [&](int j) {
                    const uint64_t dk = sdesc_sw128(sK(j % kStages), 16, 1024);
                    const uint32_t d_s = tmem + kColS0 + (uint32_t)(j & 1) * 128u;
    #pragma unroll
                    for (int k = 0; k < kD / 16; ++k) {
                        const uint64_t ko = ((uint64_t)(k >> 2) * kRegion + (uint64_t)(k & 3) * 32u) >> 4;
                        umma_ss(d_s, dq + ko, dk + ko, idS, k > 0);
                    }
                    umma_commit(&ctl.s_full[j & 1]);
                    umma_commit(&ctl.k_empty[j % kStages]);
                };
                ok = wait_bar(&ctl.q_full, 0, abort_flag, dev_status, budget);
                for (int j = 0; ok && j < 2 && j < n_kv; ++j) {
                    ok = wait_bar(&ctl.k_full[j], 0, abort_flag, dev_status, budget);
                    if (!ok) break;
                    tc_fence_after();
                    issue_s(j);
                }
                for (int j = 0; ok && j < n_kv; ++j) {
                    ok = wait_bar(&ctl.v_full[j % kStages], (j / kStages) & 1, abort_flag, dev_status, budget) &&
                         wait_bar(&ctl.p_full[j & 1], (j >> 1) & 1, abort_flag, dev_status, budget);
                    if (!ok) break;
                    tc_fence_after();
                    const uint64_t dv = sdesc_sw128(sV(j % kStages), kRegion, 1024);
                    const uint32_t a_p = tmem + kColP0 + (uint32_t)(j & 1) * 64u;
    #pragma unroll
                    for (int k = 0; k < kBN / 16; ++k)
                        umma_ts(tmem + kColO, a_p + k * 8, dv + (uint64_t)(k * 2048 / 16), idO, (j > 0 || k > 0));
                    umma_commit(&ctl.v_empty[j % kStages]);
                    umma_commit(&ctl.pv_done);
                    if (j + 2 < n_kv) {
                        ok = wait_bar(&ctl.k_full[(j + 2) % kStages], ((j + 2) / kStages) & 1, abort_flag, dev_status, budget);
                        if (!ok) break;
                        tc_fence_after();
                        issue_s(j + 2);
                    }
                }
                umma_commit(&ctl.drain);
                mbar_wait(&ctl.drain, 0, kDrainBudget);
            }
            __syncwarp();
        }
    } else {
        setmaxnreg_inc<kRegSoftmax>();
        // ------------------------------------------------------------------ softmax
        constexpr int NC = 4 / REP;                   // 32-key chunks of this warp's key group
        const int wr = warp / (4 / REP);              // replica = key group of this warp
        const int kb = wr * (kBN / REP);              // first key of the group inside a tile
        const int r = threadIdx.x;                    // TMEM lane
        const uint32_t lane_base = tmem + ((uint32_t)(warp * 32) << 16);
        const float c = p.scale_log2;
        {   // P buffers start as zeros: columns outside this warp's key group are never written
            uint32_t z[32];
#pragma unroll
            for (int i = 0; i < 32; ++i) z[i] = 0u;
#pragma unroll
            for (int cc = 0; cc < 4; ++cc) tmem_st32(lane_base + kColP0 + cc * 32, z);
            tmem_st_wait();
        }
        float m_used = -INFINITY, l_sum = 0.f;
        for (int j = 0; j < n_kv; ++j) {
            const int sb = j & 1;
            // discarded keys of this warp's key group: bit i of drop[cc] = key kb + 32 cc + i
            uint32_t drop[NC];
#pragma unroll
            for (int cc = 0; cc < NC; ++cc) drop[cc] = 0u;
            if constexpr (kDrop) {
                const int32_t* rs = p.read_slot + (int64_t)b * p.T_len;
#pragma unroll
                for (int cc = 0; cc < NC; ++cc) {
                    const int tk = (kt0 + j) * kBN + kb + cc * 32 + lane;
                    drop[cc] = __ballot_sync(0xffffffffu, tk < p.T_len && rs[tk] == ACACHE_SLOT_NONE);
                }
            }
            ok = __all_sync(0xffffffffu, wait_bar(&ctl.s_full[sb], (j >> 1) & 1, abort_flag, dev_status, budget));
            if (!ok) break;
            tc_fence_after();
            uint32_t v[NC][32];
#pragma unroll
            for (int cc = 0; cc < NC; ++cc) tmem_ld32(lane_base + kColS0 + sb * 128 + kb + cc * 32, v[cc]);
            tmem_ld_wait();
            const int valid = min(kBN, p.T_len - (kt0 + j) * kBN) - kb;   // keys of the group in range
            if (valid < kBN / REP) {
#pragma unroll
                for (int cc = 0; cc < NC; ++cc)
#pragma unroll
                    for (int i = 0; i < 32; ++i)
                        if (cc * 32 + i >= valid) v[cc][i] = __float_as_uint(-INFINITY);
            }
            if constexpr (kDrop) {
#pragma unroll
                for (int cc = 0; cc < NC; ++cc)
                    if (drop[cc]) {
#pragma unroll
                        for (int i = 0; i < 32; ++i)
                            if ((drop[cc] >> i) & 1u) v[cc][i] = __float_as_uint(-INFINITY);
                    }
            }
            float mx[NC];
#pragma unroll
            for (int cc = 0; cc < NC; ++cc) {
                mx[cc] = max3f(__uint_as_float(v[cc][0]), __uint_as_float(v[cc][1]), __uint_as_float(v[cc][2]));
#pragma unroll
                for (int i = 3; i < 31; i += 2)
                    mx[cc] = max3f(mx[cc], __uint_as_float(v[cc][i]), __uint_as_float(v[cc][i + 1]));
                mx[cc] = fmaxf(mx[cc], __uint_as_float(v[cc][31]));
            }
            float mt = mx[0];
#pragma unroll
            for (int cc = 1; cc < NC; ++cc) mt = fmaxf(mt, mx[cc]);
            mt *= c;
            float alpha = 1.f;
            bool resc = false;
            if (j == 0) {
                m_used = mt;
            } else if (mt > m_used + kRescaleThreshold) {
                alpha = fast_exp2(m_used - mt);   // 0 while no key of the group was valid
                m_used = mt;
                resc = true;
            }
            if (__any_sync(0xffffffffu, resc)) {
                // O holds tiles 0..j-1 once PV(j-1) has completed
                ok = __all_sync(0xffffffffu, wait_bar(&ctl.pv_done, (j - 1) & 1, abort_flag, dev_status, budget));
                if (!ok) break;
                tc_fence_after();
#pragma unroll
                for (int cc = 0; cc < 4; ++cc) {
                    uint32_t o[32];
                    tmem_ld32(lane_base + kColO + cc * 32, o);
                    tmem_ld_wait();
#pragma unroll
                    for (int i = 0; i < 32; ++i) o[i] = __float_as_uint(__uint_as_float(o[i]) * alpha);
                    tmem_st32(lane_base + kColO + cc * 32, o);
                }
            }
            // a group with no valid key so far exponentiates against 0 (every value is -inf)
            const float ms = m_used == -INFINITY ? 0.f : m_used;
            const uint64_t c2 = f2pack(c, c), nm2 = f2pack(-ms, -ms);
            uint64_t ls2[2] = {f2pack(0.f, 0.f), f2pack(0.f, 0.f)};
#pragma unroll
            for (int cc = 0; cc < NC; ++cc) {
                uint32_t pk[16];
#pragma unroll
                for (int i = 0; i < 32; i += 2) {
                    float x0, x1;
                    f2unpack(f2fma(f2pack(__uint_as_float(v[cc][i]), __uint_as_float(v[cc][i + 1])), c2, nm2), x0, x1);
                    const float p0 = fast_exp2(x0), p1 = fast_exp2(x1);
                    ls2[(i >> 1) & 1] = f2add(ls2[(i >> 1) & 1], f2pack(p0, p1));
                    __nv_bfloat162 two = __floats2bfloat162_rn(p0, p1);
                    pk[i >> 1] = *reinterpret_cast<uint32_t*>(&two);
                }
                tmem_st16(lane_base + kColP0 + sb * 64 + kb / 2 + cc * 16, pk);
            }
            float l0, l1, l2, l3;
            f2unpack(ls2[0], l0, l1);
            f2unpack(ls2[1], l2, l3);
            l_sum = l_sum * alpha + ((l0 + l1) + (l2 + l3));
            tmem_st_wait();
            tc_fence_before();
            mbar_arrive(&ctl.p_full[sb]);
        }
        if (ok) ok = __all_sync(0xffffffffu, wait_bar(&ctl.drain, 0, abort_flag, dev_status, budget));
        if (ok) {
            tc_fence_after();
            if (REP == 1 && cs == 1) {
                // one partial per row: normalise and write straight from TMEM (the TMEM load is
                // warp-collective; lanes past the block's rows only skip the store)
                const bool live = r < rows_valid;
                const int i = q0 + r / p.g, hh = hk * p.g + r % p.g;
                bf16* orow = p.out + (((int64_t)b * p.n_q + (live ? i : 0)) * p.Hq + hh) * kD;
                const float inv_l = l_sum > 0.f ? 1.f / l_sum : 0.f;
#pragma unroll
                for (int cc = 0; cc < 4; ++cc) {
                    uint32_t o[32];
                    tmem_ld32(lane_base + kColO + cc * 32, o);
                    tmem_ld_wait();
                    uint32_t pkd[16];
#pragma unroll
                    for (int x = 0; x < 16; ++x) {
                        __nv_bfloat162 two = __floats2bfloat162_rn(__uint_as_float(o[2 * x]) * inv_l,
                                                                   __uint_as_float(o[2 * x + 1]) * inv_l);
                        pkd[x] = *reinterpret_cast<uint32_t*>(&two);
                    }
                    if (live) {
                        uint4* dst = reinterpret_cast<uint4*>(orow + cc * 32);
#pragma unroll
                        for (int x = 0; x < 4; ++x)
                            dst[x] = make_uint4(pkd[4 * x], pkd[4 * x + 1], pkd[4 * x + 2], pkd[4 * x + 3]);
                    }
                }
            } else {
                // partial of this lane (replica wr, row r % G) into the free K ring
                uint8_t* part = base_ptr + kTileBytes;
#pragma unroll
                for (int cc = 0; cc < 4; ++cc) {
                    uint32_t o[32];
                    tmem_ld32(lane_base + kColO + cc * 32, o);
                    tmem_ld_wait();
#pragma unroll
                    for (int x = 0; x < 8; ++x)
                        *reinterpret_cast<uint4*>(part + part_off(r, cc * 8 + x)) =
                            make_uint4(o[4 * x], o[4 * x + 1], o[4 * x + 2], o[4 * x + 3]);
                }
                ctl.part_m[r] = m_used;
                ctl.part_l[r] = l_sum;
            }
        }
    }
    tc_fence_before();
    __syncthreads();
    tc_fence_after();
    if (*abort_flag) settle_after_abort(ctl.unlanded != 0);
    if (warp == kMmaWarp) tmem_dealloc(tmem, kTmemCols);
    if (REP == 1 && cs == 1) return;

    // ---------------------------------------------------------------------- combine
    // Row r of the block has REP x cs partials: replica w of cluster rank q sits at lane
    // w*G + r of CTA q.  CTA q finalises the (row, 32-column chunk) items it = q (mod cs).
    if (cs > 1) cluster_sync(); else __syncthreads();
    if (wg == 0 && !*abort_flag) {
        const uint32_t part_base = base + kTileBytes;
        const uint32_t m_base = smem_u32(&ctl.part_m[0]), l_base = smem_u32(&ctl.part_l[0]);
        for (int it = cr + cs * (int)threadIdx.x; it < rows_valid * 4; it += cs * 128) {
            const int r = it >> 2, c4 = it & 3;
            auto part_max = [&](int q, int lr) {
                return cs > 1 ? ld_cluster_f32(mapa_shared(m_base + (uint32_t)lr * 4u, (uint32_t)q))
                              : ctl.part_m[lr];
            };
            float M = -INFINITY;
            for (int q = 0; q < cs; ++q)
#pragma unroll
                for (int w = 0; w < REP; ++w) M = fmaxf(M, part_max(q, w * G + r));
            float acc[32];
#pragma unroll
            for (int x = 0; x < 32; ++x) acc[x] = 0.f;
            float lsum = 0.f;
            for (int q = 0; q < cs; ++q)
#pragma unroll
                for (int w = 0; w < REP; ++w) {
                    const int lr = w * G + r;
                    const float mv = part_max(q, lr);
                    if (mv == -INFINITY) continue;   // no valid key in this partial
                    const float e = fast_exp2(mv - M);
                    const uint32_t la = l_base + (uint32_t)lr * 4u;
                    lsum += e * (cs > 1 ? ld_cluster_f32(mapa_shared(la, (uint32_t)q)) : ctl.part_l[lr]);
#pragma unroll
                    for (int x = 0; x < 8; ++x) {
                        const uint32_t a = part_base + part_off(lr, c4 * 8 + x);
                        float4 f;
                        if (cs > 1) f = ld_cluster_v4(mapa_shared(a, (uint32_t)q));
                        else f = *reinterpret_cast<const float4*>(base_ptr + (a - base));
                        acc[4 * x] += e * f.x;
                        acc[4 * x + 1] += e * f.y;
                        acc[4 * x + 2] += e * f.z;
                        acc[4 * x + 3] += e * f.w;
                    }
                }
            const float inv_l = lsum > 0.f ? 1.f / lsum : 0.f;
            const int i = q0 + r / p.g, hh = hk * p.g + r % p.g;
            bf16* orow = p.out + (((int64_t)b * p.n_q + i) * p.Hq + hh) * kD + c4 * 32;
            uint32_t pkd[16];
#pragma unroll
            for (int x = 0; x < 16; ++x) {
                __nv_bfloat162 two = __floats2bfloat162_rn(acc[2 * x] * inv_l, acc[2 * x + 1] * inv_l);
                pkd[x] = *reinterpret_cast<uint32_t*>(&two);
            }
            uint4* dst = reinterpret_cast<uint4*>(orow);
#pragma unroll
            for (int x = 0; x < 4; ++x) dst[x] = make_uint4(pkd[4 * x], pkd[4 * x + 1], pkd[4 * x + 2], pkd[4 * x + 3]);
        }
    }
    // no CTA may leave while another still reads its shared memory
    if (cs > 1) cluster_sync();
}

// Host-side geometry of one decode launch.
struct DecodeGeom {
    int rep, qpb, n_rb, cs;
};

// Replication, row blocks and cluster size for n_q queries of g heads per KV head.
bool decode_geom(int B, int n_q, int g, int hkv, int T_len, DecodeGeom& dg) {
    const int64_t rg = (int64_t)n_q * g;
    dg.rep = rg <= 32 ? 4 : rg <= 64 ? 2 : 1;
    const int G = kBM / dg.rep;
    if (g > G) return false;
    dg.qpb = std::min(n_q, G / g);
    dg.n_rb = (n_q + dg.qpb - 1) / dg.qpb;
    // cluster size: fill the SMs -- estimated time = waves x (tiles per CTA + fixed cost of
    // about two tiles for the prologue, the last tiles' latency and the combine)
    const int64_t units = (int64_t)B * hkv * dg.n_rb;
    const int n_all = (T_len + kBN - 1) / kBN;
    const int64_t nsm = sm_count();
    dg.cs = 1;
    double best = 0;
    for (int cs = 1; cs <= kMaxCluster && cs <= n_all; cs *= 2) {
        const int64_t waves = (units * cs + nsm - 1) / nsm;
        const double est = (double)waves * ((double)((n_all + cs - 1) / cs) + 2.0);
        if (cs == 1 || est < best) {
            best = est;
            dg.cs = cs;
        }
    }
    return true;
}

// Per device and kernel variant: 0 = not prepared yet, 1 = ready, otherwise the status to
// return.  Preparing twice is harmless, so a race between threads only repeats the work.
std::atomic<int> g_prepared[6][64];

template <int REP, bool kDrop>
int prepare(int dev) {
    std::atomic<int>& st = g_prepared[(REP == 4 ? 2 : REP - 1) * 2 + (kDrop ? 1 : 0)][dev];
    const int known = st.load(std::memory_order_acquire);
    if (known) return known == 1 ? ACACHE_OK : known;
    auto kern = tc_decode_kernel<REP, kDrop>;
    int rc = ACACHE_OK;
    cudaFuncAttributes fa;
    if (cudaFuncSetAttribute(kern, cudaFuncAttributeMaxDynamicSharedMemorySize, kSmemBytes) != cudaSuccess ||
        cudaFuncGetAttributes(&fa, kern) != cudaSuccess) {
        (void)cudaGetLastError();
        return ACACHE_ERR_CUDA;   // not cached: a later call may succeed
    }
    // the register split above assumes the launch allocation; refuse to launch otherwise
    if (fa.numRegs < kLaunchRegs) rc = ACACHE_ERR_UNSUPPORTED;
    st.store(rc == ACACHE_OK ? 1 : rc, std::memory_order_release);
    return rc;
}

template <int REP, bool kDrop>
int launch_rep(const DecParams& prm, int64_t ctas, cudaStream_t stream, bool pdl) {
    auto kern = tc_decode_kernel<REP, kDrop>;
    int dev = 0;
    if (cudaGetDevice(&dev) != cudaSuccess || dev < 0 || dev >= 64) {
        (void)cudaGetLastError();
        return ACACHE_ERR_CUDA;
    }
    if (int rc = prepare<REP, kDrop>(dev)) return rc;
    cudaLaunchConfig_t cfg = {};
    cfg.gridDim = dim3((unsigned)ctas);
    cfg.blockDim = dim3(kThreads);
    cfg.dynamicSmemBytes = kSmemBytes;
    cfg.stream = stream;
    cudaLaunchAttribute attr[2];
    unsigned na = 0;
    if (prm.cs > 1) {
        attr[na].id = cudaLaunchAttributeClusterDimension;
        attr[na].val.clusterDim.x = (unsigned)prm.cs;
        attr[na].val.clusterDim.y = 1;
        attr[na].val.clusterDim.z = 1;
        ++na;
    }
    if (pdl) {
        attr[na].id = cudaLaunchAttributeProgrammaticStreamSerialization;
        attr[na].val.programmaticStreamSerializationAllowed = 1;
        ++na;
    }
    cfg.attrs = attr;
    cfg.numAttrs = na;
    if (cudaLaunchKernelEx(&cfg, kern, prm) != cudaSuccess) {
        (void)cudaGetLastError();
        return ACACHE_ERR_CUDA;
    }
    return launch_status();
}

}  // namespace

bool tc_decode_preferred(const AttnArgs& a, int B, int n_q, int T_len) {
    if (a.hkv <= 0 || a.hq % a.hkv) return false;
    const int g = a.hq / a.hkv;
    const int64_t rg = (int64_t)n_q * g;
    const int rep = rg <= 32 ? 4 : rg <= 64 ? 2 : 1;
    const int G = kBM / rep;
    if (n_q <= 0 || g > G) return false;
    const int64_t qpb = std::min(n_q, G / g);
    const int64_t streams_dec = (n_q + qpb - 1) / qpb;            // K/V streams per KV head
    const int64_t streams_main = (int64_t)g * ((n_q + 255) / 256);
    if (streams_dec != streams_main) return streams_dec < streams_main;
    // As many K/V streams either way (one query head per KV head): the recompute kernel's
    // lone-tile CTA, whose two chains split the keys, runs a stream slightly faster (measured
    // at 32 queries: 23.4 against 24.9 us with 4 requests, 249 against 267 us with 16); the
    // block-decode kernel still wins when the streams would leave most SMs idle and its
    // cluster split of the keys fills them (a request or two).
    (void)T_len;
    return n_q <= 128 && (int64_t)B * a.hkv * streams_dec * 2 <= (int64_t)sm_count();
}

int launch_tc_decode_attention(const AttnArgs& a, int B, int n_q, const void* q, int T_len,
                               const int32_t* read_slot, const void* k_cache, const void* v_cache,
                               int64_t num_slots, void* out, int32_t* dev_status, cudaStream_t stream,
                               bool drop_none, bool pdl) {
    if ((int64_t)num_slots * a.hkv >= 0x7fffffffLL || (int64_t)B * n_q >= 0x7fffffffLL)
        return ACACHE_ERR_INVALID_ARG;
    const int g = a.hq / a.hkv;
    DecodeGeom dg;
    if (!decode_geom(B, n_q, g, a.hkv, T_len, dg)) return ACACHE_ERR_UNSUPPORTED;
    const int64_t ctas = (int64_t)B * a.hkv * dg.n_rb * dg.cs;
    if (ctas == 0) return ACACHE_OK;
    if (ctas > 0x7fffffff) return ACACHE_ERR_INVALID_ARG;
    DecParams prm{};
    const uint64_t dq[4] = {(uint64_t)kD, (uint64_t)a.hq, (uint64_t)n_q, (uint64_t)B};
    const uint32_t bq[4] = {64u, (uint32_t)g, (uint32_t)dg.qpb, 1u};
    const uint64_t dp[2] = {(uint64_t)kD, (uint64_t)num_slots * a.hkv};
    if (!make_map_box(&prm.tm_q, q, 4, dq, bq) || !make_map(&prm.tm_k, k_cache, 2, dp, 1, 1) ||
        !make_map(&prm.tm_v, v_cache, 2, dp, 1, 1))
        return ACACHE_ERR_CUDA;
    prm.read_slot = read_slot;
    prm.out = (bf16*)out;
    prm.dev_status = dev_status;
    prm.num_slots = num_slots;
    prm.n_q = n_q;
    prm.Hq = a.hq;
    prm.Hkv = a.hkv;
    prm.g = g;
    prm.T_len = T_len;
    prm.qpb = dg.qpb;
    prm.n_rb = dg.n_rb;
    prm.cs = dg.cs;
    prm.scale_log2 = a.scale * kLog2e;
    prm.budget = wait_budget();
    if (drop_none) {
        switch (dg.rep) {
            case 4: return launch_rep<4, true>(prm, ctas, stream, pdl);
            case 2: return launch_rep<2, true>(prm, ctas, stream, pdl);
            default: return launch_rep<1, true>(prm, ctas, stream, pdl);
        }
    }
    switch (dg.rep) {
        case 4: return launch_rep<4, false>(prm, ctas, stream, pdl);
        case 2: return launch_rep<2, false>(prm, ctas, stream, pdl);
        default: return launch_rep<1, false>(prm, ctas, stream, pdl);
    }
}

}  // namespace acache
