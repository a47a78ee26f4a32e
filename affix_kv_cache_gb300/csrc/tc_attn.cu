// tc_attn.cu -- tensor-core (tcgen05 + TMEM, TMA-fed) attention kernels for bf16, head_dim 128.
//
// Page: "Affix Cache for Diffusion Large Language Models" -- Sec. 3.2 (the one-shot probe,
// Eq. 4-5) and Sec. 4.3 / App. C.1 (attention that reads every logical key through the
// per-request read-slot map).  The page's prototype is a Triton kernel on A100; this is a
// GB300-first design:
//
// tc_attn_kernel  (probe forward and read-slot attention at a recompute point; one CTA per
//                  256 query rows -- two 128-row Q tiles A and B -- of one (request, query
//                  head); 640 threads in five warpgroups, 1 CTA per SM)
//   WG0, WG1  softmax + epilogue of tile A / B: thread r owns query row r (= TMEM lane r).
//             Per key tile j: read S_t(j) from TMEM, row maximum, exponentiate in base 2
//             against a lazily raised maximum (it only moves when it grows by more than 2^8;
//             then O_t and the row sum are rescaled in TMEM), write P_t(j) as packed bf16 over
//             S_t(j)'s first 64 columns, keys 0-63 published before keys 64-127.  The two
//             warpgroups take turns (A(0), B(0), A(1), ...) so each has the SM's issue slots
//             to itself while the tensor core works on the other tile.
//   WG2       warp 8 allocates TMEM (S_A, S_B, O_A, O_B: 128 fp32 columns each); lane 0 of
//             warp 8 issues tile A's MMAs, lane 0 of warp 9 tile B's:
//             S_t(j) = Q_t K_j^T (SS, M = N = 128) and O_t += P_t(j) V_j (TS: P from TMEM,
//             V an MN-major shared-memory operand), S_t(j+1) right after PV_t(j).  Warps 10
//             and 11 are TMA producers.
//   WG3, WG4  TMA producers: warps 10-14 fill a 3-stage K ring, warps 15-19 a 2-stage V
//             ring.  Read-slot keys: a tile whose 128 slots are consecutive (a request's own
//             rows, a page of the shared region) is two tiled box loads of the pool; any other
//             is 64 `tile::gather4` loads (4 pool rows x 64 columns, rows resolved through the
//             read-slot map one tile ahead), 12-13 per warp -- each gather4 a lane issues costs
//             its warp tens of cycles, so the gather rate grows with the number of issuing
//             warps.  Probe keys: the affix rows and the request's own rows are contiguous per
//             KV head, so a tile is two tiled box loads.  Loads complete on the stage's
//             mbarrier by byte count.
//   setmaxnreg gives the softmax warpgroups 168 registers and WG2-WG4 48.
//   A CTA left with one Q tile (the ragged last query block) splits its keys instead: chain A
//   takes the first half of the key tiles and chain B the second half, both against the same
//   Q tile, so the two chains still ping-pong; the K/V rings then alternate A's and B's tiles,
//   the free Q buffer becomes a third V stage, and at the end chain B hands its row maximum
//   and row sum to chain A through shared memory, which merges the two partial softmax states
//   (O_A 2^(m_A-m) + O_B 2^(m_B-m), likewise the sums) before the epilogue.
//
// tc_colsum_kernel  (second probe pass: masked-to-affix attention mass; one CTA per
//                    (request, query head, 128 affix keys))
//   D = K_affix_tile Q_masked_chunk^T (SS MMA, M = 128 affix keys, N = 128 masked rows);
//   a chunk of masked query rows that are consecutive probe rows (the usual case: the
//   generation positions) is two tiled box loads, other chunks are gathered with
//   `tile::gather4`; thread r owns affix key r and sums 2^(logit - m_k) / l_k over the masked
//   rows k into four partial sums in a fixed order -- a per-thread sum, so the result is
//   deterministic and no cross-thread reduction is needed.
// tc_colsum_rows_kernel  (the same pass when the masked rows fit in two 128-row chunks; one
//                         CTA per (request, query head, run of affix tiles))
//   the masked rows stay in shared memory while the run's affix key tiles stream through
//   four stages and D alternates between two TMEM buffers; one consumer warpgroup per chunk.
//
// Every mbarrier wait is bounded (by default about a second; acache_wait_budget sets it); a
// wait that gives up raises a CTA-wide abort flag and ACACHE_DEV_TIMEOUT, every role leaves its
// loop, in-flight MMAs are drained with a bounded wait, the attention kernel's TMA loads issued
// before the abort are waited for (bounded; a fixed ~30 us hold where their barrier phase cannot
// complete, and in the other kernels), and TMEM is freed before the CTA exits.
#include <cuda.h>
#include <cudaTypedefs.h>

#include <algorithm>

#include "tc_attn.cuh"
#include "ptx.cuh"

namespace acache {
namespace {

using namespace ptx;
using bf16 = __nv_bfloat16;

constexpr int kD = 128;                     // head dim
constexpr int kBM = 128;                    // query rows per Q tile (one softmax warpgroup)
constexpr int kQT = 2;                      // Q tiles per CTA: 256 query rows share each K/V tile
constexpr int kBN = 128;                    // keys per tile
constexpr int kKStages = 3;                 // K ring: a K tile is free once S_B has read it
constexpr int kVStages = 2;                 // V ring: a V tile is free once PV_B has read it
constexpr int kMmaWarp = 8;                 // warpgroup 2: TMEM allocation; warps 8 and 9 each
                                            // issue the MMAs of one Q tile
constexpr int kProdWarp = 10;               // first TMA producer warp
constexpr int kProdPerRing = 5;             // producer warps per ring: K warps 10-14, V 15-19
constexpr int kThreads = (kProdWarp + 2 * kProdPerRing) * 32;
static_assert(kThreads % 128 == 0, "whole warpgroups");
// Registers: 640 threads x 96 at launch = 61440; the softmax warpgroups grow to 168, the MMA /
// producer warpgroups shrink to 48: 2*128*168 + 3*128*48 = 61440 (no spills).
constexpr int kRegLaunch = 65536 / kThreads / 8 * 8;
constexpr int kRegSoftmax = 168, kRegOther = 48;
static_assert(2 * 128 * kRegSoftmax + (kThreads - 256) * kRegOther <= kThreads * kRegLaunch, "register split");
constexpr uint32_t kTileBytes = kBN * kD * 2;     // 32 KB: one 128 x 128 bf16 tile
constexpr uint32_t kRegion = kBN * 128;           // 16 KB: 64 columns of a 128-row tile
constexpr uint32_t kSmemBytes = kTileBytes * (kQT + kKStages + kVStages) + 1024;
constexpr uint32_t kTmemCols = 512;               // S_A, S_B, O_A, O_B: 128 fp32 columns each
__host__ __device__ constexpr uint32_t col_s(int t) { return (uint32_t)t * 128u; }
__host__ __device__ constexpr uint32_t col_o(int t) { return 256u + (uint32_t)t * 128u; }
constexpr float kRescaleThreshold = 8.0f;         // log2 units: P values stay below 2^8
// Waits of the abort path itself (in-flight MMAs, TMA loads already issued) use fixed budgets,
// whatever budget the pipeline's waits were launched with.
constexpr long long kDrainBudget = 1LL << 31;     // cycles (~1 s): MMAs issued before an abort
constexpr long long kLandBudget = 1LL << 21;      // cycles (~1 ms): TMA loads issued before it

enum KeyMode { kSlotKeys = 0, kProbeKeys = 1 };

// n / d for 0 <= n < 2^31 and 1 <= d < 2^31 as one 64-bit multiply and a shift: with
// l = ceil(log2 d), s = 32 + l and m = ceil(2^s / d), the excess e = m d - 2^s is below d <= 2^l,
// so n e < 2^s and floor(n m / 2^s) = floor(n / d); n m < 2^64.
struct FastDiv {
    uint64_t m;
    uint32_t s;
    __host__ __device__ uint32_t operator()(uint32_t n) const { return (uint32_t)(((uint64_t)n * m) >> s); }
};
inline FastDiv make_fastdiv(uint32_t d) {
    uint32_t l = 0;
    while ((1ull << l) < d) ++l;
    const uint32_t s = 32 + l;
    return FastDiv{((1ull << s) + d - 1) / d, s};
}

struct AttnParams {
    CUtensorMap tm_q;     // 4-D [B][n_rows][Hq][d], box {64, 1, 128, 1}
    CUtensorMap tm_k0;    // slot: 2-D pool [num_slots*Hkv][d], box {64, 1} (gather4)
    CUtensorMap tm_v0;    // probe: 3-D affix [L][Hkv][d], box {64, 1, 128}
    CUtensorMap tm_k1;    // slot: 3-D pool [num_slots][Hkv][d], box {64, 1, 128} (consecutive slots)
    CUtensorMap tm_v1;    // probe: 4-D own rows [B][P][Hkv][d], box {64, 1, 128, 1}
    CUtensorMap tm_o;     // output, laid out as tm_q (valid when out is not null)
    const int32_t* read_slot;
    const int32_t* q_start;   // ragged batches (slot keys): [B+1] query-row offsets, or null
    const int32_t* kv_start;  //                              [B+1] logical-key offsets
    bf16* out;
    float* stat_m;
    float* stat_l;
    int32_t* dev_status;
    int64_t num_slots;
    // when the grid waits for the grid it follows on the stream (programmatic dependent launch):
    // 1 before any K/V load (the pool may have been written by it: store-then-attend), 0 only
    // before its CTAs exit (a chained layer: it reads nothing its predecessor writes), 2 before
    // its first global write (the probe forward of the next layer: it writes the scratch the
    // preceding grids of the probe read)
    int early_wait;
    int n_rows, Hq, Hkv, T_len, L, P;
    int g;                // Hq / Hkv
    int B;                // requests (persistent launch)
    int n_kv, n_units;    // persistent launch: key tiles (< 2^15), units (< 2^22)
    FastDiv div_bhq, div_hq, div_g;   // persistent launch: / (B Hq), / Hq, / (Hq / Hkv)
    float scale_log2;
    long long budget;     // cycles a pipeline wait may take before it gives up
};

struct AttnCtl {
    uint64_t q_full;
    uint64_t k_full[kKStages];
    uint64_t k_empty[kKStages];
    uint64_t v_full[kVStages + 1];    // + the stage in the free Q buffer (split keys)
    uint64_t v_empty[kVStages + 1];
    uint64_t s_full[kQT];
    uint64_t p_half[kQT];   // first half of P_t(j) (keys 0-63) is in TMEM
    uint64_t p_full[kQT];   // all of P_t(j) is in TMEM
    uint64_t drain[kQT];
    uint64_t turn[kQT];     // softmax ping-pong: turn[t] completes when tile t may exponentiate
    uint32_t tmem_base;
    int abort;
    int unlanded;           // abort path: some TMA load issued before the abort may not have landed
    int split_ok;           // split keys: chain B's partial state below is complete
    float split_m[kBM];     //   chain B's row maximum (the exponent offset it used) and row sum
    float split_l[kBM];
};

// Stage and lap of ring entry e in a ring of n = 2 or 3 stages (divisions by constants).
static_assert(kKStages == 3 && kVStages == 2, "ring sizes 2 and 3 (a third V stage with split keys)");
ACACHE_DEVFN int ring_lap(int e, int n) { return n == 2 ? (e >> 1) : e / 3; }
ACACHE_DEVFN int ring_stage(int e, int n) { return e - ring_lap(e, n) * n; }

// Key-tile schedule of a CTA.  Ring entry e is the e-th K/V tile the producers load; chain t
// reads its i-th key tile from entry entry(t, i).  Unsplit: every chain reads every key tile
// and entry e holds tile e.  Split (one Q tile): chain 0 reads tiles [0, n0), chain 1 tiles
// [n0, n_kv); entries alternate chain 0, chain 1, ..., and the last tile of chain 0 (odd
// n_kv) is the last entry.
struct KeySchedule {
    bool split;
    int n_kv, n0;
    ACACHE_DEVFN int n_tiles(int t) const { return split ? (t == 0 ? n0 : n_kv - n0) : n_kv; }
    ACACHE_DEVFN int tile(int t, int i) const { return (split && t == 1) ? n0 + i : i; }
    ACACHE_DEVFN int entry(int t, int i) const {
        if (!split) return i;
        const int n1 = n_kv - n0;
        return i < n1 ? 2 * i + t : n1 + i;
    }
    ACACHE_DEVFN int entry_tile(int e) const {
        if (!split) return e;
        const int n1 = n_kv - n0;
        if (e < 2 * n1) return (e & 1) ? n0 + (e >> 1) : (e >> 1);
        return e - n1;
    }
};

// Bounded wait that also leaves early once another role has aborted: after `budget` cycles it
// raises the CTA's abort flag and ACACHE_DEV_TIMEOUT.
ACACHE_DEVFN bool wait_bar(uint64_t* bar, uint32_t parity, volatile int* abort_flag,
                           int32_t* dev_status, long long budget) {
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

// Number of key tiles and the valid keys of tile j (identical on every role).  Probe tiles
// cover the affix rows first, then the request's own rows: the order of keys inside a row
// does not change the softmax.
template <int kMode>
ACACHE_DEVFN int n_key_tiles(const AttnParams& p, int T_len) {
    if (kMode == kSlotKeys) return (T_len + kBN - 1) / kBN;
    return (p.L + kBN - 1) / kBN + (p.P + kBN - 1) / kBN;
}
template <int kMode>
ACACHE_DEVFN int tile_valid(const AttnParams& p, int j, int T_len) {
    if (kMode == kSlotKeys) return min(kBN, T_len - j * kBN);
    const int n_aff = (p.L + kBN - 1) / kBN;
    return j < n_aff ? min(kBN, p.L - j * kBN) : min(kBN, p.P - (j - n_aff) * kBN);
}

// Read-slot entries of keys 4 lane .. 4 lane + 3 of key tile j: -1 where there is no key or
// the slot lies outside the pool (flagged by `flagger` unless it marks a discarded key).
// In two steps: the loads (bit u of `keys` set where key u exists), and the checks.  Issued
// apart, the loads' latency passes while the warp does other work.
ACACHE_DEVFN uint32_t tile_slots_load(const AttnParams& p, int64_t kbase, int T_len, int n_kv, int j, int lane,
                                      int (&raw)[4]) {
    uint32_t keys = 0;
#pragma unroll
    for (int u = 0; u < 4; ++u) {
        const int tk = j * kBN + 4 * lane + u;
        const bool key = j < n_kv && tk < T_len;
        raw[u] = key ? __ldg(p.read_slot + kbase + tk) : -1;
        keys |= (uint32_t)key << u;
    }
    return keys;
}
template <bool kDrop>
ACACHE_DEVFN void tile_slots_check(const AttnParams& p, bool flagger, uint32_t keys, const int (&raw)[4],
                                   int (&sl)[4]) {
#pragma unroll
    for (int u = 0; u < 4; ++u) {
        const int slot = raw[u];
        sl[u] = -1;
        if (!((keys >> u) & 1u)) continue;
        if (slot >= 0 && slot < p.num_slots)
            sl[u] = slot;
        else if (flagger && !(kDrop && slot == ACACHE_SLOT_NONE))
            flag(p.dev_status, ACACHE_DEV_BAD_SLOT);
    }
}
template <bool kDrop>
ACACHE_DEVFN void tile_slots(const AttnParams& p, int64_t kbase, int T_len, int n_kv, int j, int lane,
                             bool flagger, int (&sl)[4]) {
    int raw[4];
    const uint32_t keys = tile_slots_load(p, kbase, T_len, n_kv, j, lane, raw);
    tile_slots_check<kDrop>(p, flagger, keys, raw, sl);
}

// kDrop (read-slot keys only): a read-slot entry equal to ACACHE_SLOT_NONE marks a logical
// position whose K/V was discarded (the page's DropNA ablation, Sec. 5.3): the key takes
// no part in the softmax, and a row with no key left outputs zeros.
template <int kMode, bool kDrop>
__global__ void __launch_bounds__(kThreads, 1)
tc_attn_kernel(const __grid_constant__ AttnParams p) {
    extern __shared__ uint8_t dsm[];
    __shared__ AttnCtl ctl;
    const uint32_t base = (smem_u32(dsm) + 1023u) & ~1023u;
    // shared memory: Q_A, Q_B, the K ring, the V ring (32 KB tiles, 1024-byte aligned)
    auto sQ = [&](int t) { return base + kTileBytes * (uint32_t)t; };
    auto sK = [&](int s) { return base + kTileBytes * (uint32_t)(kQT + s); };
    auto sV = [&](int s) { return base + kTileBytes * (uint32_t)(kQT + kKStages + s); };
    // Grid (Hq, B, query blocks): the query block varies slowest, so the full 256-row blocks of
    // every (request, head) start first and the ragged last blocks fill the final wave.  (The
    // indices come straight from the grid: integer division costs a fresh CTA tens of cycles
    // each.)
    const int h = (int)blockIdx.x;
    const int b = (int)blockIdx.y;
    const int qb = (int)blockIdx.z;
    const int hk = p.g == 1 ? h : h / p.g;
    // Ragged batches (read-slot keys): request b owns query rows [q_start[b], q_start[b+1]) and
    // read-slot entries [kv_start[b], kv_start[b+1]) of the flattened tensors; p.n_rows and
    // p.T_len are then the largest per-request counts.  A CTA without rows leaves at once.
    int n_rows = p.n_rows, T_len = p.T_len;
    int64_t qbase = (int64_t)b * p.n_rows, kbase = (int64_t)b * p.T_len;
    if (kMode == kSlotKeys && p.q_start) {
        qbase = p.q_start[b];
        kbase = p.kv_start[b];
        n_rows = (int)(p.q_start[b + 1] - qbase);
        T_len = (int)(p.kv_start[b + 1] - kbase);
        if (n_rows != 0 && (n_rows < 0 || n_rows > p.n_rows || T_len < 1 || T_len > p.T_len)) {
            if (threadIdx.x == 0 && qb == 0 && h == 0) flag(p.dev_status, ACACHE_DEV_BAD_LENGTH);
            return;
        }
    }
    const int q0 = qb * kQT * kBM;
    if (q0 >= n_rows) return;
    const int n_qt = min(kQT, (n_rows - q0 + kBM - 1) / kBM);   // Q tiles present (1 or 2)
    const int n_kv = n_key_tiles<kMode>(p, T_len);
    // one Q tile and at least two key tiles: split the keys between the two chains
    const bool split = n_qt == 1 && n_kv >= 2;
    const int n_ch = split ? 2 : n_qt;                  // chains: softmax warpgroups, MMA threads
    const KeySchedule ks{split, n_kv, split ? (n_kv + 1) / 2 : n_kv};
    // with split keys the second Q buffer is free and serves as a third V stage
    const int n_vst = split ? kVStages + 1 : kVStages;
    auto sVs = [&](int s) { return s < kVStages ? sV(s) : sQ(1); };
    const int warp = threadIdx.x >> 5, lane = threadIdx.x & 31, wg = warp >> 2;
    volatile int* abort_flag = &ctl.abort;
    int32_t* dev_status = p.dev_status;
    const long long budget = p.budget;
    // The first key tile's read-slot entries are loaded by the producer lanes before the set-up
    // below and checked only after it, so their latency passes during the set-up instead of
    // holding every warp at its barrier (warp 10 flags bad slots).  The maps are not written
    // by a store grid this launch may overlap.
    const bool prod_warp = warp >= kMmaWarp + 2;
    const bool flagger = warp == kProdWarp;
    int raw0[4] = {-1, -1, -1, -1};
    uint32_t keys0 = 0;
    if (kMode == kSlotKeys && prod_warp) keys0 = tile_slots_load(p, kbase, T_len, n_kv, ks.entry_tile(0), lane, raw0);

    // read-slot K/V stages: one arrival per producer warp of the ring (see the producers)
    constexpr int kFullArrivals = kMode == kSlotKeys ? kProdPerRing : 1;
    if (threadIdx.x == 0) {
        mbar_init(&ctl.q_full, 1);
        // a K or V stage is free once every chain that reads its entry is done with it (both
        // Q tiles' chains; with split keys the one chain the entry belongs to)
        const int readers = split ? 1 : n_qt;
        for (int s = 0; s < kKStages; ++s) {
            mbar_init(&ctl.k_full[s], kFullArrivals);
            mbar_init(&ctl.k_empty[s], readers);
        }
        for (int s = 0; s < kVStages + 1; ++s) {
            mbar_init(&ctl.v_full[s], kFullArrivals);
            mbar_init(&ctl.v_empty[s], readers);
        }
        for (int t = 0; t < kQT; ++t) {
            mbar_init(&ctl.s_full[t], 1);
            mbar_init(&ctl.p_half[t], 128);
            mbar_init(&ctl.p_full[t], 128);
            mbar_init(&ctl.drain[t], 1);
            mbar_init(&ctl.turn[t], 128);
        }
        ctl.abort = 0;
        ctl.unlanded = 0;
        ctl.split_ok = 1;
        fence_mbar_init();
        // the Q tiles, as soon as their barrier exists
        mbar_arrive_expect_tx(&ctl.q_full, kTileBytes * (uint32_t)n_qt);
        for (int t = 0; t < n_qt; ++t) {
            if (kMode == kSlotKeys && p.q_start) {   // 3-D map over the flattened rows
                const int r = (int)(qbase + q0 + t * kBM);
                tma_load_3d(sQ(t), &p.tm_q, 0, h, r, &ctl.q_full);
                tma_load_3d(sQ(t) + kRegion, &p.tm_q, 64, h, r, &ctl.q_full);
            } else {
                tma_load_4d(sQ(t), &p.tm_q, 0, h, q0 + t * kBM, b, &ctl.q_full);
                tma_load_4d(sQ(t) + kRegion, &p.tm_q, 64, h, q0 + t * kBM, b, &ctl.q_full);
            }
        }
    }
    if (warp == kMmaWarp) {
        tmem_alloc(&ctl.tmem_base, kTmemCols);
        tmem_relinquish();
    }
    tc_fence_before();
    __syncthreads();
    tc_fence_after();
    const uint32_t tmem = ctl.tmem_base;

    // Each role's code sits inside the branch of its register reallocation, so the compiler
    // allocates every region against the right register limit.
    if (wg >= 2) {
        setmaxnreg_dec<kRegOther>();
        if (warp >= kMmaWarp + 2) {
            // -------------------------------------------------------------- TMA producers
            if (warp == kProdWarp && lane == 0) {
                if (p.out) tma_prefetch_desc(&p.tm_o);
                tma_prefetch_desc(&p.tm_k0);
                tma_prefetch_desc(&p.tm_v0);
                tma_prefetch_desc(&p.tm_k1);
                tma_prefetch_desc(&p.tm_v1);
            }
            // kProdPerRing warps fill the K ring, as many the V ring (a gather4 costs its warp tens
            // of cycles of issue, so a tile's 64 are spread over the ring's warps); probe tiles are
            // box loads issued by lane 0 of each ring's first warp
            const bool is_v = warp >= kProdWarp + kProdPerRing;
            const int pi = warp - kProdWarp - (is_v ? kProdPerRing : 0);    // place among the ring's warps
            const int nst = is_v ? n_vst : kKStages;
            uint64_t* full = is_v ? ctl.v_full : ctl.k_full;
            uint64_t* empty = is_v ? ctl.v_empty : ctl.k_empty;
            const CUtensorMap* tm_aff = is_v ? &p.tm_v0 : &p.tm_k0;   // slot: the pool
            const CUtensorMap* tm_own = is_v ? &p.tm_v1 : &p.tm_k1;
            const bool leader = pi == 0 && lane == 0;                  // announces the tile's bytes
            if (kMode == kSlotKeys || pi == 0) {
                const int n_aff = (p.L + kBN - 1) / kBN;
                const int oob_row = (int)(p.num_slots * p.Hkv);     // first row outside the pool
                // read-slot keys: this lane's gather x = 4-row group x / 2 of the tile, column
                // half x % 2 of the ring's matrix (K or V); lanes with x >= 64 have none
                const int x = kProdPerRing * lane + pi;
                const bool gathers = x < 64;
                const int g = x >> 1, half = x & 1;
                // Read-slot tile j, resolved one entry ahead (the loads overlap the previous tile's
                // wait and gather issue): lane l reads the slots of keys 4l..4l+3 and the warp votes
                // whether all 128 keys are present with consecutive slots (a request's own rows, a
                // page of the shared region) -- then the tile is two tiled box loads of the pool
                // (slot0 = the first slot), else 64 gather4 loads whose rows each lane takes from
                // the lane that read them.  Every warp of the ring reads the same slots and so
                // takes the same decision.  Invalid slots and keys past T read an out-of-range row.
                auto finish = [&](const int (&sl)[4], int (&rows)[4], int& slot0) -> bool {
                    bool run = sl[0] >= 0 && sl[1] == sl[0] + 1 && sl[2] == sl[0] + 2 && sl[3] == sl[0] + 3;
                    const int after = __shfl_down_sync(0xffffffffu, sl[0], 1);
                    if (lane < 31) run = run && after == sl[0] + 4;
                    slot0 = __shfl_sync(0xffffffffu, sl[0], 0);
#pragma unroll
                    for (int u = 0; u < 4; ++u) {
                        const int sv = __shfl_sync(0xffffffffu, sl[u], g & 31);
                        rows[u] = (gathers && sv >= 0) ? sv * p.Hkv + hk : oob_row;
                    }
                    return __all_sync(0xffffffffu, run);
                };
                auto resolve = [&](int j, int (&rows)[4], int& slot0) -> bool {
                    int sl[4];
                    if (kMode == kSlotKeys) tile_slots<kDrop>(p, kbase, T_len, n_kv, j, lane, flagger, sl);
                    return finish(sl, rows, slot0);
                };
                int next[4], next_slot0;
                int sl0[4];
                tile_slots_check<kDrop>(p, flagger, keys0, raw0, sl0);
                bool next_box = finish(sl0, next, next_slot0);
                // store-then-attend: the pool rows this launch reads may have been written by the
                // preceding store grid (launched ahead with programmatic stream serialisation).
                // Only then may the next grid on the stream start: in a chain of layers it runs on
                // the SMs this grid's last wave leaves idle, and reads its own layer's pool
                // without waiting (that store is complete once this wait returns).
                if (p.early_wait == 1) grid_dependency_wait();
                grid_launch_dependents();
                int armed = -1;                           // last entry this warp arrived on
                for (int e = 0; e < n_kv; ++e) {          // ring entries in load order
                    const int s = ring_stage(e, nst);
                    const int j = ks.entry_tile(e);           // the key tile entry e holds
                    const uint32_t dst_tile = is_v ? sVs(s) : sK(s);
                    int rows[4] = {next[0], next[1], next[2], next[3]};
                    const int slot0 = next_slot0;
                    const bool box = next_box;
                    next_box = resolve(e + 1 < n_kv ? ks.entry_tile(e + 1) : n_kv, next, next_slot0);
                    if (e >= nst &&
                        !__all_sync(0xffffffffu, wait_bar(&empty[s], (ring_lap(e, nst) - 1) & 1, abort_flag, dev_status, budget)))
                        break;
                    // The ring's first warp announces the tile's bytes; a gather of another warp
                    // that completes first leaves the count transiently negative (allowed).  Read-
                    // slot stages count one arrival per warp of the ring, also for a box tile that
                    // the first warp loads alone: no stage then completes a phase without every
                    // warp, so none can fall two phases behind a barrier or get ahead of it -- a
                    // parity wait cannot tell two completed phases from none.  (Without this, a box
                    // tile of split keys, whose chain runs ahead of the other, could be released
                    // twice before a warp busy with the other chain's gathers looked at its stage.)
                    if (leader) mbar_arrive_expect_tx(&full[s], kTileBytes);
                    else if (kMode == kSlotKeys && lane == 0) mbar_arrive(&full[s]);
                    armed = e;
                    __syncwarp();
                    if (kMode == kSlotKeys) {
                        if (box) {
                            if (leader) {
                                tma_load_3d(dst_tile, tm_own, 0, hk, slot0, &full[s]);
                                tma_load_3d(dst_tile + kRegion, tm_own, 64, hk, slot0, &full[s]);
                            }
                        } else if (gathers) {
                            tma_gather4(dst_tile + (uint32_t)half * kRegion + (uint32_t)g * 512u, tm_aff, half * 64,
                                        rows[0], rows[1], rows[2], rows[3], &full[s]);
                        }
                    } else if (lane == 0) {
                        if (j < n_aff) {
                            const int j0 = j * kBN;
                            tma_load_3d(dst_tile, tm_aff, 0, hk, j0, &full[s]);
                            tma_load_3d(dst_tile + kRegion, tm_aff, 64, hk, j0, &full[s]);
                        } else {
                            const int r0 = (j - n_aff) * kBN;
                            tma_load_4d(dst_tile, tm_own, 0, hk, r0, b, &full[s]);
                            tma_load_4d(dst_tile + kRegion, tm_own, 64, hk, r0, b, &full[s]);
                        }
                    }
                }
                // Abort: the loads this warp issued must land before the CTA exits.  Only the
                // last entry armed on each stage can still have loads in flight (an earlier one
                // was consumed before its stage was armed again), so wait, bounded, for those
                // phases.  A phase that another warp of the ring never armed cannot complete:
                // then the CTA holds for a fixed time before it exits instead.
                if (*abort_flag && armed >= 0) {
                    bool landed = true;
                    for (int e = max(0, armed - nst + 1); e <= armed; ++e)
                        landed = mbar_wait(&full[ring_stage(e, nst)], (uint32_t)ring_lap(e, nst) & 1u, kLandBudget) && landed;
                    if (!__all_sync(0xffffffffu, landed) && lane == 0) ctl.unlanded = 1;
                }
            }
        } else {
            // ------------------------------------------------------------------ MMA issuers
            // Warp 8 issues the MMAs of Q tile A, warp 9 those of tile B, so the two chains never
            // wait on each other and their issue runs on two SM sub-partitions.  Per key tile j a
            // thread issues PV_t(j) once P_t(j) is in TMEM, then S_t(j+1).  tcgen05 MMAs of one
            // thread run in issue order, so S_t(j+1) may overwrite the columns P_t(j) occupies,
            // and the completion of S_t(j) implies that of PV_t(j-1).
            const int t = warp - kMmaWarp;
            if (t < n_ch && lane == 0) {
                const uint32_t idS = idesc_bf16(kBM, kBN, false, false);
                const uint32_t idO = idesc_bf16(kBM, kD, false, true);
                const uint32_t d_s = tmem + col_s(t), d_o = tmem + col_o(t);
                const uint64_t dq = sdesc_sw128(sQ(split ? 0 : t), 16, 1024);
                const int nt = ks.n_tiles(t);
                // descriptor start addresses advance in 16-byte units: K step k of a K-major tile
                // is 32 bytes into region k / 4; of the MN-major V tile, 16 rows (2048 bytes)
                auto issue_s = [&](int e) {                   // e: ring entry of the K tile
                    const uint64_t dk = sdesc_sw128(sK(e % kKStages), 16, 1024);
#pragma unroll
                    for (int k = 0; k < kD / 16; ++k) {
                        const uint64_t ko = ((uint64_t)(k >> 2) * kRegion + (uint64_t)(k & 3) * 32u) >> 4;
                        umma_ss(d_s, dq + ko, dk + ko, idS, k > 0);
                    }
                    umma_commit(&ctl.s_full[t]);
                    umma_commit(&ctl.k_empty[e % kKStages]);
                };
                // PV_t(i) in two halves of the key tile: keys 0-63 (k steps 0-3) as soon as the
                // softmax has published the first half of P, keys 64-127 once all of P is in
                auto issue_pv_half = [&](int e, bool acc, int h) {
                    const uint64_t dv = sdesc_sw128(sVs(ring_stage(e, n_vst)), kRegion, 1024);
#pragma unroll
                    for (int k = 4 * h; k < 4 * h + 4; ++k)
                        umma_ts(d_o, d_s + k * 8, dv + (uint64_t)(k * 2048 / 16), idO, (acc || k > 0));
                };
                const int e0 = ks.entry(t, 0);
                bool ok = wait_bar(&ctl.q_full, 0, abort_flag, dev_status, budget) &&
                          wait_bar(&ctl.k_full[e0 % kKStages], (e0 / kKStages) & 1, abort_flag, dev_status, budget);
                if (ok) {
                    tc_fence_after();
                    issue_s(e0);
                }
                for (int i = 0; ok && i < nt; ++i) {
                    const int e = ks.entry(t, i);
                    ok = wait_bar(&ctl.v_full[ring_stage(e, n_vst)], ring_lap(e, n_vst) & 1, abort_flag, dev_status, budget) &&
                         wait_bar(&ctl.p_half[t], i & 1, abort_flag, dev_status, budget);
                    if (!ok) break;
                    tc_fence_after();
                    issue_pv_half(e, i > 0, 0);
                    ok = wait_bar(&ctl.p_full[t], i & 1, abort_flag, dev_status, budget);
                    if (!ok) break;
                    tc_fence_after();
                    issue_pv_half(e, i > 0, 1);
                    umma_commit(&ctl.v_empty[ring_stage(e, n_vst)]);
                    if (i + 1 < nt) {
                        const int en = ks.entry(t, i + 1);
                        ok = wait_bar(&ctl.k_full[en % kKStages], (en / kKStages) & 1, abort_flag, dev_status, budget);
                        if (!ok) break;
                        tc_fence_after();
                        issue_s(en);
                    }
                }
                // no MMA may still run when TMEM is released
                umma_commit(&ctl.drain[t]);
                mbar_wait(&ctl.drain[t], 0, kDrainBudget);
            }
            __syncwarp();
        }
    } else {
        setmaxnreg_inc<kRegSoftmax>();
        if (wg < n_ch) {
        // ------------------------------------------------------------------ softmax + epilogue
        const int t = wg;                                  // chain (Q tile) of this warpgroup
        const int r = threadIdx.x - t * 128;               // query row in the tile = TMEM lane
        const uint32_t lane_base = tmem + ((uint32_t)((warp & 3) * 32) << 16);
        const float c = p.scale_log2;                      // > 0
        // With two Q tiles the warpgroups take turns: A(0), B(0), A(1), B(1), ...  Each then
        // has the SM's issue slots and exponential units to itself, and the tensor core runs
        // one tile's MMAs while the other tile's softmax runs, instead of both at once.
        const bool pingpong = n_ch > 1;
        const int nt = ks.n_tiles(t);
        float m_used = -INFINITY, l_sum = 0.f;
        bool ok = true;
        for (int i = 0; i < nt; ++i) {
            const int j = ks.tile(t, i);                   // key tile of this step
            // discarded keys of tile j: bit i of drop[cc] = key 32 cc + i (loaded before the
            // wait for S_t(j), which hides the latency)
            uint32_t drop[4] = {0u, 0u, 0u, 0u};
            if constexpr (kDrop) {
                const int32_t* rs = p.read_slot + kbase;
#pragma unroll
                for (int cc = 0; cc < 4; ++cc) {
                    const int tk = j * kBN + cc * 32 + (threadIdx.x & 31);
                    drop[cc] = __ballot_sync(0xffffffffu, tk < T_len && rs[tk] == ACACHE_SLOT_NONE);
                }
            }
            ok = __all_sync(0xffffffffu, wait_bar(&ctl.s_full[t], i & 1, abort_flag, dev_status, budget));
            if (!ok) break;
            tc_fence_after();
            // S_t(j) is read into registers as soon as it is ready -- typically while the tensor
            // core is idle -- before waiting for this warpgroup's turn: TMEM reads slow down
            // concurrent MMAs, and the other tile's MMAs run during the other turn
            uint32_t v[4][32];
#pragma unroll
            for (int cc = 0; cc < 4; ++cc) tmem_ld32(lane_base + col_s(t) + cc * 32, v[cc]);
            tmem_ld_wait();
            if (pingpong && (t == 1 || i > 0))
                ok = __all_sync(0xffffffffu, wait_bar(&ctl.turn[t], (t == 0 ? i - 1 : i) & 1,
                                                      abort_flag, dev_status, budget));
            if (!ok) break;
            const int valid = tile_valid<kMode>(p, j, T_len);
            if (valid < kBN) {
#pragma unroll
                for (int cc = 0; cc < 4; ++cc)
#pragma unroll
                    for (int i = 0; i < 32; ++i)
                        if (cc * 32 + i >= valid) v[cc][i] = __float_as_uint(-INFINITY);
            }
            if constexpr (kDrop) {
#pragma unroll
                for (int cc = 0; cc < 4; ++cc)
                    if (drop[cc]) {
#pragma unroll
                        for (int i = 0; i < 32; ++i)
                            if ((drop[cc] >> i) & 1u) v[cc][i] = __float_as_uint(-INFINITY);
                    }
            }
            // row maximum of the raw logits (four independent chains of three-input maxima)
            float mx[4];
#pragma unroll
            for (int cc = 0; cc < 4; ++cc) {
                mx[cc] = max3f(__uint_as_float(v[cc][0]), __uint_as_float(v[cc][1]), __uint_as_float(v[cc][2]));
#pragma unroll
                for (int i = 3; i < 31; i += 2)
                    mx[cc] = max3f(mx[cc], __uint_as_float(v[cc][i]), __uint_as_float(v[cc][i + 1]));
                mx[cc] = fmaxf(mx[cc], __uint_as_float(v[cc][31]));
            }
            const float mt = max3f(mx[0], mx[1], fmaxf(mx[2], mx[3])) * c;
            float alpha = 1.f;
            bool resc = false;
            if (i == 0) {
                m_used = mt;
            } else if (mt > m_used + kRescaleThreshold) {
                alpha = fast_exp2(m_used - mt);
                m_used = mt;
                resc = true;
            }
            if (__any_sync(0xffffffffu, resc)) {
                // S_t(j) completed after PV_t(j-1): O_t is final up to tile j-1; rescale it,
                // 8 columns at a time (rare; the S values stay live meanwhile, so this path
                // must not raise the loop's register peak)
#pragma unroll 1
                for (int q = 0; q < kD / 8; ++q) {
                    uint32_t o[8];
                    tmem_ld8(lane_base + col_o(t) + q * 8, o);
                    tmem_ld_wait();
#pragma unroll
                    for (int x = 0; x < 8; ++x) o[x] = __float_as_uint(__uint_as_float(o[x]) * alpha);
                    tmem_st8(lane_base + col_o(t) + q * 8, o);
                }
                tmem_st_wait();
            }
            // a row whose keys so far were all discarded exponentiates against 0 (every value is -inf)
            const float ms = (kDrop && m_used == -INFINITY) ? 0.f : m_used;
            const uint64_t c2 = f2pack(c, c), nm2 = f2pack(-ms, -ms);
            uint64_t ls2[2] = {f2pack(0.f, 0.f), f2pack(0.f, 0.f)};
            // P_j as bf16 pairs (64 columns) overwrites the first half of S_j's columns, 16
            // columns at a time, so only one chunk of packed values is live.  Keys 0-63 are
            // published first (p_half) so the first half of PV_j runs while keys 64-127 are
            // exponentiated.
#pragma unroll
            for (int cc = 0; cc < 4; ++cc) {
                uint32_t pk[16];
#pragma unroll
                for (int i = 0; i < 32; i += 2) {
                    // exponent arguments of two keys with one packed FMA
                    float x0, x1;
                    f2unpack(f2fma(f2pack(__uint_as_float(v[cc][i]), __uint_as_float(v[cc][i + 1])), c2, nm2),
                             x0, x1);
                    const float p0 = fast_exp2(x0), p1 = fast_exp2(x1);
                    ls2[(i >> 1) & 1] = f2add(ls2[(i >> 1) & 1], f2pack(p0, p1));
                    __nv_bfloat162 two = __floats2bfloat162_rn(p0, p1);   // low half = lower key
                    pk[i >> 1] = *reinterpret_cast<uint32_t*>(&two);
                }
                tmem_st16(lane_base + col_s(t) + cc * 16, pk);
                if (cc == 1) {
                    tmem_st_wait();
                    tc_fence_before();
                    mbar_arrive(&ctl.p_half[t]);
                }
            }
            float l0, l1, l2, l3;
            f2unpack(ls2[0], l0, l1);
            f2unpack(ls2[1], l2, l3);
            l_sum = l_sum * alpha + ((l0 + l1) + (l2 + l3));
            tmem_st_wait();
            tc_fence_before();
            mbar_arrive(&ctl.p_full[t]);
            if (pingpong) mbar_arrive(&ctl.turn[t ^ 1]);
        }
        // drain[t] is committed after the last PV of this chain
        if (ok) ok = __all_sync(0xffffffffu, wait_bar(&ctl.drain[t], 0, abort_flag, dev_status, budget));
        // Split keys: chain B hands its row maximum and row sum to chain A, which merges the two
        // partial states -- O = O_A 2^(m_A - m) + O_B 2^(m_B - m) with m = max(m_A, m_B), the
        // sums alike -- and stores the rows.  A chain whose keys so far were all discarded has
        // m = -inf and weight 0.
        float w_a = 1.f, w_b = 0.f;
        if (split) {
            if (t == 1) {
                ctl.split_m[r] = m_used;
                ctl.split_l[r] = l_sum;
                if (!ok) ctl.split_ok = 0;
            }
            named_barrier_sync<1>(2 * kBM);
            if (t == 1) {
                ok = false;                                // chain A stores the rows
            } else if (ok) {
                ok = ctl.split_ok &&
                     __all_sync(0xffffffffu, wait_bar(&ctl.drain[1], 0, abort_flag, dev_status, budget));
                const float mb = ctl.split_m[r], lb = ctl.split_l[r];
                const float m = fmaxf(m_used, mb);
                w_a = m_used == -INFINITY ? 0.f : fast_exp2(m_used - m);
                w_b = mb == -INFINITY ? 0.f : fast_exp2(mb - m);
                l_sum = l_sum * w_a + lb * w_b;
                m_used = m;
            }
        }
        // the grids this one follows may still read the scratch it writes: wait for them
        if (p.early_wait == 2) grid_dependency_wait();
        // Output rows leave through this chain's Q buffer, free once its MMAs (and with split
        // keys chain B's) are complete, and two tensor-map stores of whole 256-byte row slices,
        // instead of per-thread 16-byte stores scattered at the query-row stride.  A ragged
        // batch's partial last block keeps per-thread stores: its box would reach into the next
        // request's rows.
        const bool writer = !split || t == 0;
        const bool boxed = p.out && !(kMode == kSlotKeys && p.q_start && q0 + (t + 1) * kBM > n_rows);
        const uint32_t stage = sQ(t);
        if (ok) {
            tc_fence_after();
            const int i = q0 + t * kBM + r;
            const float inv_l = (kDrop && !(l_sum > 0.f)) ? 0.f : 1.f / l_sum;
            bf16* orow = (p.out && !boxed) ? p.out + ((qbase + i) * p.Hq + h) * kD : nullptr;
#pragma unroll
            for (int cc = 0; cc < 4; ++cc) {
                uint32_t o[32];
                tmem_ld32(lane_base + col_o(t) + cc * 32, o);
                tmem_ld_wait();
                if (split) {
                    uint32_t ob[32];
                    tmem_ld32(lane_base + col_o(1) + cc * 32, ob);
                    tmem_ld_wait();
#pragma unroll
                    for (int x = 0; x < 32; ++x)
                        o[x] = __float_as_uint(fmaf(__uint_as_float(o[x]), w_a, __uint_as_float(ob[x]) * w_b));
                }
                if (boxed || (orow && i < n_rows)) {
                    uint32_t pkd[16];
#pragma unroll
                    for (int x = 0; x < 16; ++x) {
                        __nv_bfloat162 two = __floats2bfloat162_rn(__uint_as_float(o[2 * x]) * inv_l,
                                                                   __uint_as_float(o[2 * x + 1]) * inv_l);
                        pkd[x] = *reinterpret_cast<uint32_t*>(&two);
                    }
                    if (boxed) {
                        // 16-byte chunk k = 4 cc + x of row r: region k / 8, swizzled position
                        // (k % 8) ^ (r % 8) -- the layout the 128-byte-swizzled map expects
#pragma unroll
                        for (int x = 0; x < 4; ++x) {
                            const int k = 4 * cc + x;
                            st_shared_v4(stage + (uint32_t)(k >> 3) * kRegion + (uint32_t)r * 128u +
                                             ((uint32_t)((k & 7) ^ (r & 7)) << 4),
                                         pkd[4 * x], pkd[4 * x + 1], pkd[4 * x + 2], pkd[4 * x + 3]);
                        }
                    } else {
                        uint4* dst = reinterpret_cast<uint4*>(orow + cc * 32);
#pragma unroll
                        for (int x = 0; x < 4; ++x)
                            dst[x] = make_uint4(pkd[4 * x], pkd[4 * x + 1], pkd[4 * x + 2], pkd[4 * x + 3]);
                    }
                }
            }
            if (p.stat_m && i < p.n_rows) {
                const int64_t so = ((int64_t)b * p.Hq + h) * p.n_rows + i;
                p.stat_m[so] = m_used;
                p.stat_l[so] = l_sum;
            }
        }
        if (writer && boxed) {
            // every thread of the warpgroup arrives (ok or not); the rows go out only if all of
            // them were written
            fence_proxy_async_smem();
            const bool all_ok = t == 0 ? named_barrier_and<2>(kBM, ok) : named_barrier_and<3>(kBM, ok);
            if (r == 0 && all_ok) {
                if (kMode == kSlotKeys && p.q_start) {
                    const int row = (int)(qbase + q0 + t * kBM);
                    tma_store_3d(&p.tm_o, stage, 0, h, row);
                    tma_store_3d(&p.tm_o, stage + kRegion, 64, h, row);
                } else {
                    tma_store_4d(&p.tm_o, stage, 0, h, q0 + t * kBM, b);
                    tma_store_4d(&p.tm_o, stage + kRegion, 64, h, q0 + t * kBM, b);
                }
                bulk_commit_group();
                bulk_wait_group_read0();     // the buffer must outlive the reads
            }
        }
        }
    }
    tc_fence_before();
    __syncthreads();
    tc_fence_after();
    if (*abort_flag) {
        // the Q tiles' loads, too, land before the CTA exits
        if (threadIdx.x == 0 && !mbar_wait(&ctl.q_full, 0, kLandBudget)) ctl.unlanded = 1;
        __syncthreads();
        settle_after_abort(ctl.unlanded != 0);
    }
    if (warp == kMmaWarp) tmem_dealloc(tmem, kTmemCols);
    // A grid of a chain of layers reads nothing its predecessor writes, so it never waited
    // for it; it waits before its CTAs exit instead, so the grids of a chain complete in
    // launch order and work behind the chain on the stream sees every layer's output.  (The
    // predecessor has long finished by then: this grid started in its last wave.)  A chained
    // probe forward waited before its epilogue; a CTA that gave up a wait and skipped it waits
    // here, so that its grid still completes after the ones it follows.
    if (p.early_wait != 1 && threadIdx.x == 0) grid_dependency_wait();
}

// ------------------------------------------------------------------------------------------
// Persistent read-slot attention (the slot_attn step of the ACache page: every logical position
// reads its K/V through the request's read-slot map), for a batch of equal-length requests with
// no discarded keys, when there are more units than SMs.  tc_attn_kernel starts one CTA per
// 256-row query block of a (request, head), and each pays for starting a fresh CTA, filling its
// rings and draining its last tiles.  Here one CTA per SM works through units u = blockIdx.x,
// blockIdx.x + gridDim.x, ...  A unit is the work of one tc_attn_kernel CTA, taken in that
// kernel's grid order.  Every ring and barrier carries on from one unit into the next:
//   - the producers load the next unit's first K/V tiles while the current unit finishes;
//   - each chain's next Q tile is prefetched into L2 while the unit runs, and loaded once the
//     epilogue's store has read the rows staged in its buffer;
//   - chain A starts its next unit while chain B, a turn behind, finishes the current one.
//
// Ring accounting is uniform: both chains release every K and V entry.  A chain that does not
// read an entry releases it as soon as it has landed.  Such entries are the other chain's half
// of split keys, and every entry of the idle chain in a unit with one Q tile and one key tile.
// So each chain waits for every entry in ring order, and no barrier phase goes by unseen.
//
// With split keys both Q buffers hold the unit's tile, one per chain, so each buffer is loaded
// and read by one chain only.  Every barrier gets one phase per unit (drain, Q), per tile (S,
// P, turn) or per split unit (the hand-off), and each is waited in order.
struct PersistCtl {
    uint64_t q_full[kQT];         // Q buffer t holds the unit's tile (a bare phase when it has none)
    uint64_t k_full[kKStages];
    uint64_t k_empty[kKStages];
    uint64_t v_full[kVStages];
    uint64_t v_empty[kVStages];
    uint64_t s_full[kQT];
    uint64_t p_half[kQT];
    uint64_t p_full[kQT];
    uint64_t turn[kQT];
    uint64_t drain[kQT];          // chain t's MMAs of the unit are complete
    uint64_t split_ready;         // split keys: chain B's row statistics are written,
    uint64_t split_done;          //   and chain A has read them and O_B
    uint64_t fin[kQT];            // end of the kernel: chain t's MMAs are complete
    uint32_t tmem_base;
    int abort;
    int unlanded;
    uint32_t q_last[kQT];         // parity of the last phase issued on q_full[t] (abort path: it may be in flight)
    float split_m[kBM];
    float split_l[kBM];
};

// Unit u of a persistent launch: query block (slowest), request, query head.
struct PUnit {
    int h, b, hk, q0, n_qt;
    KeySchedule ks;
    ACACHE_DEVFN int n_ch() const { return ks.split ? 2 : n_qt; }
    ACACHE_DEVFN int nt(int t) const { return t < n_ch() ? ks.n_tiles(t) : 0; }
};
ACACHE_DEVFN PUnit punit(const AttnParams& p, int u, int n_kv) {
    PUnit w;
    const int qb = (int)p.div_bhq((uint32_t)u), bh = u - qb * p.B * p.Hq;
    w.b = (int)p.div_hq((uint32_t)bh);
    w.h = bh - w.b * p.Hq;
    w.hk = (int)p.div_g((uint32_t)w.h);
    w.q0 = qb * kQT * kBM;
    w.n_qt = min(kQT, (p.n_rows - w.q0 + kBM - 1) / kBM);
    const bool split = w.n_qt == 1 && n_kv >= 2;
    w.ks = KeySchedule{split, n_kv, split ? (n_kv + 1) / 2 : n_kv};
    return w;
}

__global__ void __launch_bounds__(kThreads, 1)
tc_slot_persist_kernel(const __grid_constant__ AttnParams p) {
    extern __shared__ uint8_t dsm[];
    __shared__ PersistCtl ctl;
    const uint32_t base = (smem_u32(dsm) + 1023u) & ~1023u;
    // shared memory: Q_A, Q_B, the K ring, the V ring (32 KB tiles, 1024-byte aligned)
    auto sQ = [&](int t) { return base + kTileBytes * (uint32_t)t; };
    auto sK = [&](int s) { return base + kTileBytes * (uint32_t)(kQT + s); };
    auto sV = [&](int s) { return base + kTileBytes * (uint32_t)(kQT + kKStages + s); };
    const int n_kv = p.n_kv;
    const int n_units = p.n_units;
    const int u_first = (int)blockIdx.x, u_step = (int)gridDim.x;
    const int warp = threadIdx.x >> 5, lane = threadIdx.x & 31, wg = warp >> 2;
    // (the pipeline waits take their abort flag, status word and budget straight from shared and
    // parameter memory: held in registers they would crowd the 48-register roles)
    volatile int* abort_flag = &ctl.abort;
    // Q buffer t of unit w: its tile t, with split keys a copy of its one tile, else a bare phase
    auto load_q = [&](const PUnit& w, int t) {
        if (t < w.n_qt || w.ks.split) {
            const int row = w.q0 + (w.ks.split ? 0 : t) * kBM;
            mbar_arrive_expect_tx(&ctl.q_full[t], kTileBytes);
            tma_load_4d(sQ(t), &p.tm_q, 0, w.h, row, w.b, &ctl.q_full[t]);
            tma_load_4d(sQ(t) + kRegion, &p.tm_q, 64, w.h, row, w.b, &ctl.q_full[t]);
        } else {
            mbar_arrive(&ctl.q_full[t]);
        }
    };
    // The producers load the read-slot entries of the first unit's first key tile before the set-
    // up and check them after it (as tc_attn_kernel does): their latency passes meanwhile.
    int raw0[4] = {-1, -1, -1, -1};
    uint32_t keys0 = 0;
    if (warp >= kMmaWarp + 2) {
        const int b0 = punit(p, u_first, n_kv).b;
        keys0 = tile_slots_load(p, (int64_t)b0 * p.T_len, p.T_len, n_kv, 0, lane, raw0);
    }
    if (threadIdx.x == 0) {
        for (int s = 0; s < kKStages; ++s) {
            mbar_init(&ctl.k_full[s], kProdPerRing);
            mbar_init(&ctl.k_empty[s], kQT);
        }
        for (int s = 0; s < kVStages; ++s) {
            mbar_init(&ctl.v_full[s], kProdPerRing);
            mbar_init(&ctl.v_empty[s], kQT);
        }
        for (int t = 0; t < kQT; ++t) {
            mbar_init(&ctl.q_full[t], 1);
            mbar_init(&ctl.s_full[t], 1);
            mbar_init(&ctl.p_half[t], 128);
            mbar_init(&ctl.p_full[t], 128);
            mbar_init(&ctl.turn[t], 128);
            mbar_init(&ctl.drain[t], 1);
            mbar_init(&ctl.fin[t], 1);
            ctl.q_last[t] = 0;
        }
        mbar_init(&ctl.split_ready, 128);
        mbar_init(&ctl.split_done, 128);
        ctl.abort = 0;
        ctl.unlanded = 0;
        fence_mbar_init();
        const PUnit w0 = punit(p, u_first, n_kv);     // gridDim.x <= the number of units
        load_q(w0, 0);
        load_q(w0, 1);
    }
    if (warp == kMmaWarp) {
        tmem_alloc(&ctl.tmem_base, kTmemCols);
        tmem_relinquish();
    }
    tc_fence_before();
    __syncthreads();
    tc_fence_after();
    const uint32_t tmem = ctl.tmem_base;

    if (wg >= 2) {
        setmaxnreg_dec<kRegOther>();
        if (warp >= kMmaWarp + 2) {
            // -------------------------------------------------------------- TMA producers
            // (as in tc_attn_kernel: kProdPerRing warps per ring, one arrival per warp and entry,
            // read-slot tiles resolved one entry ahead -- here across unit boundaries too)
            if (warp == kProdWarp && lane == 0) {
                tma_prefetch_desc(&p.tm_o);
                tma_prefetch_desc(&p.tm_k0);
                tma_prefetch_desc(&p.tm_v0);
                tma_prefetch_desc(&p.tm_k1);
                tma_prefetch_desc(&p.tm_v1);
            }
            const bool is_v = warp >= kProdWarp + kProdPerRing;
            const int pi = warp - kProdWarp - (is_v ? kProdPerRing : 0);
            const int nst = is_v ? kVStages : kKStages;
            uint64_t* full = is_v ? ctl.v_full : ctl.k_full;
            uint64_t* empty = is_v ? ctl.v_empty : ctl.k_empty;
            const CUtensorMap* tm_rows = is_v ? &p.tm_v0 : &p.tm_k0;   // pool rows (gather4)
            const CUtensorMap* tm_box = is_v ? &p.tm_v1 : &p.tm_k1;    // pool [slot][Hkv][d] (boxes)
            const bool leader = pi == 0 && lane == 0;
            const bool flagger = warp == kProdWarp;
            const int oob_row = (int)(p.num_slots * p.Hkv);
            const int x = kProdPerRing * lane + pi;
            const bool gathers = x < 64;
            const int g = x >> 1, half = x & 1;
            auto finish = [&](const int (&sl)[4], int hk, int (&rows)[4], int& slot0) -> bool {
                bool run = sl[0] >= 0 && sl[1] == sl[0] + 1 && sl[2] == sl[0] + 2 && sl[3] == sl[0] + 3;
                const int after = __shfl_down_sync(0xffffffffu, sl[0], 1);
                if (lane < 31) run = run && after == sl[0] + 4;
                slot0 = __shfl_sync(0xffffffffu, sl[0], 0);
#pragma unroll
                for (int q = 0; q < 4; ++q) {
                    const int sv = __shfl_sync(0xffffffffu, sl[q], g & 31);
                    rows[q] = (gathers && sv >= 0) ? sv * p.Hkv + hk : oob_row;
                }
                return __all_sync(0xffffffffu, run);
            };
            auto resolve = [&](const PUnit& w, int j, int (&rows)[4], int& slot0) -> bool {
                int sl[4];
                tile_slots<false>(p, (int64_t)w.b * p.T_len, p.T_len, n_kv, j, lane, flagger, sl);
                return finish(sl, w.hk, rows, slot0);
            };
            int u = u_first, e = 0;
            PUnit w = punit(p, u, n_kv);
            int next[4], next_slot0;
            int sl0[4];
            tile_slots_check<false>(p, flagger, keys0, raw0, sl0);
            bool next_box = finish(sl0, w.hk, next, next_slot0);
            // store-then-attend: the pool may have been written by the preceding grid
            if (p.early_wait == 1) grid_dependency_wait();
            grid_launch_dependents();
            int armed = -1;                                   // last entry this warp arrived on
            for (int eg = 0; u < n_units; ++eg) {             // ring entries in load order
                const int s = ring_stage(eg, nst);
                const uint32_t dst = is_v ? sV(s) : sK(s);
                const int rows[4] = {next[0], next[1], next[2], next[3]};
                const int slot0 = next_slot0, hk = w.hk;
                const bool box = next_box;
                if (++e == n_kv) {
                    e = 0;
                    u += u_step;
                    if (u < n_units) w = punit(p, u, n_kv);
                }
                if (u < n_units) next_box = resolve(w, w.ks.entry_tile(e), next, next_slot0);
                if (eg >= nst &&
                    !__all_sync(0xffffffffu, wait_bar(&empty[s], (ring_lap(eg, nst) - 1) & 1, &ctl.abort, p.dev_status, p.budget)))
                    break;
                if (leader) mbar_arrive_expect_tx(&full[s], kTileBytes);
                else if (lane == 0) mbar_arrive(&full[s]);
                armed = eg;
                __syncwarp();
                if (box) {
                    if (leader) {
                        tma_load_3d(dst, tm_box, 0, hk, slot0, &full[s]);
                        tma_load_3d(dst + kRegion, tm_box, 64, hk, slot0, &full[s]);
                    }
                } else if (gathers) {
                    tma_gather4(dst + (uint32_t)half * kRegion + (uint32_t)g * 512u, tm_rows, half * 64, rows[0],
                                rows[1], rows[2], rows[3], &full[s]);
                }
            }
            // abort: the loads this warp issued land before the CTA exits (see tc_attn_kernel)
            if (*abort_flag && armed >= 0) {
                bool landed = true;
                for (int a = max(0, armed - nst + 1); a <= armed; ++a)
                    landed = mbar_wait(&full[ring_stage(a, nst)], (uint32_t)ring_lap(a, nst) & 1u, kLandBudget) && landed;
                if (!__all_sync(0xffffffffu, landed) && lane == 0) ctl.unlanded = 1;
            }
        } else {
            // ------------------------------------------------------------------ MMA issuers
            // (as in tc_attn_kernel; chain t reads Q buffer t in every unit).  One body serves both
            // chains: compiled once per chain it spilled nothing but ran slower, the larger code
            // costing more instruction-fetch stalls than the spill.
            {
                const int t = warp - kMmaWarp;
                if (lane == 0) {
                    const uint32_t idS = idesc_bf16(kBM, kBN, false, false);
                    const uint32_t idO = idesc_bf16(kBM, kD, false, true);
                    const uint32_t d_s = tmem + col_s(t), d_o = tmem + col_o(t);
                    const uint64_t dq = sdesc_sw128(sQ(t), 16, 1024);
                    auto issue_s = [&](int eg) {
                        const uint64_t dk = sdesc_sw128(sK(ring_stage(eg, kKStages)), 16, 1024);
#pragma unroll
                        for (int kk = 0; kk < kD / 16; ++kk) {
                            const uint64_t ko = ((uint64_t)(kk >> 2) * kRegion + (uint64_t)(kk & 3) * 32u) >> 4;
                            umma_ss(d_s, dq + ko, dk + ko, idS, kk > 0);
                        }
                        umma_commit(&ctl.s_full[t]);
                        umma_commit(&ctl.k_empty[ring_stage(eg, kKStages)]);
                    };
                    auto issue_pv_half = [&](int eg, bool acc, int hh) {
                        const uint64_t dv = sdesc_sw128(sV(eg & 1), kRegion, 1024);
#pragma unroll
                        for (int kk = 4 * hh; kk < 4 * hh + 4; ++kk)
                            umma_ts(d_o, d_s + kk * 8, dv + (uint64_t)(kk * 2048 / 16), idO, (acc || kk > 0));
                    };
                    // parity bit 0 counts this chain's tiles (P), bit 1 the units (Q); E the ring
                    // entries of the units before
                    uint32_t ph = 0;
                    int E = 0;
                    for (int u = u_first; u < n_units; u += u_step) {
                        int nt, n0;
                        bool split;
                        {
                            const PUnit w = punit(p, u, n_kv);
                            nt = w.nt(t);
                            n0 = w.ks.n0;
                            split = w.ks.split;
                        }
                        // Entries this chain does not read are released once landed.  Unsplit units:
                        // both chains read every entry (the idle chain of a one-tile unit, which then
                        // has one key tile, reads none).  Split keys (KeySchedule): the entries alternate
                        // chain A, chain B, chain A's extra tile (odd n_kv) last, so the entry before
                        // each of this chain's own is the other chain's -- released (K before the S, V
                        // before the PV) -- and so is the last entry if this chain does not own it.
                        const int n1 = n_kv - n0;
                        auto entry = [&](int i) { return split ? (i < n1 ? 2 * i + t : n1 + i) : i; };
                        auto rel_k = [&](int eg) -> bool {
                            if (!wait_bar(&ctl.k_full[ring_stage(eg, kKStages)], ring_lap(eg, kKStages) & 1, &ctl.abort,
                                          p.dev_status, p.budget))
                                return false;
                            mbar_arrive(&ctl.k_empty[ring_stage(eg, kKStages)]);
                            return true;
                        };
                        auto rel_v = [&](int eg) -> bool {
                            if (!wait_bar(&ctl.v_full[eg & 1], (eg >> 1) & 1, &ctl.abort, p.dev_status, p.budget))
                                return false;
                            mbar_arrive(&ctl.v_empty[eg & 1]);
                            return true;
                        };
                        bool ok = wait_bar(&ctl.q_full[t], (ph >> 1) & 1u, &ctl.abort, p.dev_status, p.budget);
                        if (ok && nt > 0) {
                            const int e0 = entry(0);
                            ok = (!split || e0 == 0 || rel_k(E + e0 - 1)) &&
                                 wait_bar(&ctl.k_full[ring_stage(E + e0, kKStages)], ring_lap(E + e0, kKStages) & 1,
                                          &ctl.abort, p.dev_status, p.budget);
                            if (ok) {
                                tc_fence_after();
                                issue_s(E + e0);
                            }
                            for (int i = 0; ok && i < nt; ++i) {
                                const int e = entry(i), eg = E + e;
                                const uint32_t pp = (ph ^ (uint32_t)i) & 1u;
                                ok = (!split || e == 0 || rel_v(eg - 1)) &&
                                     wait_bar(&ctl.v_full[eg & 1], (eg >> 1) & 1, &ctl.abort, p.dev_status, p.budget) &&
                                     wait_bar(&ctl.p_half[t], pp, &ctl.abort, p.dev_status, p.budget);
                                if (!ok) break;
                                tc_fence_after();
                                issue_pv_half(eg, i > 0, 0);
                                ok = wait_bar(&ctl.p_full[t], pp, &ctl.abort, p.dev_status, p.budget);
                                if (!ok) break;
                                tc_fence_after();
                                issue_pv_half(eg, i > 0, 1);
                                umma_commit(&ctl.v_empty[eg & 1]);
                                if (i + 1 < nt) {
                                    const int egn = E + entry(i + 1);
                                    ok = (!split || rel_k(egn - 1)) &&
                                         wait_bar(&ctl.k_full[ring_stage(egn, kKStages)], ring_lap(egn, kKStages) & 1,
                                                  &ctl.abort, p.dev_status, p.budget);
                                    if (!ok) break;
                                    tc_fence_after();
                                    issue_s(egn);
                                }
                            }
                            // split keys: the last entry, if the other chain's
                            if (ok && split && ((n_kv & 1) == t)) ok = rel_k(E + n_kv - 1) && rel_v(E + n_kv - 1);
                        } else if (ok) {
                            // idle chain: every entry (one key tile)
                            for (int e = 0; ok && e < n_kv; ++e) ok = rel_k(E + e) && rel_v(E + e);
                        }
                        if (!ok) break;
                        umma_commit(&ctl.drain[t]);
                        E += n_kv;
                        ph ^= (uint32_t)(nt & 1) | 2u;
                    }
                    // no MMA may still run when TMEM is released
                    umma_commit(&ctl.fin[t]);
                    mbar_wait(&ctl.fin[t], 0, kDrainBudget);
                }
            }
            __syncwarp();
        }
    } else {
        setmaxnreg_inc<kRegSoftmax>();
        // ------------------------------------------------------------------ softmax + epilogue
        // (the tile loop is tc_attn_kernel's; phases count on across units)
        const int t = wg;
        const int r = threadIdx.x - t * 128;
        const uint32_t lane_base = tmem + ((uint32_t)((warp & 3) * 32) << 16);
        const float c = p.scale_log2;
        const uint32_t stage = sQ(t);
        // Barrier phases are used by parity only: bit 0 counts this chain's tiles (S, P), bits 1
        // and 2 chain A's and chain B's tiles of ping-pong units (turns), bit 3 the units (drain),
        // bit 4 the split units (hand-off).
        // (the unit and the parity bits share one register, u << 5 | bits, and the unit's tile
        // count, first key tile and ping-pong flag another: few values stay live through the
        // tile loop, whose S tile fills most of the softmax warps' registers)
        for (uint32_t su = (uint32_t)u_first << 5; (int)(su >> 5) < n_units; su += (uint32_t)u_step << 5) {
            const int u = (int)(su >> 5);
            uint32_t cfg;      // bits 0-15 tiles of this chain, 16-30 its first key tile, 31 ping-pong
            {
                const PUnit w = punit(p, u, n_kv);
                cfg = (uint32_t)w.nt(t) | (uint32_t)((w.ks.split && t == 1) ? w.ks.n0 : 0) << 16 |
                      (w.n_ch() > 1 ? 0x80000000u : 0u);
            }
            const int un = u + u_step;
            // the next unit's Q tile of this buffer into L2 while this unit runs
            if (r == 0 && un < n_units) {
                const PUnit wn = punit(p, un, n_kv);
                if (t < wn.n_qt || wn.ks.split) {
                    const int row = wn.q0 + (wn.ks.split ? 0 : t) * kBM;
                    tma_prefetch_l2_4d(&p.tm_q, 0, wn.h, row, wn.b);
                    tma_prefetch_l2_4d(&p.tm_q, 64, wn.h, row, wn.b);
                }
            }
            float m_used = -INFINITY, l_sum = 0.f;
            bool ok = true;
            const int nt = (int)(cfg & 0xffffu);
            for (int i = 0; i < nt; ++i) {
                const int j = (int)((cfg >> 16) & 0x7fffu) + i;
                ok = __all_sync(0xffffffffu, wait_bar(&ctl.s_full[t], (su ^ (uint32_t)i) & 1u, &ctl.abort, p.dev_status, p.budget));
                if (!ok) break;
                tc_fence_after();
                uint32_t v[4][32];
#pragma unroll
                for (int cc = 0; cc < 4; ++cc) tmem_ld32(lane_base + col_s(t) + cc * 32, v[cc]);
                tmem_ld_wait();
                if ((cfg >> 31) && (t == 1 || i > 0))
                    ok = __all_sync(0xffffffffu, wait_bar(&ctl.turn[t], ((t == 0 ? (su >> 2) ^ 1u : su >> 1) ^ (uint32_t)i) & 1u,
                                                          &ctl.abort, p.dev_status, p.budget));
                if (!ok) break;
                const int valid = min(kBN, p.T_len - j * kBN);
                if (valid < kBN) {
#pragma unroll
                    for (int cc = 0; cc < 4; ++cc)
#pragma unroll
                        for (int q = 0; q < 32; ++q)
                            if (cc * 32 + q >= valid) v[cc][q] = __float_as_uint(-INFINITY);
                }
                float mx[4];
#pragma unroll
                for (int cc = 0; cc < 4; ++cc) {
                    mx[cc] = max3f(__uint_as_float(v[cc][0]), __uint_as_float(v[cc][1]), __uint_as_float(v[cc][2]));
#pragma unroll
                    for (int q = 3; q < 31; q += 2)
                        mx[cc] = max3f(mx[cc], __uint_as_float(v[cc][q]), __uint_as_float(v[cc][q + 1]));
                    mx[cc] = fmaxf(mx[cc], __uint_as_float(v[cc][31]));
                }
                const float mt = max3f(mx[0], mx[1], fmaxf(mx[2], mx[3])) * c;
                float alpha = 1.f;
                bool resc = false;
                if (i == 0) {
                    m_used = mt;
                } else if (mt > m_used + kRescaleThreshold) {
                    alpha = fast_exp2(m_used - mt);
                    m_used = mt;
                    resc = true;
                }
                if (__any_sync(0xffffffffu, resc)) {
#pragma unroll 1
                    for (int q = 0; q < kD / 8; ++q) {
                        uint32_t o[8];
                        tmem_ld8(lane_base + col_o(t) + q * 8, o);
                        tmem_ld_wait();
#pragma unroll
                        for (int xx = 0; xx < 8; ++xx) o[xx] = __float_as_uint(__uint_as_float(o[xx]) * alpha);
                        tmem_st8(lane_base + col_o(t) + q * 8, o);
                    }
                    tmem_st_wait();
                }
                const uint64_t c2 = f2pack(c, c), nm2 = f2pack(-m_used, -m_used);
                uint64_t ls2[2] = {f2pack(0.f, 0.f), f2pack(0.f, 0.f)};
#pragma unroll
                for (int cc = 0; cc < 4; ++cc) {
                    uint32_t pk[16];
#pragma unroll
                    for (int q = 0; q < 32; q += 2) {
                        float x0, x1;
                        f2unpack(f2fma(f2pack(__uint_as_float(v[cc][q]), __uint_as_float(v[cc][q + 1])), c2, nm2),
                                 x0, x1);
                        const float p0 = fast_exp2(x0), p1 = fast_exp2(x1);
                        ls2[(q >> 1) & 1] = f2add(ls2[(q >> 1) & 1], f2pack(p0, p1));
                        __nv_bfloat162 two = __floats2bfloat162_rn(p0, p1);
                        pk[q >> 1] = *reinterpret_cast<uint32_t*>(&two);
                    }
                    tmem_st16(lane_base + col_s(t) + cc * 16, pk);
                    if (cc == 1) {
                        tmem_st_wait();
                        tc_fence_before();
                        mbar_arrive(&ctl.p_half[t]);
                    }
                }
                float l0, l1, l2, l3;
                f2unpack(ls2[0], l0, l1);
                f2unpack(ls2[1], l2, l3);
                l_sum = l_sum * alpha + ((l0 + l1) + (l2 + l3));
                tmem_st_wait();
                tc_fence_before();
                mbar_arrive(&ctl.p_full[t]);
                if (cfg >> 31) mbar_arrive(&ctl.turn[t ^ 1]);
            }
            // drain[t] is committed after the chain's last MMA of the unit (once per unit, also
            // when the chain has no tile); then Q buffer t is free
            if (ok) ok = __all_sync(0xffffffffu, wait_bar(&ctl.drain[t], (su >> 3) & 1u, &ctl.abort, p.dev_status, p.budget));
            // the unit's indices again (recomputed rather than held through the tile loop)
            int u2 = (int)(su >> 5);
            asm volatile("" : "+r"(u2));
            const PUnit w = punit(p, u2, n_kv);
            // Split keys: chain B hands its row statistics to chain A (split_ready) and waits
            // until A has read them and O_B (split_done) before its next tile may overwrite O_B.
            float w_a = 1.f, w_b = 0.f;
            if (w.ks.split) {
                if (t == 1) {
                    ctl.split_m[r] = m_used;
                    ctl.split_l[r] = l_sum;
                    mbar_arrive(&ctl.split_ready);
                } else if (ok) {
                    ok = __all_sync(0xffffffffu, wait_bar(&ctl.split_ready, (su >> 4) & 1u, &ctl.abort, p.dev_status, p.budget)) &&
                         !*abort_flag &&
                         __all_sync(0xffffffffu, wait_bar(&ctl.drain[1], (su >> 3) & 1u, &ctl.abort, p.dev_status, p.budget));
                    if (ok) {
                        const float mb = ctl.split_m[r], lb = ctl.split_l[r];
                        const float m = fmaxf(m_used, mb);
                        w_a = m_used == -INFINITY ? 0.f : fast_exp2(m_used - m);
                        w_b = mb == -INFINITY ? 0.f : fast_exp2(mb - m);
                        l_sum = l_sum * w_a + lb * w_b;
                    }
                }
            }
            // The rows, normalised, leave through this chain's Q buffer and two tensor-map stores
            // (as in tc_attn_kernel); the buffer then takes the next unit's Q tile.
            const bool writer = nt > 0 && (!w.ks.split || t == 0);
            if (writer && ok) {
                tc_fence_after();
                const float inv_l = 1.f / l_sum;
                // (not unrolled: it runs once per unit, and a smaller loop body keeps the
                // instruction cache for the tile loop)
#pragma unroll 1
                for (int cc = 0; cc < 4; ++cc) {
                    uint32_t o[32];
                    tmem_ld32(lane_base + col_o(t) + cc * 32, o);
                    tmem_ld_wait();
                    if (w.ks.split) {
                        uint32_t ob[32];
                        tmem_ld32(lane_base + col_o(1) + cc * 32, ob);
                        tmem_ld_wait();
#pragma unroll
                        for (int xx = 0; xx < 32; ++xx)
                            o[xx] = __float_as_uint(fmaf(__uint_as_float(o[xx]), w_a, __uint_as_float(ob[xx]) * w_b));
                    }
                    uint32_t pkd[16];
#pragma unroll
                    for (int xx = 0; xx < 16; ++xx) {
                        __nv_bfloat162 two = __floats2bfloat162_rn(__uint_as_float(o[2 * xx]) * inv_l,
                                                                   __uint_as_float(o[2 * xx + 1]) * inv_l);
                        pkd[xx] = *reinterpret_cast<uint32_t*>(&two);
                    }
#pragma unroll
                    for (int xx = 0; xx < 4; ++xx) {
                        const int kc = 4 * cc + xx;
                        st_shared_v4(stage + (uint32_t)(kc >> 3) * kRegion + (uint32_t)r * 128u +
                                         ((uint32_t)((kc & 7) ^ (r & 7)) << 4),
                                     pkd[4 * xx], pkd[4 * xx + 1], pkd[4 * xx + 2], pkd[4 * xx + 3]);
                    }
                }
            }
            if (w.ks.split) {
                if (t == 0) {
                    tc_fence_before();
                    mbar_arrive(&ctl.split_done);
                } else if (ok) {
                    ok = __all_sync(0xffffffffu, wait_bar(&ctl.split_done, (su >> 4) & 1u, &ctl.abort, p.dev_status, p.budget));
                }
            }
            if (writer) fence_proxy_async_smem();
            // every thread of the warpgroup takes part in every unit's vote, so its four warps
            // leave the loop together
            const bool all_ok = t == 0 ? named_barrier_and<2>(kBM, ok) : named_barrier_and<3>(kBM, ok);
            if (r == 0 && all_ok) {
                if (writer) {
                    const int row = w.q0 + (w.ks.split ? 0 : t) * kBM;
                    tma_store_4d(&p.tm_o, stage, 0, w.h, row, w.b);
                    tma_store_4d(&p.tm_o, stage + kRegion, 64, w.h, row, w.b);
                    bulk_commit_group();
                    bulk_wait_group_read0();
                }
                if (un < n_units) {
                    load_q(punit(p, un, n_kv), t);
                    ctl.q_last[t] = ((su >> 3) & 1u) ^ 1u;
                }
            }
            if (!all_ok) break;
            su ^= (uint32_t)(w.nt(t) & 1) | 8u | (w.ks.split ? 16u : 0u);
            if (w.n_ch() > 1) su ^= (uint32_t)((w.nt(0) & 1) << 1 | (w.nt(1) & 1) << 2);
        }
    }
    tc_fence_before();
    __syncthreads();
    tc_fence_after();
    if (*abort_flag) {
        // the last Q load issued on each buffer lands before the CTA exits (an earlier one was
        // waited for before the next was issued)
        if (threadIdx.x == 0)
            for (int t = 0; t < kQT; ++t)
                if (!mbar_wait(&ctl.q_full[t], ctl.q_last[t], kLandBudget)) ctl.unlanded = 1;
        __syncthreads();
        settle_after_abort(ctl.unlanded != 0);
    }
    if (warp == kMmaWarp) tmem_dealloc(tmem, kTmemCols);
    // a chained layer waits for the grid before it before its CTAs exit (see tc_attn_kernel)
    if (p.early_wait != 1 && threadIdx.x == 0) grid_dependency_wait();
}

// ------------------------------------------------------------------------------------------
// Second probe pass.
constexpr int kCsStages = 2;
constexpr int kCsMmaWarp = 4;
constexpr int kCsProdWarp = 5;
constexpr int kCsThreads = (kCsProdWarp + 1) * 32;   // one producer warp
constexpr uint32_t kCsSmemBytes = kTileBytes * (1 + kCsStages) + 1024;
constexpr uint32_t kCsTmemCols = 256;

struct ColsumParams {
    CUtensorMap tm_kaff;  // 3-D affix keys [L][Hkv][d], box {64, 1, 128}
    CUtensorMap tm_q;     // 2-D probe queries [B*P*Hq][d], box {64, 1} (gather4)
    CUtensorMap tm_qbox;  // 4-D probe queries [B][P][Hq][d], box {64, 1, 128, 1}
    const int32_t* masked;
    const float* stat_m;
    const float* stat_l;
    float* partial;
    int32_t* dev_status;
    int B, P, L, m, Hq, Hkv;
    float scale_log2;
    long long budget;     // cycles a pipeline wait may take before it gives up
};

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

__global__ void __launch_bounds__(kCsThreads, 2)
tc_colsum_kernel(const __grid_constant__ ColsumParams p) {
    extern __shared__ uint8_t dsm[];
    __shared__ ColsumCtl ctl;
    // launched behind the probe forward (programmatic dependent launch): its row statistics are
    // read below; the head sum after this grid may start waiting now
    grid_launch_dependents();
    grid_dependency_wait();
    const uint32_t base = (smem_u32(dsm) + 1023u) & ~1023u;
    const uint32_t sA = base;
    const int n_jt = (p.L + kBN - 1) / kBN;
    const int jt = blockIdx.x % n_jt;
    const int h = (blockIdx.x / n_jt) % p.Hq;
    const int b = blockIdx.x / (n_jt * p.Hq);
    const int hk = h / (p.Hq / p.Hkv);
    const int j0 = jt * kBN;
    const int n_ch = (p.m + kBN - 1) / kBN;
    const int warp = threadIdx.x >> 5, lane = threadIdx.x & 31;
    volatile int* abort_flag = &ctl.abort;
    int32_t* dev_status = p.dev_status;
    const long long budget = p.budget;

    if (threadIdx.x == 0) {
        mbar_init(&ctl.a_full, 1);
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
    if (warp == kCsMmaWarp) {
        tmem_alloc(&ctl.tmem_base, kCsTmemCols);
        tmem_relinquish();
    }
    tc_fence_before();
    __syncthreads();
    tc_fence_after();
    const uint32_t tmem = ctl.tmem_base;

    if (warp == kCsProdWarp) {
        const float* sm_row = p.stat_m + ((int64_t)b * p.Hq + h) * p.P;
        const float* sl_row = p.stat_l + ((int64_t)b * p.Hq + h) * p.P;
        const int32_t* mrow = p.masked + (int64_t)b * p.m;
        const int oob_row = p.B * p.P * p.Hq;               // first row outside the queries
        if (lane == 0) {
            tma_prefetch_desc(&p.tm_kaff);
            tma_prefetch_desc(&p.tm_q);
            mbar_arrive_expect_tx(&ctl.a_full, kTileBytes);
            tma_load_3d(sA, &p.tm_kaff, 0, hk, j0, &ctl.a_full);
            tma_load_3d(sA + kRegion, &p.tm_kaff, 64, hk, j0, &ctl.a_full);
        }
        for (int c = 0; c < n_ch; ++c) {
            const int s = c % kCsStages;
            const uint32_t sB = base + kTileBytes * (1 + s);
            int rows[4];
            float sm[4], sil[4];
#pragma unroll
            for (int u = 0; u < 4; ++u) {
                const int k = c * kBN + 4 * lane + u;
                const int pr = k < p.m ? mrow[k] : -1;
                const bool good = pr >= 0 && pr < p.P;
                if (k < p.m && !good) flag(dev_status, ACACHE_DEV_BAD_ROW);
                rows[u] = good ? ((b * p.P + pr) * p.Hq + h) : oob_row;
                sm[u] = good ? sm_row[pr] : INFINITY;
                sil[u] = good ? 1.f / sl_row[pr] : 0.f;
            }
            if (c >= kCsStages) {
                const uint32_t par = ((c / kCsStages) - 1) & 1;
                if (!__all_sync(0xffffffffu, wait_bar(&ctl.b_empty[s], par, abort_flag, dev_status, budget) &&
                                                 wait_bar(&ctl.cons_done[s], par, abort_flag, dev_status, budget)))
                    break;
            }
            // every lane stores its rows' statistics before its arrival on b_full publishes
            // them (lane 0 arrives through the expect_tx that announces the chunk's bytes,
            // before any lane issues its loads)
#pragma unroll
            for (int u = 0; u < 4; ++u) {
                ctl.st_m[s][4 * lane + u] = sm[u];
                ctl.st_il[s][4 * lane + u] = sil[u];
            }
            // The initially masked rows are normally one run of consecutive probe rows (the
            // generation positions): then the chunk is two tiled box loads of 128 rows instead
            // of 64 gathers.  Rows of the box past the masked set are loaded but skipped (their
            // statistics say so); rows past P read as zeros.
            const int r0 = __shfl_sync(0xffffffffu, mrow[min(c * kBN, p.m - 1)], 0);
            bool run = r0 >= 0 && r0 + kBN <= p.P + kBN;
#pragma unroll
            for (int u = 0; u < 4; ++u) {
                const int k = c * kBN + 4 * lane + u;
                if (k < p.m) run = run && mrow[k] == r0 + 4 * lane + u;
            }
            run = __all_sync(0xffffffffu, run);
            if (lane == 0) mbar_arrive_expect_tx(&ctl.b_full[s], kTileBytes);
            __syncwarp();
            if (run) {
                if (lane == 0) {
                    tma_load_4d(sB, &p.tm_qbox, 0, h, r0, b, &ctl.b_full[s]);
                    tma_load_4d(sB + kRegion, &p.tm_qbox, 64, h, r0, b, &ctl.b_full[s]);
                }
            } else {
                const uint32_t o = (uint32_t)lane * 512u;
                tma_gather4(sB + o, &p.tm_q, 0, rows[0], rows[1], rows[2], rows[3], &ctl.b_full[s]);
                tma_gather4(sB + kRegion + o, &p.tm_q, 64, rows[0], rows[1], rows[2], rows[3], &ctl.b_full[s]);
            }
            if (lane != 0) mbar_arrive(&ctl.b_full[s]);
        }
    } else if (warp == kCsMmaWarp) {
        if (lane == 0) {
            const uint32_t id = idesc_bf16(kBN, kBN, false, false);
            bool ok = wait_bar(&ctl.a_full, 0, abort_flag, dev_status, budget);
            for (int c = 0; ok && c < n_ch; ++c) {
                const int s = c % kCsStages, db = c & 1;
                ok = wait_bar(&ctl.b_full[s], (c / kCsStages) & 1, abort_flag, dev_status, budget);
                if (ok && c >= 2) ok = wait_bar(&ctl.cons_done[db], ((c >> 1) - 1) & 1, abort_flag, dev_status, budget);
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
            mbar_wait(&ctl.drain, 0, kDrainBudget);
        }
        __syncwarp();
    } else {
        const int r = threadIdx.x;                         // affix key j0 + r
        const uint32_t lane_base = tmem + ((uint32_t)(warp * 32) << 16);
        const float c2 = p.scale_log2;
        // four partial sums (masked row k goes to sum k % 4), added in a fixed order at the
        // end: deterministic, and four times shorter dependency chains
        float acc4[4] = {0.f, 0.f, 0.f, 0.f};
        bool ok = true;
        for (int c = 0; c < n_ch; ++c) {
            const int s = c % kCsStages, db = c & 1;
            // the stats of this chunk were published with b_full; D with d_full
            ok = __all_sync(0xffffffffu,
                            wait_bar(&ctl.b_full[s], (c / kCsStages) & 1, abort_flag, dev_status, budget) &&
                            wait_bar(&ctl.d_full[db], (c >> 1) & 1, abort_flag, dev_status, budget));
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
                    acc4[i & 3] = fmaf(fast_exp2(fmaf(__uint_as_float(v[i]), c2, -ctl.st_m[s][k])), ctl.st_il[s][k],
                                       acc4[i & 3]);
                }
            }
            tc_fence_before();
            mbar_arrive(&ctl.cons_done[db]);
        }
        if (ok && j0 + r < p.L)
            p.partial[((int64_t)b * p.Hq + h) * p.L + j0 + r] = (acc4[0] + acc4[1]) + (acc4[2] + acc4[3]);
    }
    tc_fence_before();
    __syncthreads();
    tc_fence_after();
    settle_after_abort(*abort_flag != 0);
    if (warp == kCsMmaWarp) tmem_dealloc(tmem, kCsTmemCols);
}

// ------------------------------------------------------------------------------------------
// Second probe pass with the masked rows resident (m <= 256: one or two chunks of 128 rows, the
// usual case).  One CTA per (request, query head, run of affix tiles): the producer loads the
// masked query rows once, with their statistics, then streams the run's affix key tiles through
// four stages; the MMA warp computes D_i = K_affix_tile_i Q_masked^T into one of two TMEM
// buffers (a 128-column block per chunk) while the consumers exponentiate the other.  Consumer
// warpgroup g takes chunk g; its thread r owns affix key r of every tile and sums over the
// chunk's masked rows k into four partial sums (k % 4), added in a fixed order; the second
// warpgroup hands its sum to the first through shared memory, which adds it last.
constexpr int kCrMaxChunks = 2;
constexpr int kCrMmaWarp = 8;                 // warps 0-7: two consumer warpgroups
constexpr int kCrProdWarp = 9;
constexpr int kCrThreads = (kCrProdWarp + 1) * 32;
constexpr int kCrKStages = 4;                 // affix key tile stages
constexpr uint32_t kCrSmemBytes = kTileBytes * (kCrMaxChunks + kCrKStages) + 1024;
constexpr uint32_t kCrTmemCols = 512;                                      // 2 buffers x 2 chunks

struct ColsumRowsCtl {
    uint64_t q_full;                  // the masked rows and their statistics
    uint64_t k_full[kCrKStages], k_empty[kCrKStages];   // affix key tile stages
    uint64_t d_full[2];               // D buffer i holds the scores of a tile
    uint64_t cons_done[2];            // the consumers are done with D buffer i
    uint64_t drain;
    uint32_t tmem_base;
    int abort;
    int unlanded;                     // abort path: a load issued before the abort may not have landed
    float st_off[kCrMaxChunks][kBN];  // per masked row: row maximum (log2 domain) + log2(row
                                      // sum), so its probabilities are 2^(logit - off); +inf = skip
    float xsum[2][kBN];               // the second consumer warpgroup's sums, by tile parity
};

__global__ void __launch_bounds__(kCrThreads, 1)
tc_colsum_rows_kernel(const __grid_constant__ ColsumParams p, int tiles_per_cta) {
    extern __shared__ uint8_t dsm[];
    __shared__ ColsumRowsCtl ctl;
    // Launched behind the probe forward (programmatic dependent launch), whose row statistics
    // it reads: the producer warp loads the masked rows and the first key tiles (inputs of the
    // call, complete before the forward started) and only then waits for the forward.  The
    // head sum after this grid may start waiting at once.
    grid_launch_dependents();
    const uint32_t base = (smem_u32(dsm) + 1023u) & ~1023u;
    // Masked rows: 64-column half r of chunk c at sQ(c, r), so that the two chunks' halves are
    // adjacent and one MMA operand of N = 256 rows covers both chunks.
    auto sQ = [&](int c, int r) { return base + kTileBytes * (uint32_t)r + kRegion * (uint32_t)c; };
    auto sKs = [&](int s) { return base + kTileBytes * (uint32_t)(kCrMaxChunks + s); };
    const int n_jt = (p.L + kBN - 1) / kBN;
    const int n_grp = (n_jt + tiles_per_cta - 1) / tiles_per_cta;
    const int grp = blockIdx.x % n_grp;
    const int h = (blockIdx.x / n_grp) % p.Hq;
    const int b = blockIdx.x / (n_grp * p.Hq);
    const int hk = h / (p.Hq / p.Hkv);
    const int jt0 = grp * tiles_per_cta;
    const int n_t = min(n_jt, jt0 + tiles_per_cta) - jt0;
    const int n_ch = (p.m + kBN - 1) / kBN;
    if (n_t <= 0 || n_ch > kCrMaxChunks) {
        grid_dependency_wait();      // the grid still completes after the forward
        return;
    }
    const int warp = threadIdx.x >> 5, lane = threadIdx.x & 31;
    volatile int* abort_flag = &ctl.abort;
    int32_t* dev_status = p.dev_status;
    const long long budget = p.budget;

    if (threadIdx.x == 0) {
        mbar_init(&ctl.q_full, 33);   // the byte count's arrival + every producer lane's statistics
        for (int s = 0; s < kCrKStages; ++s) {
            mbar_init(&ctl.k_full[s], 1);
            mbar_init(&ctl.k_empty[s], 1);
        }
        for (int s = 0; s < 2; ++s) {
            mbar_init(&ctl.d_full[s], 1);
            mbar_init(&ctl.cons_done[s], 256);
        }
        mbar_init(&ctl.drain, 1);
        ctl.abort = 0;
        ctl.unlanded = 0;
        fence_mbar_init();
    }
    if (warp == kCrMmaWarp) {
        tmem_alloc(&ctl.tmem_base, kCrTmemCols);
        tmem_relinquish();
    }
    tc_fence_before();
    __syncthreads();
    tc_fence_after();
    const uint32_t tmem = ctl.tmem_base;

    if (warp == kCrProdWarp) {
        const float* sm_row = p.stat_m + ((int64_t)b * p.Hq + h) * p.P;
        const float* sl_row = p.stat_l + ((int64_t)b * p.Hq + h) * p.P;
        const int32_t* mrow = p.masked + (int64_t)b * p.m;
        const int oob_row = p.B * p.P * p.Hq;               // first row outside the queries
        if (lane == 0) {
            tma_prefetch_desc(&p.tm_kaff);
            tma_prefetch_desc(&p.tm_q);
            tma_prefetch_desc(&p.tm_qbox);
        }
        // The masked rows (probe rows pr[c][u]; -1 = none or bad), then their loads: lane 0's
        // expect_tx announces all chunks' bytes before any load is issued.
        int rows[kCrMaxChunks][4], pr[kCrMaxChunks][4], r0[kCrMaxChunks];
        bool run[kCrMaxChunks];
#pragma unroll
        for (int c = 0; c < kCrMaxChunks; ++c) {
            run[c] = false;
            r0[c] = 0;
#pragma unroll
            for (int u = 0; u < 4; ++u) pr[c][u] = -1;
            if (c >= n_ch) continue;
#pragma unroll
            for (int u = 0; u < 4; ++u) {
                const int k = c * kBN + 4 * lane + u;
                const int x = k < p.m ? mrow[k] : -1;
                const bool good = x >= 0 && x < p.P;
                if (k < p.m && !good) flag(dev_status, ACACHE_DEV_BAD_ROW);
                rows[c][u] = good ? ((b * p.P + x) * p.Hq + h) : oob_row;
                pr[c][u] = good ? x : -1;
            }
            // a chunk of consecutive probe rows (the generation positions) is two tiled box
            // loads; rows of the box past the masked set are skipped by their statistics
            r0[c] = __shfl_sync(0xffffffffu, mrow[min(c * kBN, p.m - 1)], 0);
            bool ok_run = r0[c] >= 0 && r0[c] + kBN <= p.P + kBN;
#pragma unroll
            for (int u = 0; u < 4; ++u) {
                const int k = c * kBN + 4 * lane + u;
                if (k < p.m) ok_run = ok_run && mrow[k] == r0[c] + 4 * lane + u;
            }
            run[c] = __all_sync(0xffffffffu, ok_run);
        }
        __syncwarp();
        if (lane == 0) mbar_arrive_expect_tx(&ctl.q_full, kTileBytes * (uint32_t)n_ch);
        __syncwarp();
#pragma unroll
        for (int c = 0; c < kCrMaxChunks; ++c) {
            if (c >= n_ch) continue;
            if (run[c]) {
                if (lane == 0) {
                    tma_load_4d(sQ(c, 0), &p.tm_qbox, 0, h, r0[c], b, &ctl.q_full);
                    tma_load_4d(sQ(c, 1), &p.tm_qbox, 64, h, r0[c], b, &ctl.q_full);
                }
            } else {
                const uint32_t o = (uint32_t)lane * 512u;
                tma_gather4(sQ(c, 0) + o, &p.tm_q, 0, rows[c][0], rows[c][1], rows[c][2], rows[c][3], &ctl.q_full);
                tma_gather4(sQ(c, 1) + o, &p.tm_q, 64, rows[c][0], rows[c][1], rows[c][2], rows[c][3],
                            &ctl.q_full);
            }
        }
        // the first affix key tiles (every stage is free)
        const int n_pre = min(n_t, kCrKStages);
        if (lane == 0) {
            for (int i = 0; i < n_pre; ++i) {
                mbar_arrive_expect_tx(&ctl.k_full[i], kTileBytes);
                tma_load_3d(sKs(i), &p.tm_kaff, 0, hk, (jt0 + i) * kBN, &ctl.k_full[i]);
                tma_load_3d(sKs(i) + kRegion, &p.tm_kaff, 64, hk, (jt0 + i) * kBN, &ctl.k_full[i]);
            }
        }
        // The row statistics are the forward's output: wait for that grid, then read them past
        // L1.  Each probability is 2^(logit - off) with off = row maximum + log2(row sum).
        grid_dependency_wait();
#pragma unroll
        for (int c = 0; c < kCrMaxChunks; ++c) {
            if (c >= n_ch) continue;
#pragma unroll
            for (int u = 0; u < 4; ++u)
                ctl.st_off[c][4 * lane + u] =
                    pr[c][u] >= 0 ? __ldcg(sm_row + pr[c][u]) + log2f(__ldcg(sl_row + pr[c][u])) : INFINITY;
        }
        mbar_arrive(&ctl.q_full);
        // the rest of the run's affix key tiles, kCrKStages stages
        int armed = n_pre - 1;                               // last key tile loaded
        for (int i = n_pre; i < n_t; ++i) {
            const int s = i % kCrKStages;
            if (!__all_sync(0xffffffffu,
                            wait_bar(&ctl.k_empty[s], ((i / kCrKStages) - 1) & 1, abort_flag, dev_status, budget)))
                break;
            if (lane == 0) {
                const int j0 = (jt0 + i) * kBN;
                mbar_arrive_expect_tx(&ctl.k_full[s], kTileBytes);
                tma_load_3d(sKs(s), &p.tm_kaff, 0, hk, j0, &ctl.k_full[s]);
                tma_load_3d(sKs(s) + kRegion, &p.tm_kaff, 64, hk, j0, &ctl.k_full[s]);
            }
            armed = i;
            __syncwarp();
        }
        // Abort: every load this warp issued lands before the CTA exits.  Only the last tile
        // of each stage can still be in flight; wait, bounded, for those phases and the masked
        // rows, else hold the CTA for a fixed time.
        if (*abort_flag && lane == 0) {
            bool landed = mbar_wait(&ctl.q_full, 0, kLandBudget);
            for (int e = max(0, armed - kCrKStages + 1); e <= armed; ++e)
                landed = mbar_wait(&ctl.k_full[e % kCrKStages], (uint32_t)(e / kCrKStages) & 1u, kLandBudget) && landed;
            if (!landed) ctl.unlanded = 1;
        }
    } else if (warp == kCrMmaWarp) {
        if (lane == 0) {
            // one MMA per k-step covers every chunk: N = 128 or 256 masked rows (rows past m are
            // zero-filled by their loads, so every column the consumers read is written)
            const uint32_t id = idesc_bf16(kBN, kBN * n_ch, false, false);
            bool ok = wait_bar(&ctl.q_full, 0, abort_flag, dev_status, budget);
            for (int i = 0; ok && i < n_t; ++i) {
                const int ks = i % kCrKStages, db = i & 1;     // key stage, D buffer
                ok = wait_bar(&ctl.k_full[ks], (i / kCrKStages) & 1, abort_flag, dev_status, budget);
                if (ok && i >= 2) ok = wait_bar(&ctl.cons_done[db], ((i >> 1) - 1) & 1, abort_flag, dev_status, budget);
                if (!ok) break;
                tc_fence_after();
#pragma unroll
                for (int k = 0; k < kD / 16; ++k) {
                    const uint32_t kcol = (uint32_t)(k & 3) * 32u;     // 16 columns within a half
                    umma_ss(tmem + (uint32_t)db * 256u, sdesc_sw128(sKs(ks) + (uint32_t)(k >> 2) * kRegion + kcol, 16, 1024),
                            sdesc_sw128(sQ(0, k >> 2) + kcol, 16, 1024), id, k > 0);
                }
                umma_commit(&ctl.d_full[db]);
                umma_commit(&ctl.k_empty[ks]);
            }
            umma_commit(&ctl.drain);
            mbar_wait(&ctl.drain, 0, kDrainBudget);
        }
        __syncwarp();
    } else {
        const int cg = warp >> 2;                          // consumer warpgroup = its chunk
        const int r = threadIdx.x & 127;                   // affix key r of every tile
        const uint32_t lane_base = tmem + ((uint32_t)((warp & 3) * 32) << 16);
        const float c2 = p.scale_log2;
        bool ok = wait_bar(&ctl.q_full, 0, abort_flag, dev_status, budget);
        for (int i = 0; i < n_t; ++i) {
            const int s = i & 1;
            ok = ok && wait_bar(&ctl.d_full[s], (i >> 1) & 1, abort_flag, dev_status, budget);
            // both warpgroups take the same decision, so neither waits for the other in vain
            ok = named_barrier_and<1>(256, ok);
            if (!ok) break;
            tc_fence_after();
            float acc4[4] = {0.f, 0.f, 0.f, 0.f};
            if (cg < n_ch) {
                // the chunk's 128 columns in one round trip to TMEM
                uint32_t v[4][32];
#pragma unroll
                for (int cc = 0; cc < 4; ++cc)
                    tmem_ld32(lane_base + (uint32_t)s * 256u + (uint32_t)cg * kBN + cc * 32, v[cc]);
                tmem_ld_wait();
#pragma unroll
                for (int cc = 0; cc < 4; ++cc) {
#pragma unroll
                    for (int e = 0; e < 32; ++e)
                        acc4[e & 3] += fast_exp2(fmaf(__uint_as_float(v[cc][e]), c2, -ctl.st_off[cg][cc * 32 + e]));
                }
            }
            tc_fence_before();
            mbar_arrive(&ctl.cons_done[s]);
            const float sum = (acc4[0] + acc4[1]) + (acc4[2] + acc4[3]);
            if (cg == 1) ctl.xsum[s][r] = sum;
            named_barrier_sync<2>(256);
            const int j = (jt0 + i) * kBN + r;
            if (cg == 0 && j < p.L) p.partial[((int64_t)b * p.Hq + h) * p.L + j] = sum + ctl.xsum[s][r];
        }
    }
    tc_fence_before();
    __syncthreads();
    tc_fence_after();
    if (*abort_flag) settle_after_abort(ctl.unlanded != 0);
    if (warp == kCrMmaWarp) tmem_dealloc(tmem, kCrTmemCols);
}

// A launch with programmatic stream serialisation (the grid may start before the one it follows
// has completed; it waits for that grid itself).
template <typename... KArgs, typename... Args>
int launch_pdl(void (*kern)(KArgs...), unsigned grid, unsigned threads, uint32_t smem, cudaStream_t stream,
               Args... args) {
    cudaLaunchConfig_t cfg = {};
    cfg.gridDim = dim3(grid);
    cfg.blockDim = dim3(threads);
    cfg.dynamicSmemBytes = smem;
    cfg.stream = stream;
    cudaLaunchAttribute attr[1];
    attr[0].id = cudaLaunchAttributeProgrammaticStreamSerialization;
    attr[0].val.programmaticStreamSerializationAllowed = 1;
    cfg.attrs = attr;
    cfg.numAttrs = 1;
    if (cudaLaunchKernelEx(&cfg, kern, args...) != cudaSuccess) {
        (void)cudaGetLastError();
        return ACACHE_ERR_CUDA;
    }
    return launch_status();
}

// pdl: launched with programmatic stream serialisation after a grid that releases it early --
// a store (store-then-attend; prm.early_wait orders the pool reads after it) or the attention
// of another layer (chained layers; prm.early_wait = 0).
template <int kMode, bool kDrop = false>
int launch_attn(AttnParams prm, int B, cudaStream_t stream, bool pdl = false) {
    const int64_t n_qb = (prm.n_rows + kQT * kBM - 1) / (kQT * kBM);
    if ((int64_t)B * prm.Hq * n_qb == 0) return ACACHE_OK;
    if (B > 65535 || n_qb > 65535) return ACACHE_ERR_INVALID_ARG;
    const dim3 grid((unsigned)prm.Hq, (unsigned)B, (unsigned)n_qb);
    prm.g = prm.Hq / prm.Hkv;
    auto kern = tc_attn_kernel<kMode, kDrop>;
    if (cudaFuncSetAttribute(kern, cudaFuncAttributeMaxDynamicSharedMemorySize, kSmemBytes) != cudaSuccess) {
        (void)cudaGetLastError();
        return ACACHE_ERR_CUDA;
    }
    if (!pdl) {
        kern<<<grid, kThreads, kSmemBytes, stream>>>(prm);
        return launch_status();
    }
    cudaLaunchConfig_t cfg = {};
    cfg.gridDim = grid;
    cfg.blockDim = dim3(kThreads);
    cfg.dynamicSmemBytes = kSmemBytes;
    cfg.stream = stream;
    cudaLaunchAttribute attr[1];
    attr[0].id = cudaLaunchAttributeProgrammaticStreamSerialization;
    attr[0].val.programmaticStreamSerializationAllowed = 1;
    cfg.attrs = attr;
    cfg.numAttrs = 1;
    if (cudaLaunchKernelEx(&cfg, kern, prm) != cudaSuccess) {
        (void)cudaGetLastError();
        return ACACHE_ERR_CUDA;
    }
    return launch_status();
}

// The persistent kernel: one CTA per SM.
int launch_attn_persist(AttnParams prm, int B, cudaStream_t stream, bool pdl) {
    const int64_t n_units = (int64_t)B * prm.Hq * ((prm.n_rows + kQT * kBM - 1) / (kQT * kBM));
    prm.g = prm.Hq / prm.Hkv;
    prm.B = B;
    prm.n_kv = (prm.T_len + kBN - 1) / kBN;
    prm.n_units = (int)n_units;
    prm.div_bhq = make_fastdiv((uint32_t)(B * prm.Hq));
    prm.div_hq = make_fastdiv((uint32_t)prm.Hq);
    prm.div_g = make_fastdiv((uint32_t)prm.g);
    const unsigned grid = (unsigned)std::min<int64_t>(n_units, sm_count());
    if (cudaFuncSetAttribute(tc_slot_persist_kernel, cudaFuncAttributeMaxDynamicSharedMemorySize, kSmemBytes) !=
        cudaSuccess) {
        (void)cudaGetLastError();
        return ACACHE_ERR_CUDA;
    }
    if (!pdl) {
        tc_slot_persist_kernel<<<grid, kThreads, kSmemBytes, stream>>>(prm);
        return launch_status();
    }
    return launch_pdl(tc_slot_persist_kernel, grid, kThreads, kSmemBytes, stream, prm);
}

}  // namespace

bool tc_supported(const AttnArgs& a) { return a.dtype == ACACHE_BF16 && a.d == kD && a.scale > 0.f; }

// The persistent kernel saves a fixed time at each unit boundary.  With two query tiles per
// unit its tile loop runs a little slower per key tile (more instruction-fetch stalls under
// ncu), so there it pays for short units only: at most 20 key tiles (measured against
// tc_attn_kernel per launch: 2-6 % faster at 11 tiles, 1.5 % at 17; even at 21 and 35; 1.5-2.3 %
// slower at 68).  Units of one query tile (n_q <= 128: block decoding), whose keys the two chains
// split, measured 1-2.5 % faster at every length tried (22, 35 and 68 key tiles).  One wave or
// less stays on tc_attn_kernel: each CTA would take a single unit, and the fresh-CTA kernel
// starts a little sooner and gives a lone query tile's split keys a third V stage.
bool tc_slot_persistent(const AttnArgs& a, int B, int n_q, int T_len) {
    const int64_t n_units = (int64_t)B * a.hq * (((int64_t)n_q + kQT * kBM - 1) / (kQT * kBM));
    const int64_t n_kv = ((int64_t)T_len + kBN - 1) / kBN;
    return tc_supported(a) && n_units > sm_count() && n_units < (1 << 22) && n_kv < (1 << 15) &&
           (n_kv <= 20 || n_q <= kBM);
}

int launch_tc_slot_attention(const AttnArgs& a, int B, int n_q, const void* q, int T_len,
                             const int32_t* read_slot, const void* k_cache, const void* v_cache,
                             int64_t num_slots, void* out, int32_t* dev_status,
                             cudaStream_t stream, bool drop_none, bool pdl, bool chained) {
    if ((int64_t)num_slots * a.hkv >= 0x7fffffffLL || (int64_t)B * n_q >= 0x7fffffffLL)
        return ACACHE_ERR_INVALID_ARG;
    AttnParams prm{};
    const uint64_t dq[4] = {(uint64_t)kD, (uint64_t)a.hq, (uint64_t)n_q, (uint64_t)B};
    const uint64_t dp[2] = {(uint64_t)kD, (uint64_t)num_slots * a.hkv};
    const uint64_t d3[3] = {(uint64_t)kD, (uint64_t)a.hkv, (uint64_t)num_slots};
    if (!make_map(&prm.tm_q, q, 4, dq, 2, kBM) || !make_map(&prm.tm_k0, k_cache, 2, dp, 1, 1) ||
        !make_map(&prm.tm_v0, v_cache, 2, dp, 1, 1) || !make_map(&prm.tm_k1, k_cache, 3, d3, 2, kBN) ||
        !make_map(&prm.tm_v1, v_cache, 3, d3, 2, kBN) || (out && !make_map(&prm.tm_o, out, 4, dq, 2, kBM)))
        return ACACHE_ERR_CUDA;
    prm.read_slot = read_slot;
    prm.out = (bf16*)out;
    prm.dev_status = dev_status;
    prm.num_slots = num_slots;
    // chained: a later grid of a chain of layers, launched behind the previous layer's
    // attention; it reads only its own layer's pool, complete before the chain's first grid
    prm.early_wait = chained ? 0 : 1;
    prm.n_rows = n_q;
    prm.Hq = a.hq;
    prm.Hkv = a.hkv;
    prm.T_len = T_len;
    prm.scale_log2 = a.scale * kLog2e;
    prm.budget = wait_budget();
    if (drop_none) return launch_attn<kSlotKeys, true>(prm, B, stream, pdl || chained);
    if (out && tc_slot_persistent(a, B, n_q, T_len)) return launch_attn_persist(prm, B, stream, pdl || chained);
    return launch_attn<kSlotKeys>(prm, B, stream, pdl || chained);
}

int launch_tc_slot_attention_varlen(const AttnArgs& a, int B, const int32_t* q_start, int max_q,
                                    int total_q, const void* q, const int32_t* kv_start, int max_T,
                                    const int32_t* read_slot, const void* k_cache, const void* v_cache,
                                    int64_t num_slots, void* out, int32_t* dev_status,
                                    cudaStream_t stream, bool drop_none) {
    if ((int64_t)num_slots * a.hkv >= 0x7fffffffLL || total_q < 0) return ACACHE_ERR_INVALID_ARG;
    AttnParams prm{};
    const uint64_t dq[3] = {(uint64_t)kD, (uint64_t)a.hq, (uint64_t)(total_q > 0 ? total_q : 1)};
    const uint64_t dp[2] = {(uint64_t)kD, (uint64_t)num_slots * a.hkv};
    const uint64_t d3[3] = {(uint64_t)kD, (uint64_t)a.hkv, (uint64_t)num_slots};
    if (!make_map(&prm.tm_q, q, 3, dq, 2, kBM) || !make_map(&prm.tm_k0, k_cache, 2, dp, 1, 1) ||
        !make_map(&prm.tm_v0, v_cache, 2, dp, 1, 1) || !make_map(&prm.tm_k1, k_cache, 3, d3, 2, kBN) ||
        !make_map(&prm.tm_v1, v_cache, 3, d3, 2, kBN) || (out && !make_map(&prm.tm_o, out, 3, dq, 2, kBM)))
        return ACACHE_ERR_CUDA;
    prm.read_slot = read_slot;
    prm.q_start = q_start;
    prm.kv_start = kv_start;
    prm.out = (bf16*)out;
    prm.dev_status = dev_status;
    prm.num_slots = num_slots;
    prm.early_wait = 1;
    prm.n_rows = max_q;
    prm.Hq = a.hq;
    prm.Hkv = a.hkv;
    prm.T_len = max_T;
    prm.scale_log2 = a.scale * kLog2e;
    prm.budget = wait_budget();
    return drop_none ? launch_attn<kSlotKeys, true>(prm, B, stream) : launch_attn<kSlotKeys>(prm, B, stream);
}

int launch_tc_probe_pass_a(const AttnArgs& a, int B, int T_len, int l, int L, const void* q,
                           const void* k_req, const void* v_req, const void* k_aff,
                           const void* v_aff, void* out, float* stat_m, float* stat_l,
                           int32_t* dev_status, cudaStream_t stream, bool chained) {
    (void)l;   // key order inside a row does not change the softmax: affix tiles, then own tiles
    const int P = T_len - L;
    AttnParams prm{};
    const uint64_t dq[4] = {(uint64_t)kD, (uint64_t)a.hq, (uint64_t)P, (uint64_t)B};
    const uint64_t da[3] = {(uint64_t)kD, (uint64_t)a.hkv, (uint64_t)L};
    const uint64_t dr[4] = {(uint64_t)kD, (uint64_t)a.hkv, (uint64_t)P, (uint64_t)B};
    const void* ka = L > 0 ? k_aff : k_req;   // an unused map still needs a valid address
    const void* va = L > 0 ? v_aff : v_req;
    if (!make_map(&prm.tm_q, q, 4, dq, 2, kBM) || !make_map(&prm.tm_k0, ka, 3, da, 2, kBN) ||
        !make_map(&prm.tm_v0, va, 3, da, 2, kBN) || !make_map(&prm.tm_k1, k_req, 4, dr, 2, kBN) ||
        !make_map(&prm.tm_v1, v_req, 4, dr, 2, kBN) || (out && !make_map(&prm.tm_o, out, 4, dq, 2, kBM)))
        return ACACHE_ERR_CUDA;
    prm.out = (bf16*)out;
    prm.stat_m = stat_m;
    prm.stat_l = stat_l;
    prm.dev_status = dev_status;
    // chained: the probe of a later layer of one call, launched behind the previous layer's
    // head sum with programmatic dependent launch; it starts while the previous layer's mass
    // and head-sum grids finish, reads only its own layer's inputs (complete before the call's
    // first grid) and waits for them before it writes its output and row statistics.
    prm.early_wait = 2;
    prm.n_rows = P;
    prm.Hq = a.hq;
    prm.Hkv = a.hkv;
    prm.T_len = T_len;
    prm.L = L;
    prm.P = P;
    prm.scale_log2 = a.scale * kLog2e;
    prm.budget = wait_budget();
    return launch_attn<kProbeKeys>(prm, B, stream, chained);
}

int launch_tc_probe_pass_b(const AttnArgs& a, int B, int T_len, int L, const int32_t* masked_rows,
                           int m, const void* q, const void* k_aff, const float* stat_m,
                           const float* stat_l, float* partial, int32_t* dev_status,
                           cudaStream_t stream) {
    const int P = T_len - L;
    const int64_t ctas = (int64_t)B * a.hq * ((L + kBN - 1) / kBN);
    if (ctas == 0) return ACACHE_OK;
    if (m == 0) {   // no masked rows: every affix key receives zero mass
        if (cudaMemsetAsync(partial, 0, (size_t)B * a.hq * L * sizeof(float), stream) != cudaSuccess)
            return ACACHE_ERR_CUDA;
        return ACACHE_OK;
    }
    if ((int64_t)B * P * a.hq >= 0x7fffffffLL) return ACACHE_ERR_INVALID_ARG;
    ColsumParams prm{};
    const uint64_t da[3] = {(uint64_t)kD, (uint64_t)a.hkv, (uint64_t)L};
    const uint64_t dq[2] = {(uint64_t)kD, (uint64_t)B * P * a.hq};
    const uint64_t dqb[4] = {(uint64_t)kD, (uint64_t)a.hq, (uint64_t)P, (uint64_t)B};
    if (!make_map(&prm.tm_kaff, k_aff, 3, da, 2, kBN) || !make_map(&prm.tm_q, q, 2, dq, 1, 1) ||
        !make_map(&prm.tm_qbox, q, 4, dqb, 2, kBN))
        return ACACHE_ERR_CUDA;
    prm.masked = masked_rows;
    prm.stat_m = stat_m;
    prm.stat_l = stat_l;
    prm.partial = partial;
    prm.dev_status = dev_status;
    prm.B = B;
    prm.P = P;
    prm.L = L;
    prm.m = m;
    prm.Hq = a.hq;
    prm.Hkv = a.hkv;
    prm.scale_log2 = a.scale * kLog2e;
    prm.budget = wait_budget();
    if ((m + kBN - 1) / kBN <= kCrMaxChunks) {
        // masked rows resident: one CTA per (request, head) and run of affix tiles, the runs
        // as long as the SMs allow (one CTA per SM)
        const int n_jt = (L + kBN - 1) / kBN;
        const int64_t bh = (int64_t)B * a.hq;
        const int64_t fit = std::max<int64_t>(1, (int64_t)sm_count() / bh);
        const int per = (int)((n_jt + std::min<int64_t>(n_jt, fit) - 1) / std::min<int64_t>(n_jt, fit));
        const int64_t ctas_r = bh * ((n_jt + per - 1) / per);
        if (ctas_r > 0x7fffffff) return ACACHE_ERR_INVALID_ARG;
        if (cudaFuncSetAttribute(tc_colsum_rows_kernel, cudaFuncAttributeMaxDynamicSharedMemorySize,
                                 kCrSmemBytes) != cudaSuccess) {
            (void)cudaGetLastError();
            return ACACHE_ERR_CUDA;
        }
        return launch_pdl(tc_colsum_rows_kernel, (unsigned)ctas_r, kCrThreads, kCrSmemBytes, stream, prm, per);
    }
    if (cudaFuncSetAttribute(tc_colsum_kernel, cudaFuncAttributeMaxDynamicSharedMemorySize,
                             kCsSmemBytes) != cudaSuccess) {
        (void)cudaGetLastError();
        return ACACHE_ERR_CUDA;
    }
    return launch_pdl(tc_colsum_kernel, (unsigned)ctas, kCsThreads, kCsSmemBytes, stream, prm);
}

}  // namespace acache
