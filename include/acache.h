/*
 * acache.h -- C ABI of libacache.so, the GB300 (sm_103a) affix-cache attention path.
 *
 * The path follows the page "Affix Cache for Diffusion Large Language Models"
 * (arXiv 2608.26140):
 *   (1) anchor probe: the request's non-affix rows attend once over the shared
 *       precomputed affix K/V plus the request's own K/V (Sec. 3.2);
 *   (2) importance s_j: masked-to-affix attention mass summed over layers, heads and the
 *       initially masked rows (Sec. 3.2, Eq. 4-5);
 *   (3) anchors A = TopK({s_j}, K) (Sec. 3.2, Eq. 6);
 *   (4) store-then-attend: fresh anchor and request K/V are written to private slots and
 *       attention reads every logical position through a per-request read-slot map
 *       (Sec. 4.1, 4.3; App. C.1).
 *
 * Conventions for every call
 * --------------------------
 *  - Pointers are DEVICE pointers unless a comment says otherwise; the caller owns all
 *    memory.  The library never allocates device memory and creates no stream or event.
 *  - Every call is asynchronous on `stream` (a cudaStream_t passed as void*; NULL = the
 *    legacy default stream) and returns an acache_status synchronously.
 *  - Synchronous errors: ACACHE_ERR_INVALID_ARG (a required pointer is NULL or a scalar
 *    is out of range; nothing is launched), ACACHE_ERR_UNSUPPORTED (dtype / head_dim
 *    combination not built), ACACHE_ERR_CUDA (a launch failed; the CUDA error is cleared).
 *  - Asynchronous data errors: an index that would address memory outside its buffer is
 *    skipped (no access) and, when `dev_status` is non-NULL, the matching ACACHE_DEV_*
 *    bit is OR-ed into *dev_status.  Bounded waits that give up set ACACHE_DEV_TIMEOUT.
 *  - Layouts are row-major and contiguous: Q/O and fresh K/V are token-major
 *    [batch][rows][heads][head_dim]; a layer's KV pool is [num_slots][Hkv][head_dim]
 *    (K and V in separate pools, the caller passes each layer's base pointers).
 *  - Symbols: B batch, T logical length, F = [l, l+L) the affix span, P = T - L probe rows
 *    (non-affix positions in ascending logical order), m initially masked rows,
 *    K anchor budget, R = K + P recomputed rows, Hq / Hkv query / KV heads, d head dim.
 */
#ifndef ACACHE_H_
#define ACACHE_H_

#include <stddef.h>
#include <stdint.h>

#if defined(__GNUC__)
#define ACACHE_API __attribute__((visibility("default")))
#else
#define ACACHE_API
#endif

#ifdef __cplusplus
extern "C" {
#endif

typedef enum {
    ACACHE_OK = 0,
    ACACHE_ERR_INVALID_ARG = -1,
    ACACHE_ERR_UNSUPPORTED = -2,
    ACACHE_ERR_CUDA = -3,
    ACACHE_ERR_WORKSPACE = -4,
    ACACHE_ERR_TIMEOUT = -5
} acache_status;

typedef enum { ACACHE_F32 = 0, ACACHE_BF16 = 1 } acache_dtype;

/* bits OR-ed into *dev_status by kernels */
enum {
    ACACHE_DEV_BAD_SLOT = 1,      /* a slot index outside [0, num_slots)                  */
    ACACHE_DEV_SHARED_WRITE = 2,  /* a write slot below private_begin (shared region)     */
    ACACHE_DEV_BAD_ROW = 4,       /* a masked-row index outside [0, P)                     */
    ACACHE_DEV_BAD_ANCHOR = 8,    /* anchors not strictly ascending offsets in [0, L)      */
    ACACHE_DEV_NAN = 16,          /* a NaN importance score reached Top-K                  */
    ACACHE_DEV_TIMEOUT = 32,      /* a bounded wait inside a kernel gave up                */
    ACACHE_DEV_BAD_LENGTH = 64    /* a ragged-batch request length outside its bounds     */
};

/* Read-slot map entry of a logical position whose K/V was discarded (the page's DropNA
 * ablation, Sec. 5.3).  Only acache_slot_attention_dropna gives it that meaning; for every
 * other call it is an out-of-range slot like any other negative value. */
#define ACACHE_SLOT_NONE (-1)

/* Attention geometry shared by the attention calls. */
typedef struct {
    int32_t num_q_heads;    /* Hq                                                    */
    int32_t num_kv_heads;   /* Hkv, Hq % Hkv == 0; query head h reads KV head h/(Hq/Hkv) */
    int32_t head_dim;       /* d: 64 or 128.  The tensor-core kernels cover bf16 at 128;
                               float32 (either d) and bf16 at d = 64 run on CUDA cores
                               (same results and errors, far lower throughput)      */
    float scale;            /* softmax scale, normally 1/sqrt(d) (Eq. 4)             */
    int32_t dtype;          /* acache_dtype of Q, K, V and O                         */
} acache_attn_desc;

/* Human-readable name of a status code (host, static storage). */
ACACHE_API const char* acache_status_string(int status);
/* Library version: major*10000 + minor*100 + patch. */
ACACHE_API int acache_version(void);

/* ---------------------------------------------------------------------------------
 * Failure detection: the budget of the kernels' bounded waits (host, thread-safe).
 * Every wait of a tensor-core kernel's pipeline (a TMA load, an MMA, another role's hand-off)
 * gives up after `budget` SM clock cycles: the kernel then sets ACACHE_DEV_TIMEOUT in
 * dev_status, stops its work (its outputs are not written), lets the copies and MMAs it had
 * issued finish, releases its tensor memory and exits, so the context stays usable.  The
 * page has no counterpart: this is the library's own watchdog.
 * cycles > 0 sets the budget of kernels launched after the call; cycles <= 0 only reads it.
 * Returns the budget in force before the call (default 2^31 cycles, about 1 s at 2.07 GHz).
 * ------------------------------------------------------------------------------- */
ACACHE_API int64_t acache_wait_budget(int64_t cycles);

/* ---------------------------------------------------------------------------------
 * (1)+(2) Anchor probe of ONE layer and its importance contribution.
 * Page: Sec. 3.2, Eq. 4-5 ("one-shot probe over the current request's non-affix
 * positions while using the precomputed affix cache as fixed past KV states").
 *
 * For each request b, query head h and probe row k (P rows), the row attends over all T
 * logical keys: K_log[t] = k_affix[t-l] for t in F, else the request's own k_req row
 * (value rows likewise).  Softmax runs over the full row.  Then, for every initially
 * masked row k and affix offset j:  scores[b][j] += softmax_row_k[l + j], summed over
 * heads in ascending order.  Call layers 0..N-1 in order on one stream, after zeroing
 * `scores`; that fixes the accumulation order, so results are bit-reproducible
 * (acache_probe_scores_layers makes the same calls for every layer at once).
 *
 *   q            [B][P][Hq][d]   probe-row queries, rows in ascending logical order
 *   k_req, v_req [B][P][Hkv][d]  the request's own K/V rows (same order)
 *   k_affix, v_affix [L][Hkv][d] shared precomputed affix cache (one copy for all b)
 *   masked_rows  [B][m] int32    indices into the P probe rows; bad ones are skipped
 *                                and flagged ACACHE_DEV_BAD_ROW
 *   out          [B][P][Hq][d]   attention output of the probe rows, or NULL
 *   scores       [B][L] float    importance, ACCUMULATED in place
 *   workspace    >= acache_probe_workspace_bytes(...) bytes, 256-byte aligned; its
 *                contents need no initialisation and are clobbered
 * Returns ACACHE_ERR_WORKSPACE if the workspace is too small.
 * ------------------------------------------------------------------------------- */
ACACHE_API size_t acache_probe_workspace_bytes(const acache_attn_desc* a, int batch, int seq_len,
                                    int affix_len, int num_masked);
ACACHE_API int acache_probe_scores(const acache_attn_desc* a, int batch, int seq_len, int affix_begin,
                        int affix_len, const int32_t* masked_rows, int num_masked,
                        const void* q, const void* k_req, const void* v_req,
                        const void* k_affix, const void* v_affix, void* out, float* scores,
                        void* workspace, size_t workspace_bytes, int32_t* dev_status,
                        void* stream);

/* ---------------------------------------------------------------------------------
 * (1)+(2) Anchor probe of every layer in one call.  Page: Sec. 3.2, Eq. 4-5 (the probe runs
 * once per layer and the importance sums over layers).
 *
 * Computes exactly what acache_probe_scores(a, batch, ..., q[n], k_req[n], v_req[n],
 * k_affix[n], v_affix[n], out ? out[n] : NULL, scores, workspace, ...) does for n = 0, 1,
 * ..., layers-1 in that order on `stream`: the same kernels, the same accumulation order into
 * `scores`, so the result is bit-identical to those per-layer calls.  The shapes, batch,
 * masked rows, scores and workspace are shared by all layers; q, k_req, v_req, k_affix,
 * v_affix and out are host arrays of `layers` device pointers each (out may be NULL, and so
 * may an entry of it; k_affix/v_affix may be NULL when affix_len = 0).
 *
 * When nothing the call writes (any layer's out, scores, the workspace) overlaps any layer's
 * q/k_req/v_req/k_affix/v_affix (checked on the host), the grids of layer n > 0 are chained
 * behind layer n-1 with programmatic dependent launch (tensor-core path): layer n's probe
 * forward starts on the SMs that layer n-1's mass and head-sum grids leave idle, reading its
 * own layer's inputs at once and waiting for those grids before it writes anything.  Work
 * enqueued on the stream after the call runs after all of it.  The inputs must therefore be
 * complete before the call (as for any launch on the stream).  Otherwise -- or on the
 * CUDA-core path -- the layers run one after the other.  Every argument of every layer is
 * checked before anything is launched; errors as acache_probe_scores.
 * ------------------------------------------------------------------------------- */
ACACHE_API int acache_probe_scores_layers(const acache_attn_desc* a, int layers, int batch,
                        int seq_len, int affix_begin, int affix_len, const int32_t* masked_rows,
                        int num_masked, const void* const* q, const void* const* k_req,
                        const void* const* v_req, const void* const* k_affix,
                        const void* const* v_affix, void* const* out, float* scores,
                        void* workspace, size_t workspace_bytes, int32_t* dev_status,
                        void* stream);

/* ---------------------------------------------------------------------------------
 * Probe without a workspace.  The page has no counterpart: this entry point exists for
 * callers that cannot allocate device memory when they probe -- an engine that gives the
 * library only tensors it already owns (a memory budget split up at start-up, an allocator
 * the library cannot reach, or code that must not enter the CUDA allocator).
 *
 * Same computation, arguments, layouts and errors as acache_probe_scores, minus the
 * workspace: the scratch (row maximum and sum, per-head column sums) lives in one fixed
 * 16 MiB device array inside the library, reserved on every GPU that loads it until the
 * process exits.  A call needing more than that (2 * round256(B*Hq*P*4) +
 * round256(B*Hq*L*4) bytes) returns ACACHE_ERR_WORKSPACE and launches nothing.  The call
 * allocates nothing (no cudaMalloc/cudaFree, no allocating library routine).
 *  - Every call made while `stream` is not capturing looks up the array's device address on
 *    the current device (so the entry point keeps working after a device reset); a call made
 *    during stream capture reuses the address found by the device's last earlier call, so
 *    make the first call on each device before any stream capture starts.
 *  - All calls share the array and it keeps the last call's contents.  Nothing in it must
 *    start at zero (each call writes every scratch byte it reads), but calls whose kernels
 *    can overlap on the GPU (unordered streams) race on it: order them.
 * ------------------------------------------------------------------------------- */
ACACHE_API int acache_probe_scores_noalloc(const acache_attn_desc* a, int batch, int seq_len,
                        int affix_begin, int affix_len, const int32_t* masked_rows,
                        int num_masked, const void* q, const void* k_req, const void* v_req,
                        const void* k_affix, const void* v_affix, void* out, float* scores,
                        int32_t* dev_status, void* stream);

/* ---------------------------------------------------------------------------------
 * (3) Anchor selection.  Page: Sec. 3.2, Eq. 6, A = TopK({s_j}, K), S = F \ A.
 * anchors[b] receives the K affix offsets with the largest scores, ties broken toward the
 * lower offset, written in ascending offset order.  -0.0 counts as +0.0.  A NaN score
 * flags ACACHE_DEV_NAN (NaN ranks below every number).  0 <= K <= L.
 *   scores  [B][L] float, anchors [B][K] int32
 * ------------------------------------------------------------------------------- */
ACACHE_API int acache_topk_anchors(const float* scores, int batch, int affix_len, int k,
                        int32_t* anchors, int32_t* dev_status, void* stream);

/* ---------------------------------------------------------------------------------
 * Alternative selector: high KV deviation (CacheBlend-style), ONE layer.
 * Page: App. B.5 -- the variant keeps ACache's generation path and cache layout but ranks
 * affix tokens by the difference between the affix-only KV cache and the full-prompt KV
 * cache instead of by masked-to-affix attention.  Per request b and affix offset j:
 *   scores[b][j] += sum over KV heads hk (ascending) of
 *                   ||k_full[b][j][hk] - k_shared[j][hk]||_2 + ||v_full[b][j][hk] - v_shared[j][hk]||_2
 * (float32 sums of squares with a fixed reduction order: bit-reproducible).  Zero `scores`
 * before layer 0 and call the layers in order on one stream, then rank with
 * acache_topk_anchors exactly as for the probe's scores.
 *   k_shared, v_shared [L][Hkv][d]     the shared (affix-only) cache of the layer
 *   k_full, v_full     [B][L][Hkv][d]  the affix tokens' K/V computed inside each request
 *   scores             [B][L] float    ACCUMULATED in place
 * Pointers must be 16-byte aligned.  No device-side errors are possible.
 * ------------------------------------------------------------------------------- */
ACACHE_API int acache_kv_deviation_scores(const acache_attn_desc* a, int batch, int affix_len,
                        const void* k_shared, const void* v_shared, const void* k_full,
                        const void* v_full, float* scores, void* stream);

/* ---------------------------------------------------------------------------------
 * Admission-time maps.  Page: Sec. 4.1-4.2 (write-side recomputation map and per-request
 * read-slot map, recorded once at admission).
 * The R = K + P recomputed logical positions are the anchor positions l + A_b and every
 * non-affix position, in ascending order.
 *   write_pos[b][i] = the i-th recomputed logical position            [B][R] int32
 *   read_slot[b][t] = private_slots[b][i] if t is the i-th recomputed position,
 *                     shared_slot[t - l] otherwise (non-anchor affix)  [B][T] int32
 * The write-side slot of row i is private_slots[b][i] itself.
 *   anchors [B][K] (strictly ascending offsets in [0, L); otherwise that request's maps
 *   are left untouched and ACACHE_DEV_BAD_ANCHOR is flagged), shared_slot [L],
 *   private_slots [B][R].
 * ------------------------------------------------------------------------------- */
ACACHE_API int acache_build_slot_maps(int batch, int seq_len, int affix_begin, int affix_len, int k,
                           const int32_t* anchors, const int32_t* shared_slot,
                           const int32_t* private_slots, int32_t* write_pos,
                           int32_t* read_slot, int32_t* dev_status, void* stream);

/* ---------------------------------------------------------------------------------
 * (4a) Store step of one layer.  Page: Sec. 4.3 and App. C.1 (store-then-attend through
 * the write-side slot mapping).
 *   k_cache[write_slot[b][i]] = k_new[b][i] (all KV heads), same for V.
 * A slot outside [0, num_slots) is skipped (ACACHE_DEV_BAD_SLOT); a slot below
 * private_begin is skipped (ACACHE_DEV_SHARED_WRITE), which protects the shared region.
 * Pass private_begin = 0 to register a shared affix itself.
 *   write_slot [B][R] int32, k_new / v_new [B][R][Hkv][d], caches [num_slots][Hkv][d]
 * ------------------------------------------------------------------------------- */
ACACHE_API int acache_write_slots(const acache_attn_desc* a, int batch, int rows,
                       const int32_t* write_slot, const void* k_new, const void* v_new,
                       void* k_cache, void* v_cache, int64_t num_slots,
                       int64_t private_begin, int32_t* dev_status, void* stream);

/* ---------------------------------------------------------------------------------
 * (4a+4b) Store-then-attend of one layer in one call.  Page: Sec. 4.3 and App. C.1 (the
 * same store-then-attend interface at recompute points and in block decoding: write the
 * fresh K/V through the write-side map, then attend through the read-slot map).
 * Exactly acache_write_slots(rows, write_slot, k_new, v_new, ...) followed by
 * acache_slot_attention(n_q, q, seq_len, read_slot, ...) on the same pools, with the same
 * arguments, layouts and errors (every argument is checked before anything is launched).
 * On the tensor-core path the attention grid is launched with programmatic stream
 * serialisation: its set-up and query loads overlap the store, and it waits for the store
 * to complete before it reads any key or value row.  rows = 0 attends only; n_q = 0
 * stores only.
 * ------------------------------------------------------------------------------- */
ACACHE_API int acache_store_attend(const acache_attn_desc* a, int batch, int rows,
                        const int32_t* write_slot, const void* k_new, const void* v_new,
                        void* k_cache, void* v_cache, int64_t num_slots, int64_t private_begin,
                        int n_q, const void* q, int seq_len, const int32_t* read_slot, void* out,
                        int32_t* dev_status, void* stream);

/* ---------------------------------------------------------------------------------
 * (4b) Read-slot attention of one layer.  Page: Sec. 4.3 (queries only for recomputed
 * positions, keys and values read through the read-slot map) and App. C.1.
 * Each of the n_q dense query rows of request b attends bidirectionally over all T
 * logical keys K_log[t] = k_cache[read_slot[b][t]] (V likewise).
 *   q [B][n_q][Hq][d], read_slot [B][T] int32, caches [num_slots][Hkv][d],
 *   out [B][n_q][Hq][d].  A slot outside [0, num_slots) reads as a zero key and value
 *   row (no access) and flags ACACHE_DEV_BAD_SLOT.
 * ------------------------------------------------------------------------------- */
ACACHE_API int acache_slot_attention(const acache_attn_desc* a, int batch, int n_q, const void* q,
                          int seq_len, const int32_t* read_slot, const void* k_cache,
                          const void* v_cache, int64_t num_slots, void* out,
                          int32_t* dev_status, void* stream);

/* Which kernel acache_slot_attention (and the attention of acache_store_attend) runs for a
 * geometry (host only, no GPU call): ACACHE_PATH_RECOMPUTE -- the tcgen05 kernel of two
 * 128-row query tiles per CTA (a lone tile splits its keys between two chains);
 * ACACHE_PATH_RECOMPUTE_PERSISTENT -- the same computation in a persistent kernel (one CTA
 * per SM working through the 256-row query blocks, its rings running on from one block into
 * the next), chosen when there are more blocks than SMs and either at most 20 key tiles
 * (T <= 2560) or at most 128 query rows (one query tile per block);
 * ACACHE_PATH_BLOCK_DECODE -- the tcgen05 kernel for few query rows per KV head, chosen when
 * it streams fewer K/V tiles (a GQA group's heads share one stream) or, with as many, when
 * the streams would leave most SMs idle and its cluster split of the keys fills them;
 * ACACHE_PATH_CUDA_CORES --
 * float32 or bf16 at d = 64.  Returns a negative status for invalid arguments. */
enum {
    ACACHE_PATH_RECOMPUTE = 0,
    ACACHE_PATH_BLOCK_DECODE = 1,
    ACACHE_PATH_CUDA_CORES = 2,
    ACACHE_PATH_RECOMPUTE_PERSISTENT = 3
};
ACACHE_API int acache_slot_attention_path(const acache_attn_desc* a, int batch, int n_q, int seq_len);

/* ---------------------------------------------------------------------------------
 * (4a') Store-then-attend over the layers of one recompute point.  Page: Sec. 4.3 and
 * App. C.1 (each layer stores its recomputed rows, then attends through the read-slot map).
 * The computation of acache_store_attend for layer 0, 1, ..., layers-1 in that order on
 * the stream.  Per-layer buffers are passed as arrays of `layers` DEVICE pointers; the
 * arrays themselves are in HOST memory and are read during the call only:
 *   k_new, v_new   [layers] -> [B][rows][Hkv][d]      (ignored when rows = 0)
 *   k_cache, v_cache [layers] -> [num_slots][Hkv][d] (one pool per layer)
 *   q, out         [layers] -> [B][n_q][Hq][d]       (ignored when n_q = 0)
 * write_slot [B][rows] and read_slot [B][T] are shared by all layers.
 * When no layer's pools or output overlap any buffer of another layer (checked on the host),
 * the grids are chained with programmatic dependent launch: the stores of all layers run
 * back to back, then -- once they are complete -- the attentions (tensor-core path), each
 * starting on the SMs its predecessor's last wave leaves idle; work enqueued on the stream
 * after the call runs after all of them.  Otherwise -- or on the CUDA-core and
 * block-decode paths -- the layers run one after the other.  Every argument of every layer
 * is checked before anything is launched; errors as acache_store_attend.
 * ------------------------------------------------------------------------------- */
ACACHE_API int acache_store_attend_layers(const acache_attn_desc* a, int layers, int batch,
                        int rows, const int32_t* write_slot, const void* const* k_new,
                        const void* const* v_new, void* const* k_cache, void* const* v_cache,
                        int64_t num_slots, int64_t private_begin, int n_q, const void* const* q,
                        int seq_len, const int32_t* read_slot, void* const* out,
                        int32_t* dev_status, void* stream);

/* ---------------------------------------------------------------------------------
 * (4b') Read-slot attention with discarded keys -- the DropNA ablation.  Page: Sec. 5.3
 * (Figure 5) and App. B.4: the same anchors are recomputed, but every non-anchor affix
 * entry of the cache is discarded instead of read from the shared region.
 * Same arguments, layouts and errors as acache_slot_attention, except that a read-slot
 * entry equal to ACACHE_SLOT_NONE marks a logical position without K/V: that key takes no
 * part in the softmax (it is not a zero row) and raises no flag.  A query row whose keys
 * are all discarded outputs zeros.  A DropNA map is what acache_build_slot_maps writes when
 * every shared_slot entry is ACACHE_SLOT_NONE.
 * ------------------------------------------------------------------------------- */
ACACHE_API int acache_slot_attention_dropna(const acache_attn_desc* a, int batch, int n_q,
                          const void* q, int seq_len, const int32_t* read_slot,
                          const void* k_cache, const void* v_cache, int64_t num_slots, void* out,
                          int32_t* dev_status, void* stream);

/* ---------------------------------------------------------------------------------
 * (4b'') Read-slot attention over a ragged batch.  Page: App. C.1 (the prototype's kernel
 * takes ragged query and KV lengths besides the read-slot map) and Sec. 4.3.
 * The computation of acache_slot_attention, with per-request row counts:
 *   q_start  [B+1] int32 (device): request b's query rows are q_start[b] .. q_start[b+1]-1
 *            of q and out ([total_q_rows][Hq][d], total_q_rows = q_start[B])
 *   kv_start [B+1] int32 (device): request b's logical keys are the read-slot entries
 *            read_slot[kv_start[b] .. kv_start[b+1]-1] (one flattened int32 array)
 *   max_q_rows, max_seq_len (host): bounds on every request's row and key counts; the
 *            launch is sized by them.  total_q_rows (host) sizes the query tensor map.
 * A request with zero query rows is skipped.  A request whose counts are negative, above
 * the bounds, or that has rows but no key is skipped (its output rows are not written) and
 * flagged ACACHE_DEV_BAD_LENGTH.  drop_none != 0 gives ACACHE_SLOT_NONE the DropNA meaning
 * of acache_slot_attention_dropna.  Other errors as acache_slot_attention.
 * ------------------------------------------------------------------------------- */
ACACHE_API int acache_slot_attention_varlen(const acache_attn_desc* a, int batch,
                          const int32_t* q_start, int max_q_rows, int total_q_rows, const void* q,
                          const int32_t* kv_start, int max_seq_len, const int32_t* read_slot,
                          const void* k_cache, const void* v_cache, int64_t num_slots, void* out,
                          int drop_none, int32_t* dev_status, void* stream);

/* ---------------------------------------------------------------------------------
 * Logical KV view.  Page: Sec. 4.1 ("the same logical full-context KV view").
 * Materialises k_out[b][t] = k_cache[read_slot[b][t]] (V likewise), [B][T][Hkv][d].
 * Bad slots are skipped (the output row is left untouched) and flag ACACHE_DEV_BAD_SLOT.
 * ------------------------------------------------------------------------------- */
ACACHE_API int acache_gather_slots(const acache_attn_desc* a, int batch, int seq_len,
                        const int32_t* read_slot, const void* k_cache, const void* v_cache,
                        int64_t num_slots, void* k_out, void* v_out, int32_t* dev_status,
                        void* stream);

/* ---------------------------------------------------------------------------------
 * Position-aware affix registration.  Page: Sec. 4 (opening) and Limitations -- the cache
 * is kept after the rotary position rotation, so reusing a shared affix at another offset
 * needs its keys moved to the new positions.  Rotations compose: a key rotated for position
 * p becomes the key for position p + delta_pos after one more rotation by delta_pos x the
 * pair's frequency rope_theta^(-2i/d).  Values are unchanged.
 *   k_in, k_out [rows][Hkv][d] (may be the same buffer), 16-byte aligned
 *   interleaved = 0: pair i is (x_i, x_{i+d/2}) (rotate-half layout); 1: (x_{2i}, x_{2i+1})
 * cos/sin are computed on the host in double precision; the rotation runs in float32 and is
 * rounded once to the storage type.
 * ------------------------------------------------------------------------------- */
ACACHE_API int acache_rerotate_keys(const acache_attn_desc* a, int64_t rows, const void* k_in,
                        void* k_out, int32_t delta_pos, double rope_theta, int interleaved,
                        void* stream);

/* ---------------------------------------------------------------------------------
 * Admission runtime (host only; no device memory is touched).  Page: Sec. 4.1-4.2 -- the
 * shared region stores each common affix once and later compatible requests reuse it; each
 * request gets private slots for its anchors and its own positions; admission resolves the
 * affix and records the maps before the online loop.
 *
 * A pool describes the slot layout shared by every layer's KV pool: slots
 * [0, private_begin) are the shared region, [private_begin, num_slots) private pages of
 * page_slots slots (a partial last page is not used).  All functions are thread-safe.
 *   create:   *out receives the handle (ACACHE_ERR_WORKSPACE if host memory runs out).
 *   register_affix: the affix identified by the caller's 64-bit key (for instance a hash of
 *             its token ids and its offset) gets affix_len contiguous shared slots starting
 *             at *shared_base.  *created = 1 the first time: the caller then writes the
 *             affix's K/V there (acache_write_slots with private_begin = 0); later calls with
 *             the same key only add a reference (*created = 0).  A known key with another
 *             length is ACACHE_ERR_INVALID_ARG; a full shared region ACACHE_ERR_WORKSPACE.
 *   release_affix: drops one reference; the slots are free again at zero references.
 *   alloc_private: slots[0..rows) (host array) receives the private slots of a new request,
 *             page by page; *request_id identifies it.  ACACHE_ERR_WORKSPACE when pages run out.
 *   free_private: returns the request's pages.
 *   stats:    free shared / private slots, live affixes and requests (any pointer may be NULL).
 * ------------------------------------------------------------------------------- */
typedef struct acache_pool acache_pool;
ACACHE_API int acache_pool_create(int64_t num_slots, int64_t private_begin, int32_t page_slots,
                        acache_pool** out);
ACACHE_API void acache_pool_destroy(acache_pool* pool);
ACACHE_API int acache_pool_register_affix(acache_pool* pool, uint64_t key, int32_t affix_len,
                        int32_t* shared_base, int32_t* created);
ACACHE_API int acache_pool_release_affix(acache_pool* pool, uint64_t key);
ACACHE_API int acache_pool_alloc_private(acache_pool* pool, int32_t rows, int32_t* slots,
                        int64_t* request_id);
ACACHE_API int acache_pool_free_private(acache_pool* pool, int64_t request_id);
ACACHE_API int acache_pool_stats(acache_pool* pool, int64_t* free_shared_slots,
                        int64_t* free_private_slots, int32_t* n_affixes, int32_t* n_requests);

#ifdef __cplusplus
}
#endif
#endif /* ACACHE_H_ */
