/*
 * acache_ref.c -- plain, slow CPU oracle of the affix-cache attention path.
 *
 * TEST INFRASTRUCTURE ONLY.  Only the test suite, the smoke check and the benchmark's
 * CPU-baseline leg may load this library.  It shares no code, header, table or helper
 * with the CUDA library: it is written from the definitions on the page
 * "Affix Cache for Diffusion Large Language Models" (arXiv 2608.26140):
 *   - Sec. 3.2, Eq. 4: masked-to-affix attention weight a_{j,k} (softmax of Q K^T / sqrt(d_h));
 *   - Sec. 3.2, Eq. 5: importance s_j = sum over layers, heads and initially masked rows;
 *   - Sec. 3.2, Eq. 6: anchor set A = TopK({s_j}, K), S = F \ A;
 *   - Sec. 4.1: write-side recompute map and per-request read-slot map;
 *   - Sec. 4.3 and App. C.1: store-then-attend; attention reads every logical position
 *     through the read-slot map.
 *
 * Arithmetic is float64 throughout (bf16 / f32 inputs are widened exactly); every
 * sum is an explicit loop in a fixed order.  OpenMP only splits independent
 * (request, head) or (request) work items; all cross-item sums run serially in a
 * fixed order afterwards, so results do not depend on the thread count.
 *
 * Readings of points the page leaves open (each is a parameter or a documented choice):
 *   R1  Eq. 4 normalises over the full attention row (affix keys and the request's own
 *       keys); the literal affix-only normaliser is available as a flag.
 *   R2  Only initially masked rows (all generation positions at the first step) score.
 *   R3  With grouped KV heads, query head h reads KV head h / (Hq / Hkv); scores sum
 *       over all query heads.
 *   R4  Ties in Top-K go to the lower affix offset; anchors are emitted ascending.
 *   R5  Recomputed rows are ordered by ascending logical position (anchors interleaved
 *       with the request's own rows); the i-th one is written to private slot i.
 *   R6  The CacheBlend-style selector of App. B.5 ranks affix tokens by how far their K/V
 *       inside the full prompt moved from the affix-only cache; the measure taken is the
 *       L2 norm of the key difference plus that of the value difference, per KV head,
 *       summed over KV heads and layers.
 *   R8  Position-aware affix registration (Sec. 4 opening, Limitations): a cached key that
 *       carries the rotary rotation of position p is moved to p + delta by rotating every
 *       frequency pair i (frequency theta^(-2i/d)) by delta times that frequency.
 *   R7  DropNA (Sec. 5.3) throws away the cached K/V of every non-anchor affix position:
 *       such a position has no key at all -- it is left out of the softmax, not read as a
 *       zero row; a row left with no key outputs zeros.
 */
#include <math.h>
#include <stdint.h>
#include <stdlib.h>
#include <string.h>
#ifdef _OPENMP
#include <omp.h>
#endif

#define REF_F32 0
#define REF_BF16 1

int ref_version(void) { return 1; }

void ref_set_threads(int n) {
#ifdef _OPENMP
    if (n > 0) omp_set_num_threads(n);
#else
    (void)n;
#endif
}

int ref_get_threads(void) {
#ifdef _OPENMP
    return omp_get_max_threads();
#else
    return 1;
#endif
}

/* Widen element i of a bf16 or f32 array to double (exact for both). */
static double widen(const void* p, int dtype, int64_t i) {
    if (dtype == REF_F32) return (double)((const float*)p)[i];
    uint32_t bits = ((uint32_t)((const uint16_t*)p)[i]) << 16;
    float f;
    memcpy(&f, &bits, sizeof f);
    return (double)f;
}

static double dot_row(const void* a, int64_t a_off, const void* b, int64_t b_off, int d, int dtype) {
    double s = 0.0;
    for (int c = 0; c < d; ++c) s += widen(a, dtype, a_off + c) * widen(b, dtype, b_off + c);
    return s;
}

/*
 * Probe of one layer (Sec. 3.2): the P non-affix rows of each request attend over all T
 * logical keys, the shared affix keys K_F for t in F = [l, l+L) and the request's own
 * keys elsewhere.  Affix rows are not queries.
 *
 *   q      [B][P][Hq][d]      probe-row queries, rows in ascending logical order
 *   k_req  [B][P][Hkv][d]     the request's own keys / values (same row order)
 *   k_aff  [L][Hkv][d]        the shared precomputed affix cache
 *   masked [B][m]             indices into the probe rows of the initially masked set
 *   rows   [n_rows] or NULL   probe rows to evaluate (NULL = all P rows)
 *   out    [B][P][Hq][d]      attention output for evaluated rows (NULL = skip)
 *   scores [B][L]             ACCUMULATED: += sum over heads h (ascending) and evaluated
 *                             masked rows k (ascending) of a_{l+j, k}  (Eq. 4-5)
 *   row_max, row_sum [B][Hq][P] (NULL = skip): max_t s_kt and sum_t exp(s_kt - max)
 * Returns 0, or -1 for an invalid argument.
 */
int ref_probe_layer(int B, int T, int l, int L, int Hq, int Hkv, int d, double scale, int dtype,
                    const void* q, const void* k_req, const void* v_req,
                    const void* k_aff, const void* v_aff,
                    int m, const int32_t* masked, const int32_t* rows, int n_rows,
                    int affix_only_norm, double* out, double* scores,
                    double* row_max, double* row_sum) {
    const int P = T - L;
    if (B < 0 || l < 0 || L < 0 || l + L > T || Hq <= 0 || Hkv <= 0 || Hq % Hkv || d <= 0 || m < 0 || m > P)
        return -1;
    const int g = Hq / Hkv;
    if (!rows) n_rows = P;
    for (int b = 0; b < B; ++b)
        for (int i = 0; i < m; ++i)
            if (masked[(int64_t)b * m + i] < 0 || masked[(int64_t)b * m + i] >= P) return -1;
    for (int i = 0; rows && i < n_rows; ++i)
        if (rows[i] < 0 || rows[i] >= P) return -1;

    double* partial = NULL;
    if (scores && L > 0) {
        partial = (double*)calloc((size_t)B * Hq * L, sizeof(double));
        if (!partial) return -1;
    }
    const int64_t nitems = (int64_t)B * Hq;
#pragma omp parallel for schedule(dynamic, 1)
    for (int64_t item = 0; item < nitems; ++item) {
        const int b = (int)(item / Hq), h = (int)(item % Hq), hk = h / g;
        double* s = (double*)malloc(sizeof(double) * (T > 0 ? T : 1));
        char* is_masked = (char*)calloc(P > 0 ? P : 1, 1);
        for (int i = 0; i < m; ++i) is_masked[masked[(int64_t)b * m + i]] = 1;
        for (int ri = 0; ri < n_rows; ++ri) {
            const int p = rows ? rows[ri] : ri;
            const int64_t qoff = (((int64_t)b * P + p) * Hq + h) * d;
            /* logits over every logical key t */
            for (int t = 0; t < T; ++t) {
                int64_t koff;
                const void* kbase;
                if (t >= l && t < l + L) {
                    kbase = k_aff;
                    koff = ((int64_t)(t - l) * Hkv + hk) * d;
                } else {
                    const int pr = t < l ? t : t - L;
                    kbase = k_req;
                    koff = (((int64_t)b * P + pr) * Hkv + hk) * d;
                }
                s[t] = scale * dot_row(q, qoff, kbase, koff, d, dtype);
            }
            /* softmax over the full row (reading R1) */
            double mx = -INFINITY;
            for (int t = 0; t < T; ++t) mx = s[t] > mx ? s[t] : mx;
            double sum = 0.0;
            for (int t = 0; t < T; ++t) sum += exp(s[t] - mx);
            if (row_max) row_max[((int64_t)b * Hq + h) * P + p] = mx;
            if (row_sum) row_sum[((int64_t)b * Hq + h) * P + p] = sum;
            if (out) {
                double* o = out + qoff;
                for (int c = 0; c < d; ++c) o[c] = 0.0;
                for (int t = 0; t < T; ++t) {
                    const double pt = exp(s[t] - mx) / sum;
                    int64_t voff;
                    const void* vbase;
                    if (t >= l && t < l + L) {
                        vbase = v_aff;
                        voff = ((int64_t)(t - l) * Hkv + hk) * d;
                    } else {
                        const int pr = t < l ? t : t - L;
                        vbase = v_req;
                        voff = (((int64_t)b * P + pr) * Hkv + hk) * d;
                    }
                    for (int c = 0; c < d; ++c) o[c] += pt * widen(vbase, dtype, voff + c);
                }
            }
            /* Eq. 4-5: masked-to-affix mass */
            if (partial && is_masked[p]) {
                double* part = partial + item * L;
                if (!affix_only_norm) {
                    for (int j = 0; j < L; ++j) part[j] += exp(s[l + j] - mx) / sum;
                } else {
                    double amx = -INFINITY, asum = 0.0;
                    for (int j = 0; j < L; ++j) amx = s[l + j] > amx ? s[l + j] : amx;
                    for (int j = 0; j < L; ++j) asum += exp(s[l + j] - amx);
                    for (int j = 0; j < L; ++j) part[j] += exp(s[l + j] - amx) / asum;
                }
            }
        }
        free(s);
        free(is_masked);
    }
    if (partial) {
        for (int b = 0; b < B; ++b)
            for (int h = 0; h < Hq; ++h)
                for (int j = 0; j < L; ++j)
                    scores[(int64_t)b * L + j] += partial[((int64_t)b * Hq + h) * L + j];
        free(partial);
    }
    return 0;
}

/*
 * Top-K (Eq. 6): affix offset j is an anchor iff fewer than K offsets i beat it, where i
 * beats j when s_i > s_j, or s_i == s_j and i < j (reading R4).  Anchors are written in
 * ascending offset order.  Returns 0, -1 for bad sizes, -2 if a score is NaN.
 */
int ref_topk(int B, int L, int K, const double* scores, int32_t* anchors) {
    if (B < 0 || L < 0 || K < 0 || K > L) return -1;
    int bad = 0;
#pragma omp parallel for schedule(dynamic, 1) reduction(| : bad)
    for (int b = 0; b < B; ++b) {
        const double* s = scores + (int64_t)b * L;
        int n = 0;
        for (int j = 0; j < L; ++j) {
            if (s[j] != s[j]) { bad |= 1; continue; }
            int beaten_by = 0;
            for (int i = 0; i < L && beaten_by < K; ++i)
                if (s[i] > s[j] || (s[i] == s[j] && i < j)) ++beaten_by;
            if (beaten_by < K) anchors[(int64_t)b * K + n++] = j;
        }
        if (n != K) bad |= 1;
    }
    return bad ? -2 : 0;
}

/*
 * Admission-time maps (Sec. 4.1-4.2).  The recomputed logical positions are the anchor
 * positions l + A_b together with every non-affix position, in ascending order
 * (reading R5); there are R = K + (T - L) of them.
 *   write_pos[b][i]  = the i-th recomputed logical position
 *   read_slot[b][t]  = private_slots[b][i] if t is the i-th recomputed position,
 *                      shared_slot[t - l]  otherwise (a non-anchor affix position)
 * anchors [B][K] must be strictly ascending offsets in [0, L).  Returns 0 or -1.
 */
int ref_build_slot_maps(int B, int T, int l, int L, int K, const int32_t* anchors,
                        const int32_t* shared_slot, const int32_t* private_slots,
                        int32_t* write_pos, int32_t* read_slot) {
    if (B < 0 || l < 0 || L < 0 || l + L > T || K < 0 || K > L) return -1;
    const int R = K + (T - L);
    char* is_anchor = (char*)calloc(L > 0 ? L : 1, 1);
    int rc = 0;
    for (int b = 0; b < B && rc == 0; ++b) {
        memset(is_anchor, 0, L > 0 ? L : 1);
        for (int i = 0; i < K; ++i) {
            const int a = anchors[(int64_t)b * K + i];
            if (a < 0 || a >= L || (i > 0 && a <= anchors[(int64_t)b * K + i - 1])) { rc = -1; break; }
            is_anchor[a] = 1;
        }
        if (rc) break;
        int i = 0;
        for (int t = 0; t < T; ++t) {
            const int in_affix = t >= l && t < l + L;
            if (!in_affix || is_anchor[t - l]) {
                write_pos[(int64_t)b * R + i] = t;
                read_slot[(int64_t)b * T + t] = private_slots[(int64_t)b * R + i];
                ++i;
            } else {
                read_slot[(int64_t)b * T + t] = shared_slot[t - l];
            }
        }
    }
    free(is_anchor);
    return rc;
}

/*
 * Store step (Sec. 4.3, write-side recompute map): row i of the fresh K/V of request b
 * goes to physical slot write_slot[b][i] of the layer's pool, all KV heads at once.
 * Rows whose slot is outside [private_begin, num_slots) are skipped.
 * Returns a bitmask: 1 = slot out of range, 2 = slot inside the shared region.
 */
int ref_write_slots(int B, int R, int Hkv, int d, int esize, const int32_t* write_slot,
                    const void* k_new, const void* v_new, void* k_cache, void* v_cache,
                    int64_t num_slots, int64_t private_begin) {
    const int64_t row_bytes = (int64_t)Hkv * d * esize;
    int flags = 0;
    for (int b = 0; b < B; ++b)
        for (int i = 0; i < R; ++i) {
            const int64_t slot = write_slot[(int64_t)b * R + i];
            if (slot < 0 || slot >= num_slots) { flags |= 1; continue; }
            if (slot < private_begin) { flags |= 2; continue; }
            const int64_t src = ((int64_t)b * R + i) * row_bytes;
            for (int64_t x = 0; x < row_bytes; ++x) {
                ((char*)k_cache)[slot * row_bytes + x] = ((const char*)k_new)[src + x];
                ((char*)v_cache)[slot * row_bytes + x] = ((const char*)v_new)[src + x];
            }
        }
    return flags;
}

/*
 * Logical KV view (Sec. 4.1): k_out[b][t] = k_cache[read_slot[b][t]], same for V.
 * Returns 0, or 1 if a slot is out of range (that row is left untouched).
 */
int ref_gather_slots(int B, int T, int Hkv, int d, int esize, const int32_t* read_slot,
                     const void* k_cache, const void* v_cache, int64_t num_slots,
                     void* k_out, void* v_out) {
    const int64_t row_bytes = (int64_t)Hkv * d * esize;
    int flags = 0;
    for (int b = 0; b < B; ++b)
        for (int t = 0; t < T; ++t) {
            const int64_t slot = read_slot[(int64_t)b * T + t];
            if (slot < 0 || slot >= num_slots) { flags |= 1; continue; }
            const int64_t dst = ((int64_t)b * T + t) * row_bytes;
            for (int64_t x = 0; x < row_bytes; ++x) {
                ((char*)k_out)[dst + x] = ((const char*)k_cache)[slot * row_bytes + x];
                ((char*)v_out)[dst + x] = ((const char*)v_cache)[slot * row_bytes + x];
            }
        }
    return flags;
}

/*
 * Read-slot attention (Sec. 4.3, App. C.1): each of the nq query rows of request b attends,
 * bidirectionally, over all T logical keys K_log[t] = k_cache[read_slot[b][t]].
 *   q   [B][nq][Hq][d], caches [num_slots][Hkv][d], out [B][nq][Hq][d] (double)
 *   rows [n_rows] or NULL: query rows to evaluate (same subset for every request)
 *   drop_none: an entry equal to -1 is a discarded logical position (reading R7)
 * Returns 0, or -1 for a slot out of range.
 */
int ref_slot_attention(int B, int nq, int T, int Hq, int Hkv, int d, double scale, int dtype,
                       const void* q, const int32_t* read_slot, const void* k_cache,
                       const void* v_cache, int64_t num_slots, const int32_t* rows, int n_rows,
                       int drop_none, double* out) {
    if (Hq <= 0 || Hkv <= 0 || Hq % Hkv) return -1;
    for (int64_t x = 0; x < (int64_t)B * T; ++x)
        if ((read_slot[x] < 0 || read_slot[x] >= num_slots) && !(drop_none && read_slot[x] == -1)) return -1;
    const int g = Hq / Hkv;
    if (!rows) n_rows = nq;
    const int64_t nitems = (int64_t)B * Hq;
#pragma omp parallel for schedule(dynamic, 1)
    for (int64_t item = 0; item < nitems; ++item) {
        const int b = (int)(item / Hq), h = (int)(item % Hq), hk = h / g;
        double* s = (double*)malloc(sizeof(double) * (T > 0 ? T : 1));
        for (int ri = 0; ri < n_rows; ++ri) {
            const int i = rows ? rows[ri] : ri;
            const int64_t qoff = (((int64_t)b * nq + i) * Hq + h) * d;
            double mx = -INFINITY;
            int kept = 0;
            for (int t = 0; t < T; ++t) {
                const int64_t slot = read_slot[(int64_t)b * T + t];
                if (slot < 0) continue;                       /* discarded (R7) */
                s[t] = scale * dot_row(q, qoff, k_cache, (slot * Hkv + hk) * d, d, dtype);
                mx = s[t] > mx ? s[t] : mx;
                ++kept;
            }
            double sum = 0.0;
            for (int t = 0; t < T; ++t)
                if (read_slot[(int64_t)b * T + t] >= 0) sum += exp(s[t] - mx);
            double* o = out + qoff;
            for (int c = 0; c < d; ++c) o[c] = 0.0;
            for (int t = 0; kept > 0 && t < T; ++t) {
                const int64_t slot = read_slot[(int64_t)b * T + t];
                if (slot < 0) continue;
                const double pt = exp(s[t] - mx) / sum;
                for (int c = 0; c < d; ++c) o[c] += pt * widen(v_cache, dtype, (slot * Hkv + hk) * d + c);
            }
        }
        free(s);
    }
    return 0;
}

/*
 * Plain dense attention over an already materialised logical K/V [B][T][Hkv][d].  A second,
 * separately written path: logits are exponentiated against the row maximum and the
 * output is normalised once at the end.  Used to check that slot-mapped attention equals
 * attention over the gathered logical KV.
 */
int ref_dense_attention(int B, int nq, int T, int Hq, int Hkv, int d, double scale, int dtype,
                        const void* q, const void* k, const void* v, double* out) {
    if (Hq <= 0 || Hkv <= 0 || Hq % Hkv) return -1;
    const int g = Hq / Hkv;
#pragma omp parallel for schedule(dynamic, 1)
    for (int64_t item = 0; item < (int64_t)B * nq; ++item) {
        const int b = (int)(item / nq), i = (int)(item % nq);
        double* w = (double*)malloc(sizeof(double) * (T > 0 ? T : 1));
        for (int h = 0; h < Hq; ++h) {
            const int hk = h / g;
            const int64_t qoff = (((int64_t)b * nq + i) * Hq + h) * d;
            for (int t = 0; t < T; ++t)
                w[t] = dot_row(q, qoff, k, (((int64_t)b * T + t) * Hkv + hk) * d, d, dtype) * scale;
            double mx = -INFINITY;
            for (int t = 0; t < T; ++t) if (w[t] > mx) mx = w[t];
            double denom = 0.0;
            for (int t = 0; t < T; ++t) { w[t] = exp(w[t] - mx); denom += w[t]; }
            for (int c = 0; c < d; ++c) {
                double acc = 0.0;
                for (int t = 0; t < T; ++t)
                    acc += w[t] * widen(v, dtype, (((int64_t)b * T + t) * Hkv + hk) * d + c);
                out[qoff + c] = acc / denom;
            }
        }
        free(w);
    }
    return 0;
}

/*
 * High-KV-deviation selector of one layer (App. B.5, reading R6): for every request b and
 * affix offset j,
 *   scores[b][j] += sum_hk ( ||k_full[b][j][hk] - k_sh[j][hk]|| + ||v_full[b][j][hk] - v_sh[j][hk]|| )
 *   k_sh, v_sh [L][Hkv][d]; k_full, v_full [B][L][Hkv][d]; scores [B][L] (double, accumulated)
 */
int ref_kv_deviation(int B, int L, int Hkv, int d, int dtype, const void* k_sh, const void* v_sh,
                     const void* k_full, const void* v_full, double* scores) {
    if (B < 0 || L < 0 || Hkv <= 0 || d <= 0) return -1;
    for (int b = 0; b < B; ++b)
        for (int j = 0; j < L; ++j) {
            double dev = 0.0;
            for (int hk = 0; hk < Hkv; ++hk) {
                const int64_t so = ((int64_t)j * Hkv + hk) * d;
                const int64_t fo = (((int64_t)b * L + j) * Hkv + hk) * d;
                double sk = 0.0, sv = 0.0;
                for (int c = 0; c < d; ++c) {
                    const double dk = widen(k_full, dtype, fo + c) - widen(k_sh, dtype, so + c);
                    const double dv = widen(v_full, dtype, fo + c) - widen(v_sh, dtype, so + c);
                    sk += dk * dk;
                    sv += dv * dv;
                }
                dev += sqrt(sk) + sqrt(sv);
            }
            scores[(int64_t)b * L + j] += dev;
        }
    return 0;
}

/*
 * Re-rotation of rotary-embedded keys (reading R8).  k [rows][Hkv][d] -> out (double).
 * Pair i is (x_i, x_{i + d/2}) when interleaved == 0, (x_{2i}, x_{2i+1}) otherwise; the pair
 * (a, b) becomes (a cos w - b sin w, a sin w + b cos w) with w = delta * theta^(-2i/d).
 */
int ref_rerotate(int64_t rows, int Hkv, int d, int dtype, const void* k, int delta, double theta,
                 int interleaved, double* out) {
    if (rows < 0 || Hkv <= 0 || d <= 0 || d % 2 || !(theta > 0.0)) return -1;
    for (int64_t r = 0; r < rows * Hkv; ++r) {
        const int64_t off = r * d;
        for (int i = 0; i < d / 2; ++i) {
            const int ia = interleaved ? 2 * i : i;
            const int ib = interleaved ? 2 * i + 1 : i + d / 2;
            const double w = (double)delta * pow(theta, -2.0 * (double)i / (double)d);
            const double a = widen(k, dtype, off + ia), b = widen(k, dtype, off + ib);
            out[off + ia] = a * cos(w) - b * sin(w);
            out[off + ib] = a * sin(w) + b * cos(w);
        }
    }
    return 0;
}
