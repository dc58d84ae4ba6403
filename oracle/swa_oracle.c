/*
 * swa_oracle.c -- plain, slow, obviously-correct CPU oracle for sliding-window
 * attention, in fp64.
 *
 * TEST INFRASTRUCTURE ONLY.  Only the test suite, the smoke check and the
 * benchmark's CPU-baseline leg may load this library.  It shares no code with
 * the CUDA path and the product never calls it.
 *
 * What it computes (one query row at a time, no blocking, no fusion):
 *
 *   1. The explicit mask row over every key position s in [0, T):
 *        in_band(t, s) = (wl < 0 or s >= t - wl) and (wr < 0 or s <= t + wr)
 *        allowed(t, s) = in_band(t, s) or t in G or s in G
 *      The causal window of W keys (Sliding Window Attention, lizeman.github.io
 *      llm-arch-kb, section 2 "Derivation": N_t = [max(0, t-W+1), t], and the
 *      banded mask of section 3) is wl = W-1, wr = 0.  The bidirectional
 *      Longformer window (prathamp.com "Sliding Window Attention: From Local
 *      Windows to Global Context", section 1.1: S_i = {j : |i-j| <= r} clipped to
 *      [0, n-1]) is wl = wr = r.  Asymmetric windows (mbrenndoerfer.com "How
 *      Sliding Window Attention Works", window configurations) are any other
 *      pair.  Global positions follow the same Longformer page, section 4.3:
 *      a global row sees all n keys, every row sees each global key, and a key
 *      already in the window is not counted twice.
 *   2. count_t = number of allowed keys.
 *   3. x_s = scale * sum_d q[t,d] k[s,d] for allowed s (the scaled dot product
 *      of the Derivation section; the additive -inf mask of the mbrenndoerfer
 *      page is realised as exclusion from the set).
 *   4. m = max x, l = sum exp(x - m), o = sum exp(x - m) v_s / l,
 *      lse = m + ln l.  An empty row gives o = 0, lse = -inf, count 0.
 *
 * Variants of step 1 (swa_oracle_mask_row_ex / swa_oracle_fwd_ex):
 *   - Dilation (Longformer page, section 3.1: S_i = {i + k*d : k in [-r, r]},
 *     clipped; lizeman page, "Dilation"): with dilation d the band is
 *     {t + k*d : -wl <= k <= wr} -- wl and wr count steps of d -- clipped to
 *     [0, T).  Every query head may have its own d (Longformer page, 3.6).
 *   - Global mode 1, attention sinks (lizeman page, failure mode 1; StreamingLLM
 *     as cited there): the listed positions are pinned key columns -- every row
 *     sees them as long as they are not right of its band's right edge (for a
 *     causal window: not in its future) -- and their rows are ordinary rows.
 *   - Separate global projections (Longformer page, section 5.2): a global row
 *     uses Q_g for its query and K_g, V_g for every key; a local row uses Q for
 *     its query, K_g, V_g for the keys of global positions and K, V for the rest.
 *
 * Decode (ring-buffer cache): the cache of S slots holds, per slot j, the true
 * token position slot_pos[b][j] (Gemma 3 sliding-window note, ai-engineer-
 * exhaustive.pages.dev: positions are stored in the cache and the window is
 * computed from them).  Slot j is allowed for the query at t = q_pos[b] iff
 * 0 <= p <= t and (t - W < p or p < n_sink): the window of W positions plus the
 * first n_sink positions pinned as sinks.  The rest is steps 2-4.
 *
 * Ring append (lizeman page, KV cache paragraph, quoting Mistral 7B section 2):
 * token p is stored in slot p mod S, overwriting what was there.  A cache that
 * pins n_sink sinks keeps position p < n_sink in slot p and rings the rest through
 * the other S - n_sink slots: slot n_sink + (p - n_sink) mod (S - n_sink).  Chunked
 * prefill: C new tokens at positions p0 .. p0+C-1 attend to the cached history
 * (slots holding positions below p0) and to the chunk itself, under the decode
 * rule above.
 *
 * Inputs are bf16 bit patterns (uint16) widened exactly to fp64; outputs are
 * fp64.  Grouped-query attention maps query head h to key/value head
 * h / (Hq / Hkv) (contiguous groups).  Rows are independent; OpenMP spreads
 * them over host threads.
 */
#include <math.h>
#include <stdint.h>
#include <stdlib.h>
#include <string.h>
#ifdef _OPENMP
#include <omp.h>
#endif

static double widen_bf16(uint16_t h) {
    uint32_t u = (uint32_t)h << 16;
    float f;
    memcpy(&f, &u, sizeof f);
    return (double)f;
}

static int is_member(const int32_t *set, int64_t n, int64_t x) {
    for (int64_t i = 0; i < n; ++i)
        if (set[i] == x) return 1;
    return 0;
}

/*
 * Step 1: the explicit mask row of query t over keys [0, T), with band dilation
 * dil >= 1 and global mode gmode (0: global rows and columns, 1: sink columns).
 */
void swa_oracle_mask_row_ex(int64_t T, int64_t t, int32_t wl, int32_t wr, int32_t dil, const int32_t *G,
                            int64_t nG, int32_t gmode, uint8_t *allowed) {
    const int row_is_global = gmode == 0 && is_member(G, nG, t);
    for (int64_t s = 0; s < T; ++s) {
        const int64_t off = s - t; /* s = t + k * dil */
        const int on_grid = off % dil == 0;
        const int64_t k = off / dil;
        const int in_band = on_grid && (wl < 0 || k >= -wl) && (wr < 0 || k <= wr);
        int column = is_member(G, nG, s);
        if (gmode == 1) column = column && (wr < 0 || off <= (int64_t)wr * dil);
        allowed[s] = (uint8_t)(in_band || row_is_global || column);
    }
}

void swa_oracle_mask_row(int64_t T, int64_t t, int32_t wl, int32_t wr, const int32_t *G, int64_t nG,
                         uint8_t *allowed) {
    swa_oracle_mask_row_ex(T, t, wl, wr, 1, G, nG, 0, allowed);
}

/* Steps 3-4 over the n allowed keys whose rows are krow[i] / vrow[i]. */
static void attend(const double *q, int64_t D, double scale, const uint16_t *const *krow,
                   const uint16_t *const *vrow, int64_t n, double *x, double *o, double *lse) {
    for (int64_t c = 0; c < D; ++c) o[c] = 0.0;
    if (n == 0) {
        *lse = -INFINITY;
        return;
    }
    double m = -INFINITY;
    for (int64_t i = 0; i < n; ++i) {
        double dot = 0.0;
        for (int64_t c = 0; c < D; ++c) dot += q[c] * widen_bf16(krow[i][c]);
        x[i] = scale * dot;
        if (x[i] > m) m = x[i];
    }
    double l = 0.0;
    for (int64_t i = 0; i < n; ++i) {
        const double p = exp(x[i] - m);
        l += p;
        for (int64_t c = 0; c < D; ++c) o[c] += p * widen_bf16(vrow[i][c]);
    }
    for (int64_t c = 0; c < D; ++c) o[c] /= l;
    *lse = m + log(l);
}

/*
 * Prefill / encoder.  q: [B,T,Hq,D], k and v: [B,T,Hkv,D], all contiguous bf16 bits.
 * qg, kg, vg: the separate global projections (same shapes as q, k, v), or all
 * NULL; only with gmode 0.  dil: per-query-head dilation [Hq] (each >= 1) or NULL
 * for 1.  rows: nrows (b, h, t) triples to evaluate, or NULL for every row in
 * (b, h, t) order (nrows must then be B*Hq*T).  Outputs per evaluated row i:
 * o[i*D ..], lse[i], counts[i] (counts may be NULL).  Returns 0, or -1 on a bad
 * argument.
 */
int swa_oracle_fwd_ex(const uint16_t *q, const uint16_t *k, const uint16_t *v, const uint16_t *qg,
                      const uint16_t *kg, const uint16_t *vg, int64_t B, int64_t T, int64_t Hq, int64_t Hkv,
                      int64_t D, int32_t wl, int32_t wr, const int32_t *dil, double scale, const int32_t *G,
                      int64_t nG, int32_t gmode, const int64_t *rows, int64_t nrows, double *o, double *lse,
                      int64_t *counts) {
    if (B < 0 || T < 0 || Hq <= 0 || Hkv <= 0 || D <= 0 || Hq % Hkv != 0 || nrows < 0) return -1;
    if (rows == NULL && nrows != B * Hq * T) return -1;
    if (gmode != 0 && gmode != 1) return -1;
    const int separate = qg != NULL;
    if (separate && (kg == NULL || vg == NULL || gmode != 0)) return -1;
    if (dil)
        for (int64_t h = 0; h < Hq; ++h)
            if (dil[h] < 1) return -1;
    const int64_t group = Hq / Hkv;
    int bad = 0;
#pragma omp parallel
    {
        uint8_t *allowed = (uint8_t *)malloc((size_t)(T > 0 ? T : 1));
        double *x = (double *)malloc(sizeof(double) * (size_t)(T > 0 ? T : 1));
        double *qd = (double *)malloc(sizeof(double) * (size_t)D);
        const uint16_t **krow = (const uint16_t **)malloc(sizeof(void *) * (size_t)(T > 0 ? T : 1));
        const uint16_t **vrow = (const uint16_t **)malloc(sizeof(void *) * (size_t)(T > 0 ? T : 1));
#pragma omp for schedule(dynamic, 8)
        for (int64_t i = 0; i < nrows; ++i) {
            int64_t b, h, t;
            if (rows) {
                b = rows[3 * i];
                h = rows[3 * i + 1];
                t = rows[3 * i + 2];
            } else {
                b = i / (Hq * T);
                h = (i / T) % Hq;
                t = i % T;
            }
            if (b < 0 || b >= B || h < 0 || h >= Hq || t < 0 || t >= T) {
#pragma omp atomic write
                bad = 1;
                continue;
            }
            const int64_t kvh = h / group;
            swa_oracle_mask_row_ex(T, t, wl, wr, dil ? dil[h] : 1, G, nG, gmode, allowed);
            const int row_global = separate && is_member(G, nG, t);
            int64_t n = 0;
            for (int64_t s = 0; s < T; ++s) {
                if (!allowed[s]) continue;
                /* which projection supplies this key and value (section 5.2) */
                const int from_global = separate && (row_global || is_member(G, nG, s));
                const int64_t kv_off = ((b * T + s) * Hkv + kvh) * D;
                krow[n] = (from_global ? kg : k) + kv_off;
                vrow[n] = (from_global ? vg : v) + kv_off;
                ++n;
            }
            const uint16_t *qrow = (row_global ? qg : q) + ((b * T + t) * Hq + h) * D;
            for (int64_t c = 0; c < D; ++c) qd[c] = widen_bf16(qrow[c]);
            attend(qd, D, scale, krow, vrow, n, x, o + i * D, lse + i);
            if (counts) counts[i] = n;
        }
        free(allowed);
        free(x);
        free(qd);
        free(krow);
        free(vrow);
    }
    return bad ? -1 : 0;
}

int swa_oracle_fwd(const uint16_t *q, const uint16_t *k, const uint16_t *v, int64_t B, int64_t T, int64_t Hq,
                   int64_t Hkv, int64_t D, int32_t wl, int32_t wr, double scale, const int32_t *G, int64_t nG,
                   const int64_t *rows, int64_t nrows, double *o, double *lse, int64_t *counts) {
    return swa_oracle_fwd_ex(q, k, v, NULL, NULL, NULL, B, T, Hq, Hkv, D, wl, wr, NULL, scale, G, nG, 0, rows,
                             nrows, o, lse, counts);
}

/* Slot rule of decode and chunked prefill: position p is attended from t. */
static int slot_allowed(int64_t p, int64_t t, int64_t W, int64_t n_sink) {
    return p >= 0 && p <= t && (p > t - W || p < n_sink);
}

/*
 * Ring-buffer decode.  q: [B,Hq,D]; k_cache, v_cache: [B,Hkv,S,D]; slot_pos: [B,S];
 * q_pos: [B]; W: the window (positions); n_sink: pinned first positions (0: none).
 * Outputs o: [B,Hq,D], lse: [B,Hq], counts: [B,Hq] (may be NULL).
 */
int swa_oracle_decode_ex(const uint16_t *q, const uint16_t *kc, const uint16_t *vc, const int32_t *slot_pos,
                         const int32_t *q_pos, int64_t B, int64_t Hq, int64_t Hkv, int64_t D, int64_t S, int64_t W,
                         int64_t n_sink, double scale, double *o, double *lse, int64_t *counts) {
    if (B < 0 || Hq <= 0 || Hkv <= 0 || D <= 0 || S <= 0 || W <= 0 || n_sink < 0 || Hq % Hkv != 0) return -1;
    const int64_t group = Hq / Hkv;
#pragma omp parallel
    {
        double *x = (double *)malloc(sizeof(double) * (size_t)S);
        double *qd = (double *)malloc(sizeof(double) * (size_t)D);
        const uint16_t **krow = (const uint16_t **)malloc(sizeof(void *) * (size_t)S);
        const uint16_t **vrow = (const uint16_t **)malloc(sizeof(void *) * (size_t)S);
#pragma omp for schedule(dynamic, 4)
        for (int64_t i = 0; i < B * Hq; ++i) {
            const int64_t b = i / Hq, h = i % Hq, kvh = h / group;
            const int64_t t = q_pos[b];
            int64_t n = 0;
            for (int64_t j = 0; j < S; ++j) {
                if (slot_allowed(slot_pos[b * S + j], t, W, n_sink)) {
                    krow[n] = kc + ((b * Hkv + kvh) * S + j) * D;
                    vrow[n] = vc + ((b * Hkv + kvh) * S + j) * D;
                    ++n;
                }
            }
            const uint16_t *qrow = q + (b * Hq + h) * D;
            for (int64_t c = 0; c < D; ++c) qd[c] = widen_bf16(qrow[c]);
            attend(qd, D, scale, krow, vrow, n, x, o + i * D, lse + i);
            if (counts) counts[i] = n;
        }
        free(x);
        free(qd);
        free(krow);
        free(vrow);
    }
    return 0;
}

int swa_oracle_decode(const uint16_t *q, const uint16_t *kc, const uint16_t *vc, const int32_t *slot_pos,
                      const int32_t *q_pos, int64_t B, int64_t Hq, int64_t Hkv, int64_t D, int64_t W, double scale,
                      double *o, double *lse, int64_t *counts) {
    return swa_oracle_decode_ex(q, kc, vc, slot_pos, q_pos, B, Hq, Hkv, D, W, W, 0, scale, o, lse, counts);
}

/*
 * Ring append.  Token i (0 <= i < n) of sequence b has position p = p0[b] + i; in
 * order of i its key and value rows (k_new, v_new: [B,n,Hkv,D]) are written to slot
 * j(p) of every kv head of the caches ([B,Hkv,S,D]) and slot_pos[b][j(p)] = p, with
 * j(p) = p for a sink (p < n_sink) and n_sink + (p - n_sink) mod (S - n_sink) else.
 * Returns -1 on a bad argument (a negative position, no ring slot).
 */
int swa_oracle_cache_append_ex(uint16_t *kc, uint16_t *vc, int32_t *slot_pos, int64_t B, int64_t Hkv, int64_t S,
                               int64_t D, int64_t n_sink, const uint16_t *k_new, const uint16_t *v_new, int64_t n,
                               const int32_t *p0) {
    if (B < 0 || Hkv <= 0 || S <= 0 || D <= 0 || n < 0 || n_sink < 0 || n_sink >= S) return -1;
    for (int64_t b = 0; b < B; ++b) {
        if (p0[b] < 0) return -1;
        for (int64_t i = 0; i < n; ++i) {
            const int64_t p = (int64_t)p0[b] + i;
            const int64_t j = p < n_sink ? p : n_sink + (p - n_sink) % (S - n_sink);
            slot_pos[b * S + j] = (int32_t)p;
            for (int64_t h = 0; h < Hkv; ++h) {
                memcpy(kc + ((b * Hkv + h) * S + j) * D, k_new + ((b * n + i) * Hkv + h) * D, sizeof(uint16_t) * D);
                memcpy(vc + ((b * Hkv + h) * S + j) * D, v_new + ((b * n + i) * Hkv + h) * D, sizeof(uint16_t) * D);
            }
        }
    }
    return 0;
}

int swa_oracle_cache_append(uint16_t *kc, uint16_t *vc, int32_t *slot_pos, int64_t B, int64_t Hkv, int64_t S,
                            int64_t D, const uint16_t *k_new, const uint16_t *v_new, int64_t n, const int32_t *p0) {
    return swa_oracle_cache_append_ex(kc, vc, slot_pos, B, Hkv, S, D, 0, k_new, v_new, n, p0);
}

/*
 * Chunked prefill against a ring cache.  q: [B,C,Hq,D]; k_new, v_new: [B,C,Hkv,D]
 * (the chunk, positions p0[b] + i); caches [B,Hkv,S,D] with slot_pos [B,S] holding
 * the history.  Key candidates of a query at t = p0[b] + i: every cache slot whose
 * position p satisfies p < p0[b] (history only; a slot at or beyond p0[b] is not
 * history), then every chunk token; each kept when slot_allowed(p, t, W, n_sink).
 * Outputs in (b, h, i) order: o [B,Hq,C,D], lse [B,Hq,C], counts [B,Hq,C].
 */
int swa_oracle_chunk(const uint16_t *q, const uint16_t *k_new, const uint16_t *v_new, const uint16_t *kc,
                     const uint16_t *vc, const int32_t *slot_pos, const int32_t *p0, int64_t B, int64_t C,
                     int64_t Hq, int64_t Hkv, int64_t D, int64_t S, int64_t W, int64_t n_sink, double scale,
                     double *o, double *lse, int64_t *counts) {
    if (B < 0 || C < 0 || Hq <= 0 || Hkv <= 0 || D <= 0 || S <= 0 || W <= 0 || n_sink < 0 || Hq % Hkv != 0)
        return -1;
    const int64_t group = Hq / Hkv;
    const int64_t cap = S + (C > 0 ? C : 1);
#pragma omp parallel
    {
        double *x = (double *)malloc(sizeof(double) * (size_t)cap);
        double *qd = (double *)malloc(sizeof(double) * (size_t)D);
        const uint16_t **krow = (const uint16_t **)malloc(sizeof(void *) * (size_t)cap);
        const uint16_t **vrow = (const uint16_t **)malloc(sizeof(void *) * (size_t)cap);
#pragma omp for schedule(dynamic, 4)
        for (int64_t r = 0; r < B * Hq * C; ++r) {
            const int64_t b = r / (Hq * C), h = (r / C) % Hq, i = r % C, kvh = h / group;
            const int64_t t = (int64_t)p0[b] + i;
            int64_t n = 0;
            for (int64_t j = 0; j < S; ++j) {
                const int64_t p = slot_pos[b * S + j];
                if (p < p0[b] && slot_allowed(p, t, W, n_sink)) {
                    krow[n] = kc + ((b * Hkv + kvh) * S + j) * D;
                    vrow[n] = vc + ((b * Hkv + kvh) * S + j) * D;
                    ++n;
                }
            }
            for (int64_t jj = 0; jj < C; ++jj) {
                if (slot_allowed((int64_t)p0[b] + jj, t, W, n_sink)) {
                    krow[n] = k_new + ((b * C + jj) * Hkv + kvh) * D;
                    vrow[n] = v_new + ((b * C + jj) * Hkv + kvh) * D;
                    ++n;
                }
            }
            const uint16_t *qrow = q + ((b * C + i) * Hq + h) * D;
            for (int64_t c = 0; c < D; ++c) qd[c] = widen_bf16(qrow[c]);
            attend(qd, D, scale, krow, vrow, n, x, o + r * D, lse + r);
            if (counts) counts[r] = n;
        }
        free(x);
        free(qd);
        free(krow);
        free(vrow);
    }
    return 0;
}

int swa_oracle_num_threads(void) {
#ifdef _OPENMP
    return omp_get_max_threads();
#else
    return 1;
#endif
}
