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
 * Decode (ring-buffer cache): the cache of W slots holds, per slot j, the true
 * token position slot_pos[b][j] (Gemma 3 sliding-window note, ai-engineer-
 * exhaustive.pages.dev: positions are stored in the cache and the window is
 * computed from them).  Slot j is allowed for the query at t = q_pos[b] iff
 * p >= 0 and t - W < p <= t.  The rest is steps 2-4.
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

/* Step 1: the explicit mask row of query t over keys [0, T). */
void swa_oracle_mask_row(int64_t T, int64_t t, int32_t wl, int32_t wr, const int32_t *G,
                         int64_t nG, uint8_t *allowed) {
    const int row_is_global = is_member(G, nG, t);
    for (int64_t s = 0; s < T; ++s) {
        const int in_band = (wl < 0 || s >= t - wl) && (wr < 0 || s <= t + wr);
        allowed[s] = (uint8_t)(in_band || row_is_global || is_member(G, nG, s));
    }
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
 * rows: nrows (b, h, t) triples to evaluate, or NULL for every row in (b, h, t)
 * order (nrows must then be B*Hq*T).  Outputs per evaluated row i: o[i*D ..],
 * lse[i], counts[i] (counts may be NULL).  Returns 0, or -1 on a bad argument.
 */
int swa_oracle_fwd(const uint16_t *q, const uint16_t *k, const uint16_t *v, int64_t B, int64_t T,
                   int64_t Hq, int64_t Hkv, int64_t D, int32_t wl, int32_t wr, double scale,
                   const int32_t *G, int64_t nG, const int64_t *rows, int64_t nrows, double *o,
                   double *lse, int64_t *counts) {
    if (B < 0 || T < 0 || Hq <= 0 || Hkv <= 0 || D <= 0 || Hq % Hkv != 0 || nrows < 0) return -1;
    if (rows == NULL && nrows != B * Hq * T) return -1;
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
            swa_oracle_mask_row(T, t, wl, wr, G, nG, allowed);
            int64_t n = 0;
            for (int64_t s = 0; s < T; ++s) {
                if (!allowed[s]) continue;
                krow[n] = k + ((b * T + s) * Hkv + kvh) * D;
                vrow[n] = v + ((b * T + s) * Hkv + kvh) * D;
                ++n;
            }
            const uint16_t *qrow = q + ((b * T + t) * Hq + h) * D;
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

/*
 * Ring-buffer decode.  q: [B,Hq,D]; k_cache, v_cache: [B,Hkv,W,D]; slot_pos: [B,W];
 * q_pos: [B].  Outputs o: [B,Hq,D], lse: [B,Hq], counts: [B,Hq] (may be NULL).
 */
int swa_oracle_decode(const uint16_t *q, const uint16_t *kc, const uint16_t *vc,
                      const int32_t *slot_pos, const int32_t *q_pos, int64_t B, int64_t Hq,
                      int64_t Hkv, int64_t D, int64_t W, double scale, double *o, double *lse,
                      int64_t *counts) {
    if (B < 0 || Hq <= 0 || Hkv <= 0 || D <= 0 || W <= 0 || Hq % Hkv != 0) return -1;
    const int64_t group = Hq / Hkv;
#pragma omp parallel
    {
        double *x = (double *)malloc(sizeof(double) * (size_t)W);
        double *qd = (double *)malloc(sizeof(double) * (size_t)D);
        const uint16_t **krow = (const uint16_t **)malloc(sizeof(void *) * (size_t)W);
        const uint16_t **vrow = (const uint16_t **)malloc(sizeof(void *) * (size_t)W);
#pragma omp for schedule(dynamic, 4)
        for (int64_t i = 0; i < B * Hq; ++i) {
            const int64_t b = i / Hq, h = i % Hq, kvh = h / group;
            const int64_t t = q_pos[b];
            int64_t n = 0;
            for (int64_t j = 0; j < W; ++j) {
                const int64_t p = slot_pos[b * W + j];
                if (p >= 0 && p > t - W && p <= t) {
                    krow[n] = kc + ((b * Hkv + kvh) * W + j) * D;
                    vrow[n] = vc + ((b * Hkv + kvh) * W + j) * D;
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

int swa_oracle_num_threads(void) {
#ifdef _OPENMP
    return omp_get_max_threads();
#else
    return 1;
#endif
}
