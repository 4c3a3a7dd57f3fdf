/*
 * oracle.c -- plain, slow CPU oracle for incremental decoding against a
 * preallocated KV cache.
 *
 * TEST INFRASTRUCTURE ONLY.  Nothing in the product path may link, load or
 * call this file: only tests/, the smoke check and the benchmark's CPU
 * baseline do.  It shares no code, header, table or constant with the CUDA
 * library; the two agree only because both follow the same published
 * definitions.
 *
 * What it computes is cache-free attention: for every query it rotates that
 * query and every visible key of the row's history from scratch and runs a
 * plain max-subtracted softmax in double precision.  There is no cache, no
 * blocking, no split and no online softmax here -- those are the product's
 * business.
 *
 * Sources (web pages, by title and section):
 *  - tiny_agent/generate.py, `_rope_pos`: half-split RoPE pairing
 *    (x1, x2) = halves of the head vector -> (x1 c - x2 s, x1 s + x2 c).
 *  - tiny_agent/generate.py, `_append_chunk`: per-row absolute positions
 *    pos = lens + i; grouped queries (head h reads kv head h / rep);
 *    scale 1/sqrt(D); local mask lpos <= pos and pos - lpos < W; the
 *    "keep the last W real tokens" ring rule.
 *  - Lab 07 -- KV cache and sampling, section 2 "The offset mask": query i
 *    of a forward that starts at pos sees key j iff j <= pos + i.
 *  - pycraft-1 model/kv_cache.py, `build_attn_mask`: bottom-right aligned
 *    mask[i, j] = (j <= offset + i); the cache holds post-RoPE keys.
 *  - "inkling: ring-buffer KV cache for sliding-window layers", section
 *    "What this does": the sliding scan starts at t0 = qpos - window + 1;
 *    "How it works": a sliding layer's ring has `window` rows addressed at
 *    t % window.
 *
 * Readings taken where the pages leave a step open (each one is listed in
 * the design notes of the repository):
 *  - RoPE frequencies theta_i = theta^(-2i/D) for i < D/2; the exponent is
 *    the double quotient (-2i)/D, the angle p*theta_i is formed in double,
 *    and cos/sin are rounded once to float.
 *  - RoPE arithmetic is float with no fused multiply-add (build with
 *    -ffp-contract=off), rounded once to bfloat16 (round to nearest even).
 *  - A sliding window of W keeps W keys including the query's own position:
 *    keys j in [max(0, p - W + 1), p].  W <= 0 means a global layer.
 *  - The attention itself is evaluated in double from the bf16 values.
 */
#include <math.h>
#include <stdint.h>
#include <stdlib.h>
#include <string.h>

#ifdef _OPENMP
#include <omp.h>
#endif

/* ---------------------------------------------------------------- bf16 */

/* Round a float to bfloat16, round to nearest, ties to even. */
uint16_t oracle_f32_to_bf16(float f)
{
    uint32_t u;
    memcpy(&u, &f, sizeof u);
    if ((u & 0x7F800000u) == 0x7F800000u && (u & 0x007FFFFFu) != 0u)
        return (uint16_t)((u >> 16) | 0x0040u); /* quiet NaN */
    uint32_t lsb = (u >> 16) & 1u;
    u += 0x7FFFu + lsb;
    return (uint16_t)(u >> 16);
}

float oracle_bf16_to_f32(uint16_t h)
{
    uint32_t u = (uint32_t)h << 16;
    float f;
    memcpy(&f, &u, sizeof f);
    return f;
}

/* ---------------------------------------------------------------- RoPE */

/* cos/sin of position p for frequency pair i, as floats (the table entry). */
void oracle_rope_cs(int p, int i, int D, double theta, float *c, float *s)
{
    double inv_freq = pow(theta, (double)(-2 * i) / (double)D);
    double angle = (double)p * inv_freq;
    *c = (float)cos(angle);
    *s = (float)sin(angle);
}

/* Fill cos/sin tables [n_pos][D/2] (used by tests as a pin target). */
void oracle_rope_table(int n_pos, int D, double theta, float *cos_out, float *sin_out)
{
    int half = D / 2;
    for (int p = 0; p < n_pos; ++p)
        for (int i = 0; i < half; ++i)
            oracle_rope_cs(p, i, D, theta, &cos_out[(size_t)p * half + i],
                           &sin_out[(size_t)p * half + i]);
}

/* Rotate one head vector x[D] (bf16 bits) to position p; result in bf16 bits. */
void oracle_rope_bf16(const uint16_t *x, int p, int D, double theta, uint16_t *out)
{
    int half = D / 2;
    for (int i = 0; i < half; ++i) {
        float c, s;
        oracle_rope_cs(p, i, D, theta, &c, &s);
        float x1 = oracle_bf16_to_f32(x[i]);
        float x2 = oracle_bf16_to_f32(x[i + half]);
        float a = x1 * c;
        float b = x2 * s;
        float lo = a - b;
        float e = x1 * s;
        float f = x2 * c;
        float hi = e + f;
        out[i] = oracle_f32_to_bf16(lo);
        out[i + half] = oracle_f32_to_bf16(hi);
    }
}

/* Rotate n head vectors x[n][D], vector r to position pos[r]. */
void oracle_rope_rows(const uint16_t *x, const int32_t *pos, int n, int D, double theta,
                      uint16_t *out)
{
#pragma omp parallel for schedule(static)
    for (int r = 0; r < n; ++r)
        oracle_rope_bf16(&x[(size_t)r * D], pos[r], D, theta, &out[(size_t)r * D]);
}

/* ---------------------------------------------------------------- masks */

/* Is key position j visible to a query at absolute position p?
 * Global layers (W <= 0): 0 <= j <= p.  Sliding layers: p - W < j <= p. */
int oracle_visible(int p, int j, int W)
{
    if (j < 0 || j > p) return 0;
    if (W > 0 && p - j >= W) return 0;
    return 1;
}

/* Expected ring-slot occupancy after `lens` tokens of one row have been
 * appended under the keep-the-last-W rule: slot s holds the largest
 * position t < lens with t % W == s, or -1 when no such position exists. */
void oracle_ring_positions(int lens, int W, int32_t *slot_pos)
{
    for (int s = 0; s < W; ++s) {
        int best = -1;
        for (int t = 0; t < lens; ++t)
            if (t % W == s) best = t;
        slot_pos[s] = best;
    }
}

/* ------------------------------------------------------------ attention */

/*
 * Cache-free attention for one cache row.
 *
 *   q      [n_q][Hq][D]  bf16 bits, pre-RoPE, query i sits at position qpos[i]
 *   k, v   [n_k][Hk][D]  bf16 bits, pre-RoPE keys / values of positions
 *                        k_base .. k_base + n_k - 1 of the same row
 *   out    [n_q][Hq][D]  double
 *
 * For each query and head h (kv head g = h / (Hq/Hk)): rotate the query to
 * its position and every visible key to its own position, score
 * s_j = (Q . K_j) / sqrt(D), w = softmax(s) (max subtracted), out = sum w_j V_j.
 *
 * Returns 0, or -1 when the arguments are invalid or the supplied history
 * does not cover some query's visible keys.
 */
int oracle_attend(const uint16_t *q, const int32_t *qpos, int n_q,
                  const uint16_t *k, const uint16_t *v, int k_base, int n_k,
                  int Hq, int Hk, int D, int W, double theta, double *out)
{
    if (n_q < 0 || n_k < 0 || Hq <= 0 || Hk <= 0 || D <= 0 || (D % 2) != 0 ||
        (Hq % Hk) != 0)
        return -1;
    int rep = Hq / Hk;
    for (int i = 0; i < n_q; ++i) {
        int p = qpos[i];
        int lo = (W > 0 && p - W + 1 > 0) ? p - W + 1 : 0;
        if (p < 0 || lo < k_base || p >= k_base + n_k) return -1;
    }

    /* rotate every key once (still no cache: this call recomputes them) */
    uint16_t *kr = (uint16_t *)malloc((size_t)n_k * Hk * D * sizeof(uint16_t));
    if (!kr && n_k > 0) return -1;
#pragma omp parallel for schedule(static)
    for (int j = 0; j < n_k; ++j)
        for (int g = 0; g < Hk; ++g)
            oracle_rope_bf16(&k[((size_t)j * Hk + g) * D], k_base + j, D, theta,
                             &kr[((size_t)j * Hk + g) * D]);

    int rc = 0;
#pragma omp parallel for collapse(2) schedule(dynamic)
    for (int i = 0; i < n_q; ++i) {
        for (int h = 0; h < Hq; ++h) {
            int p = qpos[i];
            int g = h / rep;
            uint16_t *qr = (uint16_t *)malloc((size_t)D * sizeof(uint16_t));
            double *s = (double *)malloc((size_t)(p + 1) * sizeof(double));
            double *acc = &out[((size_t)i * Hq + h) * D];
            if (!qr || !s) {
                free(qr);
                free(s);
#pragma omp atomic write
                rc = -1;
                continue;
            }
            oracle_rope_bf16(&q[((size_t)i * Hq + h) * D], p, D, theta, qr);

            /* scores over the visible keys */
            double m = -INFINITY;
            for (int j = 0; j <= p; ++j) {
                if (!oracle_visible(p, j, W)) {
                    s[j] = -INFINITY;
                    continue;
                }
                const uint16_t *kj = &kr[((size_t)(j - k_base) * Hk + g) * D];
                double dot = 0.0;
                for (int d = 0; d < D; ++d)
                    dot += (double)oracle_bf16_to_f32(qr[d]) * (double)oracle_bf16_to_f32(kj[d]);
                s[j] = dot / sqrt((double)D);
                if (s[j] > m) m = s[j];
            }
            /* softmax weights and the weighted sum of values */
            double denom = 0.0;
            for (int d = 0; d < D; ++d) acc[d] = 0.0;
            for (int j = 0; j <= p; ++j) {
                if (s[j] == -INFINITY) continue;
                double w = exp(s[j] - m);
                denom += w;
                const uint16_t *vj = &v[((size_t)(j - k_base) * Hk + g) * D];
                for (int d = 0; d < D; ++d) acc[d] += w * (double)oracle_bf16_to_f32(vj[d]);
            }
            for (int d = 0; d < D; ++d) acc[d] /= denom;
            free(qr);
            free(s);
        }
    }
    free(kr);
    return rc;
}

/*
 * Hybrid attention (tiny_agent/generate.py, module docstring and `_append_chunk`): a layer
 * of a group scores its query against two key sets in ONE softmax -- the group's global
 * keys (written by the group's full layer) at every position j <= p, and the layer's own
 * local keys at the positions of its window (j <= p and p - j < W) -- and sums both sets'
 * values with those weights: the two score vectors form one vector over which a single
 * max-subtracted softmax is taken, and the output is the weighted sum of the global values
 * plus the weighted sum of the local values.
 *
 *   q            [n_q][Hq][D] bf16 bits, pre-RoPE
 *   qpos         [n_q]
 *   kg, vg       [n_k][Hk][D] bf16 bits: pre-RoPE global keys / values of positions 0..n_k-1
 *   kl, vl       [n_k][Hk][D] bf16 bits: pre-RoPE local keys / values of the same positions
 *   out          [n_q][Hq][D] double
 *
 * Returns 0, or -1 when the arguments are invalid or a query's position is not covered.
 */
int oracle_attend_hybrid(const uint16_t *q, const int32_t *qpos, int n_q,
                         const uint16_t *kg, const uint16_t *vg, const uint16_t *kl,
                         const uint16_t *vl, int n_k, int Hq, int Hk, int D, int W,
                         double theta, double *out)
{
    if (n_q < 0 || n_k < 0 || Hq <= 0 || Hk <= 0 || D <= 0 || (D % 2) != 0 ||
        (Hq % Hk) != 0 || W < 1)
        return -1;
    int rep = Hq / Hk;
    for (int i = 0; i < n_q; ++i)
        if (qpos[i] < 0 || qpos[i] >= n_k) return -1;

    size_t nkv = (size_t)n_k * Hk * D;
    uint16_t *kgr = (uint16_t *)malloc(nkv * sizeof(uint16_t) + 1);
    uint16_t *klr = (uint16_t *)malloc(nkv * sizeof(uint16_t) + 1);
    if (!kgr || !klr) {
        free(kgr);
        free(klr);
        return -1;
    }
#pragma omp parallel for schedule(static)
    for (int j = 0; j < n_k; ++j)
        for (int g = 0; g < Hk; ++g) {
            size_t o = ((size_t)j * Hk + g) * D;
            oracle_rope_bf16(&kg[o], j, D, theta, &kgr[o]);
            oracle_rope_bf16(&kl[o], j, D, theta, &klr[o]);
        }

    int rc = 0;
#pragma omp parallel for collapse(2) schedule(dynamic)
    for (int i = 0; i < n_q; ++i) {
        for (int h = 0; h < Hq; ++h) {
            int p = qpos[i];
            int g = h / rep;
            uint16_t *qr = (uint16_t *)malloc((size_t)D * sizeof(uint16_t));
            double *s = (double *)malloc((size_t)2 * (p + 1) * sizeof(double)); /* [global | local] */
            double *acc = &out[((size_t)i * Hq + h) * D];
            if (!qr || !s) {
                free(qr);
                free(s);
#pragma omp atomic write
                rc = -1;
                continue;
            }
            oracle_rope_bf16(&q[((size_t)i * Hq + h) * D], p, D, theta, qr);
            double m = -INFINITY;
            for (int set = 0; set < 2; ++set) {
                const uint16_t *kr = set == 0 ? kgr : klr;
                for (int j = 0; j <= p; ++j) {
                    double *sj = &s[(size_t)set * (p + 1) + j];
                    if (set == 1 && !oracle_visible(p, j, W)) {
                        *sj = -INFINITY;
                        continue;
                    }
                    const uint16_t *kj = &kr[((size_t)j * Hk + g) * D];
                    double dot = 0.0;
                    for (int d = 0; d < D; ++d)
                        dot += (double)oracle_bf16_to_f32(qr[d]) * (double)oracle_bf16_to_f32(kj[d]);
                    *sj = dot / sqrt((double)D);
                    if (*sj > m) m = *sj;
                }
            }
            double denom = 0.0;
            for (int d = 0; d < D; ++d) acc[d] = 0.0;
            for (int set = 0; set < 2; ++set) {
                const uint16_t *vv = set == 0 ? vg : vl;
                for (int j = 0; j <= p; ++j) {
                    double sj = s[(size_t)set * (p + 1) + j];
                    if (sj == -INFINITY) continue;
                    double w = exp(sj - m);
                    denom += w;
                    const uint16_t *vj = &vv[((size_t)j * Hk + g) * D];
                    for (int d = 0; d < D; ++d) acc[d] += w * (double)oracle_bf16_to_f32(vj[d]);
                }
            }
            for (int d = 0; d < D; ++d) acc[d] /= denom;
            free(qr);
            free(s);
        }
    }
    free(kgr);
    free(klr);
    return rc;
}

/* ---------------------------------------------------------------- memory */

/* K+V bytes of a cache whose global layers keep max_len rows per (row, kv
 * head) and whose sliding layers keep W rows; `extra_slots` rows per
 * (row, kv head) are added to both kinds (1 for a scratch slot, 0 for none).
 * Lab 07 section "Check yourself" answer 1, and the inkling pull request's
 * memory table, count bytes this way (2 for K and V). */
int64_t oracle_kv_nbytes(int B, int max_len, int W, int D, int elem_bytes,
                         int n_global, int Hk_global, int n_sliding, int Hk_sliding,
                         int extra_slots)
{
    int64_t ring = (W > 0 && W < max_len) ? W : max_len;
    int64_t g = 2LL * n_global * B * Hk_global * (int64_t)(max_len + extra_slots) * D * elem_bytes;
    int64_t s = 2LL * n_sliding * B * Hk_sliding * (int64_t)(ring + extra_slots) * D * elem_bytes;
    return g + s;
}

/* Number of threads the parallel loops above use (for reporting). */
int oracle_num_threads(void)
{
#ifdef _OPENMP
    return omp_get_max_threads();
#else
    return 1;
#endif
}
