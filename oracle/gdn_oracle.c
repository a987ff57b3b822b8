/*
 * Gated DeltaNet oracle: plain fp64 CPU recurrence.  TEST INFRASTRUCTURE.
 *
 * Only the test-suite, the smoke check and the benchmark's CPU-baseline arm
 * may load this library.  The CUDA product path never calls it and shares no
 * code with it.
 *
 * What it computes: the gated delta rule of Gated DeltaNet (Yang, Kautz and
 * Hatamizadeh, "Gated Delta Networks: Improving Mamba2 with Delta Rule",
 * ICLR 2025, the gated delta rule update), the "recurrent arithmetic" that
 * the vLLM page "Enable batch-invariant mixed decode and prefill for Qwen
 * GDN" (section "Why") routes cached rows through.  For one chain (one
 * sequence, one value head) with state S in R^{d_k x d_v}, token by token:
 *
 *     alpha_t = exp(g_t)
 *     S_t     = alpha_t S_{t-1} - beta_t k_t (k_t^T (alpha_t S_{t-1}))
 *               + beta_t k_t v_t^T
 *     o_t     = scale * S_t^T q_t            (post-update state)
 *
 * Inputs are taken exactly as stored (bf16 bit patterns widened exactly,
 * fp32 gates widened exactly) and all arithmetic is fp64.  Nothing is blocked,
 * fused or reordered beyond the three terms above.
 *
 * Value heads map to key heads in contiguous groups: value head h reads the
 * q/k of key head h / (h_v / h_k) (the pages do not state the mapping; this
 * is the reading used throughout).
 *
 * Intermediate states: when emit_every > 0 the state after every
 * emit_every-th token of a chain is copied out, in order (the vLLM page
 * "GatedDeltaNet Automatic Prefix Caching", section "Purpose": the chunk
 * kernel optionally returns per-chunk intermediate states as a flat stream).
 */
#include <math.h>
#include <stdint.h>
#include <stdlib.h>
#include <string.h>
#ifdef _OPENMP
#include <omp.h>
#endif

static double bf16_to_double(uint16_t bits)
{
    uint32_t u = ((uint32_t)bits) << 16;
    float f;
    memcpy(&f, &u, sizeof f);
    return (double)f;
}

/*
 * Run one chain.  Layouts (row-major):
 *   q, k  : [T_total][h_k][d_k]  bf16 bits
 *   v     : [T_total][h_v][d_v]  bf16 bits
 *   g,beta: [T_total][h_v]       fp32
 *   s     : [d_k][d_v] fp64, holds S_0 on entry and S_T on exit
 *   o     : [T_seq][d_v] fp64 (this chain's outputs, compact)
 *   emits : [floor(T_seq / emit_every)][d_k][d_v] fp64
 */
static void run_chain(int64_t tok0, int64_t n_tok, int head, int h_k, int h_v,
                      int d_k, int d_v, double scale,
                      const uint16_t *q, const uint16_t *k, const uint16_t *v,
                      const float *g, const float *beta,
                      double *s, double *o, int64_t emit_every, double *emits)
{
    const int kh = head / (h_v / h_k);
    double *kt = malloc(sizeof(double) * (size_t)d_k);
    double *qt = malloc(sizeof(double) * (size_t)d_k);
    double *vt = malloc(sizeof(double) * (size_t)d_v);
    double *ka = malloc(sizeof(double) * (size_t)d_v); /* k_t^T (alpha S) */

    for (int64_t t = 0; t < n_tok; ++t) {
        const int64_t tok = tok0 + t;
        const uint16_t *qp = q + ((size_t)tok * h_k + kh) * d_k;
        const uint16_t *kp = k + ((size_t)tok * h_k + kh) * d_k;
        const uint16_t *vp = v + ((size_t)tok * h_v + head) * d_v;
        for (int i = 0; i < d_k; ++i) {
            kt[i] = bf16_to_double(kp[i]);
            qt[i] = bf16_to_double(qp[i]);
        }
        for (int j = 0; j < d_v; ++j) vt[j] = bf16_to_double(vp[j]);
        const double alpha = exp((double)g[(size_t)tok * h_v + head]);
        const double b = (double)beta[(size_t)tok * h_v + head];

        /* ka_j = sum_i k_i (alpha S_ij), summed over i in ascending order */
        for (int j = 0; j < d_v; ++j) ka[j] = 0.0;
        for (int i = 0; i < d_k; ++i)
            for (int j = 0; j < d_v; ++j) ka[j] += kt[i] * (alpha * s[(size_t)i * d_v + j]);
        /* S_ij <- alpha S_ij - beta k_i ka_j + beta k_i v_j */
        for (int i = 0; i < d_k; ++i)
            for (int j = 0; j < d_v; ++j) {
                double *sij = &s[(size_t)i * d_v + j];
                *sij = alpha * *sij - b * kt[i] * ka[j] + b * kt[i] * vt[j];
            }
        /* o_j = scale * sum_i S_ij q_i, summed over i in ascending order */
        double *ot = o + (size_t)t * d_v;
        for (int j = 0; j < d_v; ++j) ot[j] = 0.0;
        for (int i = 0; i < d_k; ++i)
            for (int j = 0; j < d_v; ++j) ot[j] += s[(size_t)i * d_v + j] * qt[i];
        for (int j = 0; j < d_v; ++j) ot[j] *= scale;
        if (emit_every > 0 && (t + 1) % emit_every == 0) {
            memcpy(emits + (size_t)((t + 1) / emit_every - 1) * d_k * d_v, s,
                   sizeof(double) * (size_t)d_k * d_v);
        }
    }
    free(kt);
    free(qt);
    free(vt);
    free(ka);
}

/*
 * Run n_pairs chains (pair p = sequence pair_seq[p], value head pair_head[p])
 * of a packed varlen batch whose sequence s spans tokens
 * [cu_seqlens[s], cu_seqlens[s+1]).
 *
 *   s0      : [n_pairs][d_k][d_v] fp64 initial states, or NULL for zeros
 *   o       : concatenation over pairs of [T_seq][d_v] fp64
 *   s_final : [n_pairs][d_k][d_v] fp64
 *   emits   : concatenation over pairs of [floor(T_seq/emit_every)][d_k][d_v]
 *             (ignored when emit_every == 0)
 *   n_threads <= 0 uses the OpenMP default.
 * Returns 0, or -1 on a bad argument.
 */
int gdn_oracle_chains(int n_pairs, const int32_t *pair_seq, const int32_t *pair_head,
                      int n_seq, const int64_t *cu_seqlens, int h_k, int h_v,
                      int d_k, int d_v, double scale,
                      const uint16_t *q, const uint16_t *k, const uint16_t *v,
                      const float *g, const float *beta, const double *s0,
                      double *o, double *s_final, int64_t emit_every, double *emits,
                      int n_threads)
{
    if (n_pairs < 0 || h_k <= 0 || h_v <= 0 || h_v % h_k != 0 || d_k <= 0 || d_v <= 0)
        return -1;
    if (emit_every < 0 || (emit_every > 0 && emits == NULL)) return -1;
    int64_t *o_off = malloc(sizeof(int64_t) * (size_t)(n_pairs + 1));
    int64_t *e_off = malloc(sizeof(int64_t) * (size_t)(n_pairs + 1));
    o_off[0] = 0;
    e_off[0] = 0;
    for (int p = 0; p < n_pairs; ++p) {
        if (pair_seq[p] < 0 || pair_seq[p] >= n_seq || pair_head[p] < 0 || pair_head[p] >= h_v) {
            free(o_off);
            free(e_off);
            return -1;
        }
        const int64_t len = cu_seqlens[pair_seq[p] + 1] - cu_seqlens[pair_seq[p]];
        o_off[p + 1] = o_off[p] + len;
        e_off[p + 1] = e_off[p] + (emit_every > 0 ? len / emit_every : 0);
    }
#ifdef _OPENMP
    if (n_threads > 0) omp_set_num_threads(n_threads);
#pragma omp parallel for schedule(dynamic, 1)
#endif
    for (int p = 0; p < n_pairs; ++p) {
        const size_t ss = (size_t)d_k * d_v;
        double *s = s_final + (size_t)p * ss;
        if (s0) {
            memcpy(s, s0 + (size_t)p * ss, sizeof(double) * ss);
        } else {
            memset(s, 0, sizeof(double) * ss);
        }
        const int64_t t0 = cu_seqlens[pair_seq[p]];
        const int64_t len = cu_seqlens[pair_seq[p] + 1] - t0;
        run_chain(t0, len, pair_head[p], h_k, h_v, d_k, d_v, scale, q, k, v, g, beta, s,
                  o + (size_t)o_off[p] * d_v, emit_every,
                  emit_every > 0 ? emits + (size_t)e_off[p] * ss : NULL);
    }
    free(o_off);
    free(e_off);
    return 0;
}

int gdn_oracle_max_threads(void)
{
#ifdef _OPENMP
    return omp_get_max_threads();
#else
    return 1;
#endif
}
