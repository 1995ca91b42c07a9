/*
 * sa_oracle.c -- plain fp64 CPU oracle for DeepSeek-V4.1-style sparse latent
 * attention and its fused output tail.
 *
 * TEST INFRASTRUCTURE ONLY.  Nothing in the product library links, includes or
 * calls this file; only the test suite, the smoke check and the benchmark's
 * CPU-baseline leg load it (through ctypes).  It shares no code, header, table
 * or helper with the CUDA path.
 *
 * Sources (pages by title and section):
 *   [P1] "DeepSeek-V4.1 > Output projection" page, code excerpts
 *        `Attention.forward` and `Attention.__init__`: the call
 *        `sparse_attn(q, kv, attn_sink, topk_idxs, softmax_scale)`, the inverse
 *        rotary embedding of the last rope_head_dim output features, and the
 *        block-diagonal `einsum("bsgd,grd->bsgr", o, wo_a)`; `attn_sink` is one
 *        fp32 logit per head; `softmax_scale = head_dim ** -0.5`.
 *   [P2] "DeepSeek-V4.1 > 40 layers" (re-indexing groups) page, excerpts
 *        `_compress_topk_idxs` / `_compress_kv` and config.json: index lists are
 *        int32, compressed positions are offset by the window length,
 *        head_dim 512, rope_head_dim 64, compress_rope_theta 160000.
 *   [P3] "GLM-5 > Sparse latent attention > key_states" page, excerpt
 *        `eager_attention_forward`: scaled scores, softmax over the kept
 *        positions, probability-weighted sum of values.
 *   The sink term and the meaning of -1 (skip) are not printed on the pages;
 *   the reading used here is: the sink is one extra logit in the softmax
 *   denominator with a zero value vector and is not multiplied by the scale;
 *   an index of -1 contributes nothing wherever it sits in the list; every
 *   other listed index contributes one term (a repeated index counts twice).
 *
 * Arithmetic: every input is promoted exactly to double (bf16 -> fp32 -> fp64)
 * and all sums, exponentials and divisions run in double.  No blocking,
 * fusion or online-softmax reordering: scores are formed, the maximum taken,
 * the exponentials summed, and the weighted rows accumulated, in that order.
 *
 * Parity pins (tests/test_oracle_pins.py): dense masked brute force, closed
 * forms for one valid index / equal scores / sink -> -inf, permutation
 * invariance, the all-skip row, the one-hot index probe, the rotary group
 * law and special angles, and a block-diagonal dense matmul for wo_a.
 */
#include <math.h>
#include <stdint.h>
#include <stdlib.h>
#include <string.h>
#ifdef _OPENMP
#include <omp.h>
#endif

static double bf16_to_f64(uint16_t h)
{
    uint32_t u = ((uint32_t)h) << 16;
    float f;
    memcpy(&f, &u, sizeof f);
    return (double)f;
}

/* Number of OpenMP threads the oracle will use when asked for n (0 = all). */
int sa_oracle_threads(int n)
{
#ifdef _OPENMP
    return n > 0 ? n : omp_get_max_threads();
#else
    (void)n;
    return 1;
#endif
}

/*
 * One output row o[h, :] for query (b, t) and head h  ([P1] sparse_attn call).
 *
 *   S     = { j : idx[b,t,j] != -1 }                   (each listed entry a term)
 *   s_j   = scale * sum_d q[b,t,h,d] * kv[b, idx_j, d]
 *   M     = max(sink[h], max_j s_j)
 *   den   = exp(sink[h] - M) + sum_j exp(s_j - M)
 *   o     = sum_j exp(s_j - M) * kv[b, idx_j, :] / den
 *
 * An empty S gives o = 0 (its numerator is an empty sum); with sink = -inf and
 * an empty S the 0/0 is also defined as 0.
 * Returns 1 if an entry outside [-1, N) was met (it is then left out).
 */
static int one_head(const uint16_t *qrow, const uint16_t *kvb, double sink,
                    const int32_t *idx, double scale, int D, int N, int K,
                    double *s, double *o)
{
    int bad = 0;
    int j, d;
    double M = sink;
    double den;

    for (d = 0; d < D; ++d)
        o[d] = 0.0;

    /* scores */
    for (j = 0; j < K; ++j) {
        int r = idx[j];
        if (r == -1) {
            s[j] = -INFINITY;
            continue;
        }
        if (r < -1 || r >= N) {
            bad = 1;
            s[j] = -INFINITY;
            continue;
        }
        {
            const uint16_t *kr = kvb + (size_t)r * D;
            double acc = 0.0;
            for (d = 0; d < D; ++d)
                acc += bf16_to_f64(qrow[d]) * bf16_to_f64(kr[d]);
            s[j] = scale * acc;
        }
        if (s[j] > M)
            M = s[j];
    }

    if (M == -INFINITY) /* no valid entry and a sink of -inf */
        return bad;

    /* softmax denominator, the sink included */
    den = exp(sink - M);
    for (j = 0; j < K; ++j)
        if (s[j] != -INFINITY)
            den += exp(s[j] - M);

    /* probability-weighted rows */
    for (j = 0; j < K; ++j) {
        double p;
        const uint16_t *kr;
        if (s[j] == -INFINITY)
            continue;
        p = exp(s[j] - M) / den;
        kr = kvb + (size_t)idx[j] * D;
        for (d = 0; d < D; ++d)
            o[d] += p * bf16_to_f64(kr[d]);
    }
    return bad;
}

/*
 * sparse_attn over a list of queries.
 *   q    bf16 [B, T, H, D]      kv bf16 [B, N, D]      sink fp32 [H]
 *   idx  int32 [B, T, K]        scale: softmax scale (the pages: D ** -0.5)
 *   queries: flattened query numbers b*T + t to evaluate (NULL = all B*T)
 *   out  fp64 [n_queries, H, D]
 * Returns the number of queries in which an out-of-range index was met.
 */
int64_t sa_oracle_sparse_attn(const uint16_t *q, const uint16_t *kv,
                              const float *sink, const int32_t *idx,
                              double scale, int B, int T, int H, int D, int N,
                              int K, const int64_t *queries, int64_t n_queries,
                              double *out, int n_threads)
{
    int64_t nq = queries ? n_queries : (int64_t)B * T;
    int64_t n_bad = 0;
    int64_t i;

#ifdef _OPENMP
#pragma omp parallel for schedule(dynamic, 1) reduction(+ : n_bad) num_threads(sa_oracle_threads(n_threads))
#endif
    for (i = 0; i < nq; ++i) {
        int64_t qi = queries ? queries[i] : i;
        int64_t b = qi / T;
        int h, bad = 0;
        double *s = (double *)malloc(sizeof(double) * (size_t)(K > 0 ? K : 1));
        const uint16_t *kvb = kv + (size_t)b * N * D;
        const int32_t *il = idx + (size_t)qi * K;
        for (h = 0; h < H; ++h)
            bad |= one_head(q + ((size_t)qi * H + h) * D, kvb, (double)sink[h],
                            il, scale, D, N, K, s, out + ((size_t)i * H + h) * D);
        free(s);
        n_bad += bad;
    }
    (void)B;
    return n_bad;
}

/*
 * Inverse rotary embedding on the last rope_dim features of every head
 * ([P1] `apply_rotary_emb(o[..., -rd:], freqs_cis, True)`), in place.
 * Reading: consecutive feature pairs (2i, 2i+1) form one complex number
 * a + i*b; frequency i is theta ** (-2i / rope_dim); the forward embedding at
 * position p multiplies by exp(+i*p*w_i), the inverse by exp(-i*p*w_i):
 *   (a, b) -> (a cos phi + b sin phi, -a sin phi + b cos phi),  phi = p * w_i.
 *   o    fp64 [n, H, D] (in place)      pos: position of each of the n rows
 */
void sa_oracle_inverse_rope(double *o, int64_t n, const int64_t *pos, int H,
                            int D, int rope_dim, double theta, int n_threads)
{
    int64_t r;
#ifdef _OPENMP
#pragma omp parallel for schedule(static) num_threads(sa_oracle_threads(n_threads))
#endif
    for (r = 0; r < n; ++r) {
        int h, i;
        for (h = 0; h < H; ++h) {
            double *x = o + ((size_t)r * H + h) * D + (D - rope_dim);
            for (i = 0; i < rope_dim / 2; ++i) {
                double w = pow(theta, -2.0 * i / rope_dim);
                double phi = (double)pos[r] * w;
                double c = cos(phi), sn = sin(phi);
                double a = x[2 * i], b = x[2 * i + 1];
                x[2 * i] = a * c + b * sn;
                x[2 * i + 1] = -a * sn + b * c;
            }
        }
    }
}

/*
 * Grouped low-rank output projection ([P1] `o.view(B, T, G, -1)`,
 * `wo_a.weight.view(G, R, -1)`, `einsum("bsgd,grd->bsgr")`):
 *   y[n, g, r] = sum_{d < Din} o[n, g, d] * W[g, r, d]
 *   o fp64 [n, G, Din]     W bf16 [G, R, Din]     y fp64 [n, G, R]
 */
void sa_oracle_wo_a(const double *o, const uint16_t *W, int64_t n, int G,
                    int R, int Din, double *y, int n_threads)
{
    int64_t t;
#ifdef _OPENMP
#pragma omp parallel for schedule(static) num_threads(sa_oracle_threads(n_threads))
#endif
    for (t = 0; t < n; ++t) {
        int g, r, d;
        for (g = 0; g < G; ++g) {
            const double *x = o + ((size_t)t * G + g) * Din;
            for (r = 0; r < R; ++r) {
                const uint16_t *w = W + ((size_t)g * R + r) * Din;
                double acc = 0.0;
                for (d = 0; d < Din; ++d)
                    acc += x[d] * bf16_to_f64(w[d]);
                y[((size_t)t * G + g) * R + r] = acc;
            }
        }
    }
}
