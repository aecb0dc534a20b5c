/*
 * CPU oracle for the routed-expert MoE forward.
 *
 * TEST INFRASTRUCTURE ONLY.  Only the test suite, the smoke check and the
 * benchmark's CPU-baseline leg may load this library.  The CUDA library never
 * links, includes or calls anything here, and nothing here comes from it.
 *
 * Plain loops over plain arrays, written to be checked by eye against the
 * pages they follow:
 *   - "mslk/moe/gather_scatter.py" (mslk-cuda-nightly 2026.1.19): the gather,
 *     gather + FP8-rowwise quantise and scatter-add kernels;
 *   - "mslk/moe/layers.py" (same wheel): RoutedExperts.build (weight layout),
 *     BaselineMoE._forward / _fake_quant (the dense definition of the forward),
 *     MetaShufflingMoE._route / _routed_expert / _combine_outputs (stage order),
 *     the router scores of _route and the shared expert of
 *     _shared_expert_part1 / _shared_expert_part2.
 *
 * Precision: fp32 where the pages fix it (the gather and quantise kernels
 * upcast to fp32 and do their arithmetic there); fp64 for the GEMM dot
 * products and the SiLU product, which the pages leave to library code;
 * results are rounded to the stage's output type (bf16 or e4m3) once.
 *
 * Number formats are written from their definitions: bf16 is the upper half
 * of an IEEE binary32 (round to nearest, ties to even); e4m3 is the OCP FP8
 * E4M3 format (1 sign, 4 exponent bits with bias 7, 3 mantissa bits, no
 * infinities, S.1111.111 is NaN, largest finite 448).
 *
 * Build: gcc -O2 -ffp-contract=off -fPIC -shared [-fopenmp] -lm.  OpenMP only
 * splits independent output rows across cores; every row is computed by the
 * same sequential loop whatever the thread count.
 */
#include <math.h>
#include <stdint.h>
#include <stdlib.h>
#include <string.h>

#ifdef _OPENMP
#include <omp.h>
#endif

#define ORACLE_FP8_MAX 448.0f
/* The pages take EPS from get_fp8_constants(), which they do not show. Reading: 1e-12. */
#define ORACLE_FP8_EPS 1e-12f

enum { ORACLE_BF16 = 0, ORACLE_F32 = 1 };

int oracle_num_threads(void) {
#ifdef _OPENMP
    return omp_get_max_threads();
#else
    return 1;
#endif
}

/* ------------------------------------------------------------------ bf16 */

static float bf16_to_f32(uint16_t h) {
    uint32_t u = (uint32_t)h << 16;
    float f;
    memcpy(&f, &u, sizeof f);
    return f;
}

/* Round a binary32 to the nearest bf16, ties to the even neighbour. */
static uint16_t f32_to_bf16(float f) {
    uint32_t u;
    memcpy(&u, &f, sizeof u);
    if ((u & 0x7f800000u) == 0x7f800000u && (u & 0x007fffffu) != 0)
        return (uint16_t)((u >> 16) | 0x0040u); /* NaN stays NaN (quiet) */
    uint32_t lower = u & 0xffff0000u; /* truncation: the neighbour towards zero */
    uint32_t rest = u & 0x0000ffffu;  /* the dropped half, as a fraction of one bf16 ulp */
    if (rest > 0x8000u || (rest == 0x8000u && (lower & 0x00010000u)))
        lower += 0x00010000u; /* the neighbour away from zero (a carry may reach the exponent) */
    return (uint16_t)(lower >> 16);
}

/* ------------------------------------------------------------------ e4m3 */

static float e4m3_to_f32(uint8_t b) {
    int sign = b >> 7, exp = (b >> 3) & 0xf, man = b & 0x7;
    float mag;
    if (exp == 0xf && man == 0x7)
        mag = NAN;
    else if (exp == 0)
        mag = ldexpf((float)man, -9); /* subnormal: man/8 * 2^(1-7) */
    else
        mag = ldexpf(1.0f + (float)man / 8.0f, exp - 7);
    return sign ? -mag : mag;
}

/* Nearest e4m3 value to v, ties to even, magnitudes above 448 saturate to 448. */
static uint8_t f32_to_e4m3(float v) {
    uint8_t sign = signbit(v) ? 0x80 : 0x00;
    double a = fabs((double)v);
    if (isnan(v))
        return (uint8_t)(sign | 0x7f);
    if (a > 448.0)
        a = 448.0;
    if (a == 0.0)
        return sign;
    /* Spacing of the grid around a: 2^(b-3) in binade [2^b, 2^(b+1)), b >= -6;
     * the subnormals below 2^-6 share the spacing 2^-9 of binade -6. */
    int e2;
    frexp(a, &e2); /* a = f * 2^e2, f in [0.5, 1): binade b = e2 - 1 */
    int b = e2 - 1;
    if (b < -6)
        b = -6;
    double spacing = ldexp(1.0, b - 3);
    double q = a / spacing;          /* exact: division by a power of two */
    double r = floor(q);
    double frac = q - r;
    if (frac > 0.5 || (frac == 0.5 && fmod(r, 2.0) != 0.0))
        r += 1.0;
    double val = r * spacing;        /* a multiple of the spacing, at most 448 */
    if (val == 0.0)
        return sign;
    if (val < ldexp(1.0, -6))        /* subnormal code: exponent field 0 */
        return (uint8_t)(sign | (uint8_t)(val / ldexp(1.0, -9)));
    frexp(val, &e2);                  /* rounding may have carried into the next binade */
    int be = e2 - 1;
    int man = (int)((val / ldexp(1.0, be) - 1.0) * 8.0);
    return (uint8_t)(sign | (uint8_t)((be + 7) << 3) | (uint8_t)man);
}

void oracle_bf16_round(const float* in, uint16_t* out, int64_t n) {
    for (int64_t i = 0; i < n; ++i) out[i] = f32_to_bf16(in[i]);
}

void oracle_bf16_to_f32(const uint16_t* in, float* out, int64_t n) {
    for (int64_t i = 0; i < n; ++i) out[i] = bf16_to_f32(in[i]);
}

void oracle_e4m3_encode(const float* in, uint8_t* out, int64_t n) {
    for (int64_t i = 0; i < n; ++i) out[i] = f32_to_e4m3(in[i]);
}

void oracle_e4m3_decode(const uint8_t* in, float* out, int64_t n) {
    for (int64_t i = 0; i < n; ++i) out[i] = e4m3_to_f32(in[i]);
}

/* ------------------------------------------------- FP8 row quantisation */

/*
 * One row v[0..n) -> e4m3 codes q[0..n) and the dequantisation scale, as in
 * mslk/moe/gather_scatter.py, kernel _mslk_gather_scale_fp8_rowwise_quant_dense_tokens:
 *   m = max_j |v_j|; m = clamp(m, EPS, ub) when an upper bound is given, else
 *   max(m, EPS); s = MAX_FP8 / m; stored scale = 1 / s;
 *   q_j = e4m3(clamp(v_j * s, -MAX_FP8, MAX_FP8)).
 * All in fp32 (binary32 operations, each correctly rounded).
 */
static void quant_row(const float* v, int64_t n, const float* ub, uint8_t* q, float* scale_out) {
    float m = 0.0f;
    for (int64_t j = 0; j < n; ++j) {
        float a = fabsf(v[j]);
        if (a > m) m = a;
    }
    if (ub) {
        if (m < ORACLE_FP8_EPS) m = ORACLE_FP8_EPS;
        if (m > *ub) m = *ub;
    } else if (m < ORACLE_FP8_EPS) {
        m = ORACLE_FP8_EPS;
    }
    float s = ORACLE_FP8_MAX / m;
    *scale_out = 1.0f / s;
    for (int64_t j = 0; j < n; ++j) {
        float w = v[j] * s;
        if (w > ORACLE_FP8_MAX) w = ORACLE_FP8_MAX;
        if (w < -ORACLE_FP8_MAX) w = -ORACLE_FP8_MAX;
        q[j] = f32_to_e4m3(w);
    }
}

/* Per-row FP8 quantisation of an fp32 matrix (weights; the FP8 branch of
 * mslk/moe/layers.py keeps one fp32 scale per weight row, RoutedExperts.build). */
void oracle_quantize_rows(const float* w, int64_t rows, int64_t cols, const float* ub,
                          uint8_t* q, float* scale) {
#pragma omp parallel for schedule(static)
    for (int64_t r = 0; r < rows; ++r)
        quant_row(w + r * cols, cols, ub, q + r * cols, scale + r);
}

/* --------------------------------------------------------------- routing */

static float score_at(const void* scores, int dtype, int64_t st, int64_t se, int t, int e) {
    int64_t off = (int64_t)t * st + (int64_t)e * se;
    if (dtype == ORACLE_F32) return ((const float*)scores)[off];
    return bf16_to_f32(((const uint16_t*)scores)[off]);
}

/*
 * Top-k routing and the by-expert permutation (index_shuffling in
 * mslk/moe/layers.py, MetaShufflingMoE._route; the selection is torch.topk in
 * BaselineMoE._forward).
 *
 * For every valid token t < Tv, pick k experts one at a time: the not yet
 * picked expert with the largest score, the lower index on equal scores
 * (+0 and -0 are equal).  Then list the (expert, token) pairs in ascending
 * expert order and, within an expert, ascending token order: pair number r is
 * routed row r.
 *   counts[e]      = rows of expert e; counts[E] = Tv * k (the extra total
 *                    entry that layers.py slices off with token_counts[:E])
 *   offsets[e]     = first row of expert e (exclusive prefix sum); offsets[E] = Tv * k
 *   expert_indices[r], token_indices[r] = the pair of row r
 *   inv[t * k + j] = the j-th smallest row that belongs to token t (if inv)
 * Rows r >= Tv * k of the index arrays are not written.
 * Returns 0, or -1 when k is outside [1, E] or Tv outside [0, T].
 */
int oracle_route(const void* scores, int dtype, int64_t st, int64_t se, int T, int E, int k,
                 int Tv, int32_t* counts, int32_t* offsets, int32_t* expert_indices,
                 int32_t* token_indices, int32_t* inv) {
    if (k < 1 || k > E || Tv < 0 || Tv > T) return -1;
    int32_t* chosen = (int32_t*)malloc(sizeof(int32_t) * (size_t)(Tv > 0 ? Tv : 1) * (size_t)k);
    char* taken = (char*)malloc((size_t)E);
    for (int t = 0; t < Tv; ++t) {
        memset(taken, 0, (size_t)E);
        for (int j = 0; j < k; ++j) {
            int best = -1;
            for (int e = 0; e < E; ++e) {
                if (taken[e]) continue;
                if (best < 0 || score_at(scores, dtype, st, se, t, e) >
                                    score_at(scores, dtype, st, se, t, best))
                    best = e;
            }
            taken[best] = 1;
            chosen[(int64_t)t * k + j] = best;
        }
    }
    for (int e = 0; e <= E; ++e) counts[e] = 0;
    int row = 0;
    int32_t* seen = (int32_t*)calloc((size_t)(Tv > 0 ? Tv : 1), sizeof(int32_t));
    for (int e = 0; e < E; ++e) {
        offsets[e] = row;
        for (int t = 0; t < Tv; ++t) {
            for (int j = 0; j < k; ++j) {
                if (chosen[(int64_t)t * k + j] != e) continue;
                expert_indices[row] = e;
                token_indices[row] = t;
                if (inv) inv[(int64_t)t * k + seen[t]] = row;
                seen[t] += 1;
                counts[e] += 1;
                row += 1;
            }
        }
    }
    counts[E] = row;
    offsets[E] = row;
    free(seen);
    free(taken);
    free(chosen);
    return 0;
}

/* -------------------------------------------------------- gather + scale */

/*
 * mslk/moe/gather_scatter.py, kernel _mslk_gather_scale_dense_tokens:
 * for rows i < valid_rows, out[i, :] = x[token_indices[i], :] * scores[t, e],
 * with t = token_indices[i], e = expert_indices[i]; the product is taken in
 * fp32 and stored in x's dtype (bf16).  Rows i >= valid_rows are not written.
 */
void oracle_gather_scale(const uint16_t* x, int D, const int32_t* token_indices,
                         const int32_t* expert_indices, int valid_rows, const void* scores,
                         int dtype, int64_t st, int64_t se, uint16_t* out) {
#pragma omp parallel for schedule(static)
    for (int i = 0; i < valid_rows; ++i) {
        int t = token_indices[i], e = expert_indices[i];
        float s = score_at(scores, dtype, st, se, t, e);
        for (int d = 0; d < D; ++d)
            out[(int64_t)i * D + d] = f32_to_bf16(bf16_to_f32(x[(int64_t)t * D + d]) * s);
    }
}

/*
 * mslk/moe/gather_scatter.py, kernel _mslk_gather_scale_fp8_rowwise_quant_dense_tokens:
 * the fp32 row v = x[t, :] * scores[t, e] is quantised with quant_row (scale
 * bound ub when given).  Rows i >= valid_rows are not written.
 */
void oracle_gather_scale_quant(const uint16_t* x, int D, const int32_t* token_indices,
                               const int32_t* expert_indices, int valid_rows,
                               const void* scores, int dtype, int64_t st, int64_t se,
                               const float* ub, uint8_t* out, float* out_scale) {
#pragma omp parallel for schedule(static)
    for (int i = 0; i < valid_rows; ++i) {
        int t = token_indices[i], e = expert_indices[i];
        float s = score_at(scores, dtype, st, se, t, e);
        float* v = (float*)malloc(sizeof(float) * (size_t)D);
        for (int d = 0; d < D; ++d) v[d] = bf16_to_f32(x[(int64_t)t * D + d]) * s;
        quant_row(v, D, ub, out + (int64_t)i * D, out_scale + i);
        free(v);
    }
}

/* ---------------------------------------------------------- grouped GEMM */

/*
 * Grouped GEMM of mslk/moe/layers.py, MetaShufflingMoE._routed_expert:
 * grouped_gemm(x, w.view(-1, K), token_counts).  Expert e owns the rows
 * [off_e, off_e + counts[e]) of x (off_e = sum of the earlier counts) and the
 * weight rows w[e * N : (e + 1) * N, :] (each of length K), and
 *   y[r, n] = sum_k x[r, k] * w[e * N + n, k]
 * accumulated in fp64 over ascending k and rounded to bf16 once.
 * Rows past the last expert are not written.
 */
void oracle_grouped_gemm_bf16(const uint16_t* x, const uint16_t* w, const int32_t* counts,
                              int E, int N, int K, uint16_t* y) {
    int64_t off = 0;
    for (int e = 0; e < E; ++e) {
        int64_t cnt = counts[e];
#pragma omp parallel for collapse(2) schedule(static)
        for (int64_t r = off; r < off + cnt; ++r) {
            for (int n = 0; n < N; ++n) {
                const uint16_t* wr = w + ((int64_t)e * N + n) * K;
                const uint16_t* xr = x + r * K;
                double acc = 0.0;
                for (int kk = 0; kk < K; ++kk)
                    acc += (double)bf16_to_f32(xr[kk]) * (double)bf16_to_f32(wr[kk]);
                y[r * N + n] = f32_to_bf16((float)acc);
            }
        }
        off += cnt;
    }
}

/*
 * FP8-rowwise grouped GEMM (grouped_gemm_fp8_rowwise in _routed_expert), with
 * the dequantisation order of BaselineMoE._fake_quant: the product of the
 * decoded e4m3 operands, times the row's activation scale x_scale[r], times
 * the weight row's scale w_scale[e * N + n].  fp64, one rounding to bf16.
 */
void oracle_grouped_gemm_fp8(const uint8_t* x, const uint8_t* w, const int32_t* counts,
                             const float* x_scale, const float* w_scale, int E, int N, int K,
                             uint16_t* y) {
    int64_t off = 0;
    for (int e = 0; e < E; ++e) {
        int64_t cnt = counts[e];
#pragma omp parallel for collapse(2) schedule(static)
        for (int64_t r = off; r < off + cnt; ++r) {
            for (int n = 0; n < N; ++n) {
                const uint8_t* wr = w + ((int64_t)e * N + n) * K;
                const uint8_t* xr = x + r * K;
                double acc = 0.0;
                for (int kk = 0; kk < K; ++kk)
                    acc += (double)e4m3_to_f32(xr[kk]) * (double)e4m3_to_f32(wr[kk]);
                acc = acc * (double)x_scale[r] * (double)w_scale[(int64_t)e * N + n];
                y[r * N + n] = f32_to_bf16((float)acc);
            }
        }
        off += cnt;
    }
}

/* ------------------------------------------------------------ top-k finalize */

/*
 * Top-k finalize of an unfinalized MoE output (the single-GPU part of
 * AllReduceRMSNormWithReduceScatterEarlyExit.finalize on the "kimi_k3 ...
 * allreduce_rmsnorm_reduce_scatter_early_exit" page): the routing weights are
 * applied to the unweighted GEMM2 rows.  For every token t < M and column d:
 *   acc = 0; for slot j = 0 .. k-1: p = idx[t, j]; if p >= 0:
 *       acc = acc + w[t, j] * rows[p, d]          (fp32 multiply, fp32 add)
 *   r = bf16(acc), a negative zero written as +0
 *   out[t, d] = shared ? bf16(f32(r) + f32(shared[t, d])) : r
 * rows bf16 [n_rows, D]; w fp32 [M, k]; idx int32 [M, k]; shared bf16 [M, D] or NULL.
 * An index >= n_rows is skipped (the GPU flags it).
 */
void oracle_topk_finalize(const uint16_t* rows, int64_t n_rows, int D, const float* w, const int32_t* idx,
                          int M, int k, const uint16_t* shared, uint16_t* out) {
#pragma omp parallel for schedule(static)
    for (int t = 0; t < M; ++t) {
        for (int d = 0; d < D; ++d) {
            float acc = 0.0f;
            for (int j = 0; j < k; ++j) {
                const int32_t p = idx[(int64_t)t * k + j];
                if (p < 0 || p >= n_rows) continue;
                const float prod = w[(int64_t)t * k + j] * bf16_to_f32(rows[(int64_t)p * D + d]);
                acc = acc + prod;
            }
            uint16_t r = f32_to_bf16(acc);
            if (r == 0x8000u) r = 0; /* negative zero -> +0 */
            if (shared) r = f32_to_bf16(bf16_to_f32(r) + bf16_to_f32(shared[(int64_t)t * D + d]));
            out[(int64_t)t * D + d] = r;
        }
    }
}

/* ---------------------------------------------------------- router scores */

/*
 * Router scores of MetaShufflingMoE._route (the same two steps open
 * BaselineMoE._forward): scores = sigmoid(linear(tokens, router_DE.T)), both
 * in the model dtype, bf16.  The weight comes transposed, w[e, d] =
 * router_DE[d, e].  For each token t < valid_tokens and expert e:
 *   logit = bf16( sum_d x[t, d] * w[e, d] )      fp64 over ascending d
 *   score = bf16( 1 / (1 + e^-logit) )           fp64, from the bf16 logit
 * Rows t >= valid_tokens are not written.  `logits` may be NULL.
 */
void oracle_router_scores(const uint16_t* x, const uint16_t* w, int T, int D, int E, int valid_tokens,
                          uint16_t* scores, uint16_t* logits) {
    (void)T;
#pragma omp parallel for schedule(static)
    for (int t = 0; t < valid_tokens; ++t) {
        for (int e = 0; e < E; ++e) {
            const uint16_t* xr = x + (int64_t)t * D;
            const uint16_t* wr = w + (int64_t)e * D;
            double acc = 0.0;
            for (int d = 0; d < D; ++d)
                acc += (double)bf16_to_f32(xr[d]) * (double)bf16_to_f32(wr[d]);
            const uint16_t l = f32_to_bf16((float)acc);
            const double lv = (double)bf16_to_f32(l);
            scores[(int64_t)t * E + e] = f32_to_bf16((float)(1.0 / (1.0 + exp(-lv))));
            if (logits) logits[(int64_t)t * E + e] = l;
        }
    }
}

/* -------------------------------------------------------------- silu_mul */

/* z = y0 * sigmoid(y0) * y1 (BaselineMoE._forward), sigmoid(a) = 1 / (1 + e^-a), in fp64. */
static double silu_mul(double y0, double y1) { return y0 * (1.0 / (1.0 + exp(-y0))) * y1; }

/*
 * silu_mul(x0, x1) of MetaShufflingMoE._fused_silu_mul, with x0 = y[:, :H] and
 * x1 = y[:, H:] (row stride ld): z[r, j] = bf16(silu_mul(x0[r, j], x1[r, j]))
 * for rows r < valid_rows.
 */
void oracle_silu_mul(const uint16_t* x0, const uint16_t* x1, int64_t ld, int valid_rows, int H,
                     uint16_t* z) {
#pragma omp parallel for schedule(static)
    for (int r = 0; r < valid_rows; ++r)
        for (int j = 0; j < H; ++j)
            z[(int64_t)r * H + j] = f32_to_bf16((float)silu_mul(
                bf16_to_f32(x0[(int64_t)r * ld + j]), bf16_to_f32(x1[(int64_t)r * ld + j])));
}

/*
 * silu_mul_quant(x0, x1, scale_ub): the row of z, held in fp32, is quantised
 * with quant_row over its H entries.
 */
void oracle_silu_mul_quant(const uint16_t* x0, const uint16_t* x1, int64_t ld, int valid_rows,
                           int H, const float* ub, uint8_t* z, float* z_scale) {
#pragma omp parallel for schedule(static)
    for (int r = 0; r < valid_rows; ++r) {
        float* v = (float*)malloc(sizeof(float) * (size_t)H);
        for (int j = 0; j < H; ++j)
            v[j] = (float)silu_mul(bf16_to_f32(x0[(int64_t)r * ld + j]),
                                   bf16_to_f32(x1[(int64_t)r * ld + j]));
        quant_row(v, H, ub, z + (int64_t)r * H, z_scale + r);
        free(v);
    }
}

/* ----------------------------------------------------------- scatter-add */

/*
 * Combine (mslk/moe/gather_scatter.py, kernel _mslk_scatter_add_dense_tokens,
 * called by MetaShufflingMoE._combine_outputs): every routed row r <
 * valid_rows is added into out[token_indices[r], :].  The pages add in bf16
 * with relaxed atomics, so their order is unspecified; here each touched
 * token is accumulated in fp32, starting from its current out value and
 * adding its rows in ascending row order, then rounded to bf16 once.  Tokens
 * that receive no row are not written.
 */
void oracle_scatter_add(uint16_t* out, int T, int D, const uint16_t* in,
                        const int32_t* token_indices, int valid_rows) {
    float* acc = (float*)malloc(sizeof(float) * (size_t)T * (size_t)D);
    char* hit = (char*)calloc((size_t)T, 1);
    for (int r = 0; r < valid_rows; ++r) {
        int t = token_indices[r];
        if (!hit[t]) {
            hit[t] = 1;
            for (int d = 0; d < D; ++d) acc[(int64_t)t * D + d] = bf16_to_f32(out[(int64_t)t * D + d]);
        }
        for (int d = 0; d < D; ++d) acc[(int64_t)t * D + d] += bf16_to_f32(in[(int64_t)r * D + d]);
    }
    for (int t = 0; t < T; ++t)
        if (hit[t])
            for (int d = 0; d < D; ++d) out[(int64_t)t * D + d] = f32_to_bf16(acc[(int64_t)t * D + d]);
    free(hit);
    free(acc);
}
