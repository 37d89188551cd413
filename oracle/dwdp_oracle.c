/*
 * dwdp_oracle.c: plain, slow, fp64 CPU oracle of one DWDP MoE layer.
 *
 * TEST INFRASTRUCTURE ONLY.  The test suite, the package smoke check and the
 * benchmark's CPU-baseline leg are the only code that loads this library.  It
 * shares no code, header, table or helper with the CUDA path, and nothing in
 * the CUDA path loads it.
 *
 * Sources ("DWDP" = "DWDP: Distributed Weight Data Parallelism for
 * High-Performance LLM Inference on NVL72", read through its summary pages):
 *   - DWDP §2 (Methodology Overview): each rank keeps some experts resident and
 *     fetches the others from peers; where an expert's weights live changes
 *     nothing in what the layer computes.  Placement may be redundant.
 *   - DWDP §4.2 (Eliminating Split-Weight Merge Overhead): the grouped GEMM
 *     reads local and prefetched weights from separate buffers; again the
 *     result is the ordinary grouped GEMM's.
 * The pages do not print the router or the expert FFN.  This oracle takes the
 * plain reading of the workload they describe (a DeepSeek-R1-shaped MoE
 * block): softmax over all E experts, the k largest probabilities, weights
 * renormalised over the chosen k; each expert a SwiGLU FFN
 * (gate/up projection, SiLU(gate)*up, down projection); one optional shared
 * expert added with weight 1.
 *
 * Storage convention (shared with the inputs, not with any kernel): bf16 values
 * are passed as their 16-bit patterns.  x is [T][H].  The router weight is
 * stored [E][H] (row e holds column e of the math-layout H x E matrix).  One
 * expert's w13 is [2I][H]: rows 0..I-1 are W_gate transposed, rows I..2I-1 are
 * W_up transposed.  Its w2 is [H][I]: W_down transposed.  So, in math layout,
 * W_gate[h][i] = w13[i][h], W_up[h][i] = w13[I+i][h], W_down[i][h] = w2[h][i].
 *
 * Rounding points ("mirrored" mode, mirrored != 0): the activation a, each
 * expert's output y and the layer output are rounded to bf16 with
 * round-to-nearest-even; every other quantity stays in fp64.  With
 * mirrored == 0 ("strict" mode) nothing is rounded.
 *
 * ORACLE_MUTANT (compile-time, default 0) plants one known mistake; the test
 * suite builds each mutant and checks that its pins catch it.
 */
#include <math.h>
#include <stdint.h>
#include <stdlib.h>
#include <string.h>

#ifndef ORACLE_MUTANT
#define ORACLE_MUTANT 0
#endif

#ifdef _OPENMP
#include <omp.h>
#endif

/* ---------------------------------------------------------------- bf16 -- */

/* The bf16 value whose bit pattern is b (bf16 is the top half of an IEEE
 * binary32). */
double oracle_bf16_to_double(uint16_t b) {
    uint32_t u = ((uint32_t)b) << 16;
    float f;
    memcpy(&f, &u, sizeof f);
    return (double)f;
}

/* Round v to the nearest bf16 value, ties to even, straight from fp64 (no
 * detour through binary32, so no double rounding).  bf16 has an 8-bit
 * significand and binary32's exponent range; below 2^-126 the quantum stays
 * 2^-133 (subnormals).  Returns the bit pattern. */
uint16_t oracle_round_bf16(double v) {
    if (isnan(v)) return (uint16_t)0x7FC0;
    if (v == 0.0) return signbit(v) ? (uint16_t)0x8000 : (uint16_t)0x0000;
    double a = fabs(v);
    int e = ilogb(a);            /* 2^e <= a < 2^(e+1) */
    if (e < -126) e = -126;      /* subnormal range: fixed quantum */
    double q = ldexp(a, 7 - e);  /* significand scaled so the quantum is 1 */
#if ORACLE_MUTANT == 11
    double r = floor(q);         /* planted mistake: truncation */
#else
    double r = nearbyint(q);     /* default rounding mode: ties to even */
#endif
    double rounded = ldexp(r, e - 7);
    float f = (float)rounded;    /* exact: rounded has <= 8 significant bits */
    if (rounded > 3.3895313892515355e38) f = INFINITY;
    uint32_t u;
    memcpy(&u, &f, sizeof u);
    uint16_t bits = (uint16_t)(u >> 16);
    if (signbit(v)) bits |= 0x8000;
    return bits;
}

static double rb(double v) { return oracle_bf16_to_double(oracle_round_bf16(v)); }

/* ------------------------------------------------------------ routing -- */

/* Router logits z[t][e] = sum_h x[t][h] * Wr[h][e] (+ bias[e]), fp64.
 * bias may be NULL. */
void oracle_router_logits(const uint16_t* x, int64_t T, int64_t H,
                          const uint16_t* wr, int64_t E, const float* bias,
                          double* z) {
#pragma omp parallel for schedule(static)
    for (int64_t t = 0; t < T; ++t) {
        for (int64_t e = 0; e < E; ++e) {
            double s = 0.0;
            for (int64_t h = 0; h < H; ++h)
                s += oracle_bf16_to_double(x[t * H + h]) * oracle_bf16_to_double(wr[e * H + h]);
            if (bias) {
#if ORACLE_MUTANT == 10
                s -= (double)bias[e];  /* planted mistake: bias sign */
#else
                s += (double)bias[e];
#endif
            }
            z[t * E + e] = s;
        }
    }
}

/* Top-k selection and renormalised weights for each token.
 *
 * The choice of experts is an integer decision taken on floating point: it is
 * made on the logits rounded to binary32 (the precision a GPU router computes
 * its logits in) when decide_fp32 != 0, else on the fp64 logits.  Softmax is
 * monotone, so the k largest probabilities are the k largest logits.  Equal
 * values go to the lower expert id.  The chosen set is listed in ascending
 * expert id (slot j of token t is ids[t*k + j]).
 *
 * The weights are computed in fp64 from the fp64 logits: p = softmax(z) over
 * all E experts, then w_j = p_{e_j} / sum over the chosen set of p. */
void oracle_topk(const double* z, int64_t T, int64_t E, int64_t k, int decide_fp32,
                 int32_t* ids, double* w) {
#pragma omp parallel for schedule(static)
    for (int64_t t = 0; t < T; ++t) {
        const double* zt = z + t * E;
        char* taken = (char*)calloc((size_t)E, 1);
        for (int64_t j = 0; j < k; ++j) {
            int64_t best = -1;
            double bv = 0.0;
            for (int64_t e = 0; e < E; ++e) {
                if (taken[e]) continue;
                double v = decide_fp32 ? (double)(float)zt[e] : zt[e];
#if ORACLE_MUTANT == 4
                if (best < 0 || v >= bv) { best = e; bv = v; }  /* planted: ties to higher id */
#else
                if (best < 0 || v > bv) { best = e; bv = v; }
#endif
            }
            if (best < 0) break;  /* k > E: rejected by the caller */
            taken[best] = 1;
        }
        /* list the chosen set in ascending id */
        int64_t j = 0;
#if ORACLE_MUTANT == 12
        for (int64_t e = E - 1; e >= 0; --e)  /* planted: descending id */
#else
        for (int64_t e = 0; e < E; ++e)
#endif
            if (taken[e]) ids[t * k + (j++)] = (int32_t)e;
        free(taken);

        double zmax = zt[0];
        for (int64_t e = 1; e < E; ++e) if (zt[e] > zmax) zmax = zt[e];
        double denom = 0.0;
        for (int64_t e = 0; e < E; ++e) denom += exp(zt[e] - zmax);
        double psel = 0.0;
        for (int64_t jj = 0; jj < k; ++jj) psel += exp(zt[ids[t * k + jj]] - zmax) / denom;
        for (int64_t jj = 0; jj < k; ++jj) {
            double p = exp(zt[ids[t * k + jj]] - zmax) / denom;
#if ORACLE_MUTANT == 6
            w[t * k + jj] = p;  /* planted: no renormalisation */
#else
            w[t * k + jj] = p / psel;
#endif
        }
    }
}

/* Group the T*k (token, slot) pairs by expert.
 *   counts[e]   = number of pairs routed to e
 *   offsets     = exclusive scan of counts (E+1 entries; offsets[E] = T*k)
 *   perm[r]     = flat index f = t*k + j of the pair at grouped row r
 *   inv[f]      = grouped row of pair f
 * Within an expert's rows, pairs keep ascending flat index (a stable counting
 * sort).  The pages do not fix an order; this one is the library's documented
 * order (dwdp_route_out.perm), so grouped rows compare bit for bit. */
void oracle_group(const int32_t* ids, int64_t T, int64_t E, int64_t k,
                  int32_t* counts, int32_t* offsets, int32_t* perm, int32_t* inv) {
    int64_t n = T * k;
    for (int64_t e = 0; e < E; ++e) counts[e] = 0;
    for (int64_t f = 0; f < n; ++f) counts[ids[f]] += 1;
    offsets[0] = 0;
#if ORACLE_MUTANT == 8
    for (int64_t e = 0; e < E; ++e) offsets[e] = (e ? offsets[e - 1] : 0) + counts[e];  /* planted: inclusive */
    offsets[E] = (int32_t)n;
#else
    for (int64_t e = 0; e < E; ++e) offsets[e + 1] = offsets[e] + counts[e];
#endif
    int32_t* fill = (int32_t*)calloc((size_t)E, sizeof(int32_t));
#if ORACLE_MUTANT == 7
    for (int64_t f = n - 1; f >= 0; --f) {  /* planted: reversed order in a group */
#else
    for (int64_t f = 0; f < n; ++f) {
#endif
        int32_t e = ids[f];
        int32_t r = offsets[e] + fill[e];
        fill[e] += 1;
        if (r < 0 || r >= n) { inv[f] = -1; continue; }  /* only a broken scan gets here */
        perm[r] = (int32_t)f;
        inv[f] = r;
    }
    free(fill);
}

/* ---------------------------------------------------------------- FFN -- */

/* One expert on one token: g = x W_gate, u = x W_up, a = SiLU(g) * u,
 * y = a W_down, with SiLU(g) = g / (1 + exp(-g)).  fp64 sums; in mirrored
 * mode a and y are rounded to bf16.  a_tmp holds I doubles. */
static void expert_ffn(const uint16_t* xrow, int64_t H, int64_t I,
                       const uint16_t* w13, const uint16_t* w2, int mirrored,
                       double* a_tmp, double* y) {
    for (int64_t i = 0; i < I; ++i) {
        const uint16_t* wg = w13 + i * H;
        const uint16_t* wu = w13 + (I + i) * H;
        double g = 0.0, u = 0.0;
        for (int64_t h = 0; h < H; ++h) {
            double xv = oracle_bf16_to_double(xrow[h]);
            g += xv * oracle_bf16_to_double(wg[h]);
            u += xv * oracle_bf16_to_double(wu[h]);
        }
#if ORACLE_MUTANT == 1
        double a = g / (1.0 + exp(-g));            /* planted: up projection dropped */
#elif ORACLE_MUTANT == 2
        double a = g / (1.0 + exp(g)) * u;         /* planted: sign inside SiLU */
#elif ORACLE_MUTANT == 3
        double a = u / (1.0 + exp(-u)) * g;        /* planted: gate and up swapped */
#else
        double a = g / (1.0 + exp(-g)) * u;
#endif
        a_tmp[i] = mirrored ? rb(a) : a;
    }
    for (int64_t h = 0; h < H; ++h) {
        const uint16_t* wd = w2 + h * I;
        double s = 0.0;
        for (int64_t i = 0; i < I; ++i) s += a_tmp[i] * oracle_bf16_to_double(wd[i]);
        y[h] = mirrored ? rb(s) : s;
    }
}

/* Public single-expert entry (used by the pins). */
void oracle_expert_ffn(const uint16_t* xrow, int64_t H, int64_t I,
                       const uint16_t* w13, const uint16_t* w2, int mirrored, double* y) {
    double* a = (double*)malloc((size_t)I * sizeof(double));
    expert_ffn(xrow, H, I, w13, w2, mirrored, a, y);
    free(a);
}

/* The MoE output for n_sel tokens (rows tok[0..n_sel-1] of x), given their
 * routing (ids/w, k slots per token, indexed by token) and per-expert weight
 * pointers:
 *     out[s][:] = sum_j w[t][j] * y_{ids[t][j]}(x_t) + y_shared(x_t)
 * summed in fp64 in slot order, then the shared expert; rounded to bf16 in
 * mirrored mode.  expert_w13[e] / expert_w2[e] point at expert e's weights
 * wherever they live (the placement map resolved by the caller);
 * shared_w13 may be NULL (no shared expert). */
void oracle_moe_tokens(const uint16_t* x, int64_t H, int64_t I, int64_t k,
                       const int64_t* tok, int64_t n_sel,
                       const int32_t* ids, const double* w,
                       const uint16_t* const* expert_w13, const uint16_t* const* expert_w2,
                       const uint16_t* shared_w13, const uint16_t* shared_w2,
                       int mirrored, double* out) {
#pragma omp parallel
    {
        double* a = (double*)malloc((size_t)I * sizeof(double));
        double* y = (double*)malloc((size_t)H * sizeof(double));
        double* acc = (double*)malloc((size_t)H * sizeof(double));
#pragma omp for schedule(dynamic, 1)
        for (int64_t s = 0; s < n_sel; ++s) {
            int64_t t = tok[s];
            const uint16_t* xr = x + t * H;
            for (int64_t h = 0; h < H; ++h) acc[h] = 0.0;
            for (int64_t j = 0; j < k; ++j) {
                int32_t e = ids[t * k + j];
#if ORACLE_MUTANT == 9
                double wj = w[t * k + (j + 1) % k];  /* planted: wrong slot weight */
#else
                double wj = w[t * k + j];
#endif
                expert_ffn(xr, H, I, expert_w13[e], expert_w2[e], mirrored, a, y);
                for (int64_t h = 0; h < H; ++h) acc[h] += wj * y[h];
            }
#if ORACLE_MUTANT != 5
            if (shared_w13) {
                expert_ffn(xr, H, I, shared_w13, shared_w2, mirrored, a, y);
                for (int64_t h = 0; h < H; ++h) acc[h] += y[h];
            }
#endif
            for (int64_t h = 0; h < H; ++h) out[s * H + h] = mirrored ? rb(acc[h]) : acc[h];
        }
        free(a);
        free(y);
        free(acc);
    }
}

/* Threads the OpenMP runtime will use (1 without OpenMP). */
int oracle_num_threads(void) {
#ifdef _OPENMP
    return omp_get_max_threads();
#else
    return 1;
#endif
}

void oracle_set_num_threads(int n) {
#ifdef _OPENMP
    if (n > 0) omp_set_num_threads(n);
#else
    (void)n;
#endif
}

/* -------------------------------------------------------- grouped GEMM -- */

/* The grouped GEMM over split weight buffers (DWDP §4.2): for each group g,
 * rows r in [row_offsets[g], row_offsets[g+1]) of a [rows][K]:
 *   epilogue 0 or 2: d[r][n] = sum_k a[r][k] * B_g[n][k]              (n < N)
 *   epilogue 1:      d[r][n] = SiLU(sum_k a[r][k] B_g[n][k]) * sum_k a[r][k] B_g[N+n][k]
 * B_g points at group g's weights ([N][K], or [2N][K] for epilogue 1)
 * wherever they live.  fp64 sums; d is fp64 (the caller rounds or compares). */
void oracle_grouped_gemm(const uint16_t* a, int64_t K, const int32_t* row_offsets, int64_t G,
                         const uint16_t* const* b, int64_t N, int epilogue, double* d) {
    for (int64_t g = 0; g < G; ++g) {
        const uint16_t* bg = b[g];
#pragma omp parallel for schedule(static)
        for (int64_t r = row_offsets[g]; r < row_offsets[g + 1]; ++r) {
            for (int64_t n = 0; n < N; ++n) {
                double s = 0.0, s2 = 0.0;
                for (int64_t k = 0; k < K; ++k) {
                    double av = oracle_bf16_to_double(a[r * K + k]);
                    s += av * oracle_bf16_to_double(bg[n * K + k]);
                    if (epilogue == 1) s2 += av * oracle_bf16_to_double(bg[(N + n) * K + k]);
                }
                d[r * N + n] = (epilogue == 1) ? s / (1.0 + exp(-s)) * s2 : s;
            }
        }
    }
}

/* ------------------------------------------------------- FP8 (E4M3) -- */

/* The FP8 path (next row of the build, not on the pages, which run NVFP4
 * weights): expert weights are E4M3 codes with one scale per expert tensor;
 * activations are quantized per row (per token for x, per (token, expert)
 * row for a) to E4M3 with scale = amax / 448.
 *
 * E4M3 as used here: 1 sign bit, 4 exponent bits (bias 7), 3 mantissa bits;
 * no infinities; 0x7F / 0xFF are NaN; largest finite 448 = 1.75 * 2^8;
 * smallest normal 2^-6; subnormals are multiples of 2^-9.  Encoding rounds
 * to nearest, ties to even, and saturates to +-448 ("satfinite"). */
double oracle_e4m3_to_double(uint8_t b) {
    int s = b >> 7, e = (b >> 3) & 15, m = b & 7;
    double v;
    if (e == 15 && m == 7) return NAN;
    if (e == 0) v = ldexp((double)m, -9);
    else v = ldexp(1.0 + m / 8.0, e - 7);
    return s ? -v : v;
}

uint8_t oracle_e4m3_encode(double v) {
    if (isnan(v)) return 0x7F;
    uint8_t sign = signbit(v) ? 0x80 : 0x00;
    double a = fabs(v);
    double r;
    if (a >= 448.0) {
        r = 448.0;
    } else if (a == 0.0) {
        return sign;
    } else {
        int e = ilogb(a);
        if (e < -6) e = -6;                       /* subnormal range: quantum 2^-9 */
#if ORACLE_MUTANT == 13
        r = ldexp(floor(ldexp(a, 3 - e)), e - 3); /* planted: truncation */
#else
        r = ldexp(nearbyint(ldexp(a, 3 - e)), e - 3);
#endif
        if (r > 448.0) r = 448.0;
    }
    if (r == 0.0) return sign;
    int er = ilogb(r);
    if (er < -6) return sign | (uint8_t)(r / ldexp(1.0, -9));         /* subnormal */
    int mant = (int)((r / ldexp(1.0, er) - 1.0) * 8.0);
    return sign | (uint8_t)((er + 7) << 3) | (uint8_t)mant;
}

/* Quantize one row of n values (each a binary32 value) to E4M3 with
 * scale = amax / 448 computed in binary32 (1 when the row is all zero); each
 * code is the E4M3 encoding of the binary32 quotient v / scale.  Both
 * divisions are binary32 operations, as the kernels perform them, so the
 * codes are integer decisions taken in the kernels' precision. */
void oracle_quantize_row_e4m3(const float* v, int64_t n, uint8_t* codes, float* scale) {
    float amax = 0.0f;
    for (int64_t i = 0; i < n; ++i) {
        float a = fabsf(v[i]);
        if (a > amax) amax = a;
    }
#if ORACLE_MUTANT == 14
    float s = amax > 0.0f ? amax / 440.0f : 1.0f;   /* planted: wrong full-scale value */
#else
    float s = amax > 0.0f ? amax / 448.0f : 1.0f;
#endif
    for (int64_t i = 0; i < n; ++i) {
        volatile float q = v[i] / s;                 /* one binary32 rounding */
        codes[i] = oracle_e4m3_encode((double)q);
    }
    *scale = s;
}

/* One expert on one token with E4M3 weights (w13 [2I][H], w2 [H][I] codes,
 * per-tensor scales s13, s2): x is quantized per row, g and u are fp64 sums
 * of products of decoded codes times sx * s13, a = SiLU(g) * u (bf16 in
 * mirrored mode), a is quantized per row, y = fp64 sum times sa * s2 (bf16
 * in mirrored mode).  xq / sx are the token's quantized row, computed once
 * by the caller. */
static void expert_ffn_fp8(const uint8_t* xq, float sx, int64_t H, int64_t I, const uint8_t* w13, float s13,
                           const uint8_t* w2, float s2, int mirrored, float* a_tmp, uint8_t* aq_tmp, double* y) {
    for (int64_t i = 0; i < I; ++i) {
        const uint8_t* wg = w13 + i * H;
        const uint8_t* wu = w13 + (I + i) * H;
        double g = 0.0, u = 0.0;
        for (int64_t h = 0; h < H; ++h) {
            double xv = oracle_e4m3_to_double(xq[h]);
            g += xv * oracle_e4m3_to_double(wg[h]);
            u += xv * oracle_e4m3_to_double(wu[h]);
        }
#if ORACLE_MUTANT == 15
        g *= (double)s13;                          /* planted: activation scale dropped */
        u *= (double)s13;
#else
        g *= (double)sx * (double)s13;
        u *= (double)sx * (double)s13;
#endif
        double a = g / (1.0 + exp(-g)) * u;
        a_tmp[i] = (float)(mirrored ? rb(a) : a);
    }
    float sa;
    oracle_quantize_row_e4m3(a_tmp, I, aq_tmp, &sa);
    for (int64_t h = 0; h < H; ++h) {
        const uint8_t* wd = w2 + h * I;
        double s = 0.0;
        for (int64_t i = 0; i < I; ++i) s += oracle_e4m3_to_double(aq_tmp[i]) * oracle_e4m3_to_double(wd[i]);
        s *= (double)sa * (double)s2;
        y[h] = mirrored ? rb(s) : s;
    }
}

/* The FP8 layer for n_sel tokens: as oracle_moe_tokens, with E4M3 expert
 * weights and scales (w13_scale[e], w2_scale[e]; shared_* for the shared
 * expert, whose w13 may be NULL).  In strict mode (mirrored == 0) a is
 * quantized from its fp64 value rounded once to binary32. */
void oracle_moe_tokens_fp8(const uint16_t* x, int64_t H, int64_t I, int64_t k, const int64_t* tok, int64_t n_sel,
                           const int32_t* ids, const double* w, const uint8_t* const* expert_w13,
                           const uint8_t* const* expert_w2, const float* w13_scale, const float* w2_scale,
                           const uint8_t* shared_w13, const uint8_t* shared_w2, float shared_s13,
                           float shared_s2, int mirrored, double* out) {
#pragma omp parallel
    {
        float* xr = (float*)malloc((size_t)H * sizeof(float));
        uint8_t* xq = (uint8_t*)malloc((size_t)H);
        float* a = (float*)malloc((size_t)I * sizeof(float));
        uint8_t* aq = (uint8_t*)malloc((size_t)I);
        double* y = (double*)malloc((size_t)H * sizeof(double));
        double* acc = (double*)malloc((size_t)H * sizeof(double));
#pragma omp for schedule(dynamic, 1)
        for (int64_t s = 0; s < n_sel; ++s) {
            int64_t t = tok[s];
            for (int64_t h = 0; h < H; ++h) xr[h] = (float)oracle_bf16_to_double(x[t * H + h]);
            float sx;
            oracle_quantize_row_e4m3(xr, H, xq, &sx);
            for (int64_t h = 0; h < H; ++h) acc[h] = 0.0;
            for (int64_t j = 0; j < k; ++j) {
                int32_t e = ids[t * k + j];
                expert_ffn_fp8(xq, sx, H, I, expert_w13[e], w13_scale[e], expert_w2[e], w2_scale[e], mirrored, a, aq,
                               y);
                for (int64_t h = 0; h < H; ++h) acc[h] += w[t * k + j] * y[h];
            }
            if (shared_w13) {
                expert_ffn_fp8(xq, sx, H, I, shared_w13, shared_s13, shared_w2, shared_s2, mirrored, a, aq, y);
                for (int64_t h = 0; h < H; ++h) acc[h] += y[h];
            }
            for (int64_t h = 0; h < H; ++h) out[s * H + h] = mirrored ? rb(acc[h]) : acc[h];
        }
        free(xr);
        free(xq);
        free(a);
        free(aq);
        free(y);
        free(acc);
    }
}

/* ------------------------------------------------------------ NVFP4 -- */

/* The NVFP4 path (the pages run DeepSeek-R1 with NVFP4 MoE weights, DWDP
 * §5.1 Experimental Setup; they do not restate the format).  NVFP4 as
 * publicly defined: each value is an E2M1 code times an E4M3 scale shared by
 * a block of 16 consecutive elements along the contraction dimension, times
 * one binary32 scale for the whole tensor (weights: one per expert tensor;
 * activations here: one per row).
 *
 * E2M1: 1 sign bit, 2 exponent bits (bias 1), 1 mantissa bit; no infinities
 * or NaN.  Exponent field 0 is subnormal (0 or 0.5); otherwise
 * 2^(e-1) * (1 + m/2).  Magnitudes: 0, 0.5, 1, 1.5, 2, 3, 4, 6.  Codes are
 * passed one per byte (0..15) in math layout [rows][K]; block scales as
 * E4M3 codes [rows][K / 16]. */
double oracle_e2m1_to_double(uint8_t c) {
    int s = (c >> 3) & 1, e = (c >> 1) & 3, m = c & 1;
    double v = (e == 0) ? 0.5 * m : ldexp(1.0 + 0.5 * m, e - 1);
    return s ? -v : v;
}

/* Round to nearest E2M1 magnitude, ties to the even mantissa, saturating to
 * +-6; the sign is kept (a negative value that rounds to 0 gives code 8). */
uint8_t oracle_e2m1_encode(double v) {
    uint8_t sign = signbit(v) ? 8 : 0;
    double a = fabs(v);
    /* quantum: 0.5 below 2, 1 in [2, 4), 2 from 4 up */
    int q = (a < 2.0) ? -1 : (a < 4.0) ? 0 : 1;
#if ORACLE_MUTANT == 16
    double r = ldexp(round(ldexp(a, -q)), q);    /* planted: ties away from zero */
#else
    double r = ldexp(nearbyint(ldexp(a, -q)), q);
#endif
    if (r > 6.0) r = 6.0;
    if (r == 0.0) return sign;
    if (r == 0.5) return sign | 1;
    int e = ilogb(r) + 1;                         /* 1 for 1..1.5, 2 for 2..3, 3 for 4..6 */
    int m = (int)((r / ldexp(1.0, e - 1) - 1.0) * 2.0);
    return sign | (uint8_t)(e << 1) | (uint8_t)m;
}

/* Quantize one row of n binary32 values (n a multiple of 16) to NVFP4:
 *   s   = amax(row) / (6 * 448)           (1 for an all-zero row)
 *   d   = 6 * s
 *   sf  = E4M3(amax(block) / d)           per block of 16 (RNE, saturating)
 *   eff = E4M3 value of sf * s
 *   c   = E2M1(v / eff)                   (0 for every element when sf is 0)
 * Every operation is one binary32 operation, as a kernel performs it, so
 * each code is an integer decision taken in the kernel's precision.  The row's
 * largest element lands on E2M1 +-6 with block scale 448. */
void oracle_quantize_row_nvfp4(const float* v, int64_t n, uint8_t* codes, uint8_t* block_scales, float* scale) {
    float amax = 0.0f;
    for (int64_t i = 0; i < n; ++i) {
        float a = fabsf(v[i]);
        if (a > amax) amax = a;
    }
#if ORACLE_MUTANT == 17
    float s = amax > 0.0f ? amax / 448.0f : 1.0f;    /* planted: block range 6 forgotten */
#else
    float s = amax > 0.0f ? amax / 2688.0f : 1.0f;
#endif
    volatile float d = 6.0f * s;
    for (int64_t b = 0; b < n / 16; ++b) {
        float ab = 0.0f;
        for (int i = 0; i < 16; ++i) {
            float a = fabsf(v[b * 16 + i]);
            if (a > ab) ab = a;
        }
        volatile float q = ab / d;
        uint8_t sf = oracle_e4m3_encode((double)q);
        block_scales[b] = sf;
        double sfv = oracle_e4m3_to_double(sf);
        volatile float eff = (float)sfv * s;
        for (int i = 0; i < 16; ++i) {
            if (sfv == 0.0) {
                codes[b * 16 + i] = 0;
            } else {
                volatile float qq = v[b * 16 + i] / eff;
                codes[b * 16 + i] = oracle_e2m1_encode((double)qq);
            }
        }
    }
    *scale = s;
}

/* Dequantized NVFP4 element: E2M1 code times its block's E4M3 scale (the
 * tensor scale is applied by the caller). */
static double nvfp4_elem(const uint8_t* codes, const uint8_t* sf, int64_t i) {
#if ORACLE_MUTANT == 18
    return oracle_e2m1_to_double(codes[i]) * oracle_e4m3_to_double(sf[i / 32]);   /* planted: 32-wide blocks */
#else
    return oracle_e2m1_to_double(codes[i]) * oracle_e4m3_to_double(sf[i / 16]);
#endif
}

/* One expert on one token with NVFP4 weights: w13 codes [2I][H] with block
 * scales w13sf [2I][H/16] and tensor scale s13, w2 codes [H][I] with w2sf
 * [H][I/16] and s2.  The token's row arrives quantized (xq, xsf, sx).  g and u
 * are fp64 sums of dequantized products times sx * s13; a = SiLU(g) * u
 * (bf16 in mirrored mode) is quantized per row; y = fp64 sum times sa * s2
 * (bf16 in mirrored mode). */
static void expert_ffn_nvfp4(const uint8_t* xq, const uint8_t* xsf, float sx, int64_t H, int64_t I,
                             const uint8_t* w13, const uint8_t* w13sf, float s13, const uint8_t* w2,
                             const uint8_t* w2sf, float s2, int mirrored, float* a_tmp, uint8_t* aq, uint8_t* asf,
                             double* y) {
    for (int64_t i = 0; i < I; ++i) {
        const uint8_t* wg = w13 + i * H;
        const uint8_t* wu = w13 + (I + i) * H;
        const uint8_t* sg = w13sf + i * (H / 16);
        const uint8_t* su = w13sf + (I + i) * (H / 16);
        double g = 0.0, u = 0.0;
        for (int64_t h = 0; h < H; ++h) {
            double xv = nvfp4_elem(xq, xsf, h);
            g += xv * nvfp4_elem(wg, sg, h);
            u += xv * nvfp4_elem(wu, su, h);
        }
        g *= (double)sx * (double)s13;
        u *= (double)sx * (double)s13;
        double a = g / (1.0 + exp(-g)) * u;
        a_tmp[i] = (float)(mirrored ? rb(a) : a);
    }
    float sa;
    oracle_quantize_row_nvfp4(a_tmp, I, aq, asf, &sa);
    for (int64_t h = 0; h < H; ++h) {
        const uint8_t* wd = w2 + h * I;
        const uint8_t* sd = w2sf + h * (I / 16);
        double s = 0.0;
        for (int64_t i = 0; i < I; ++i) s += nvfp4_elem(aq, asf, i) * nvfp4_elem(wd, sd, i);
#if ORACLE_MUTANT == 19
        s *= (double)sa;                           /* planted: down-projection tensor scale dropped */
#else
        s *= (double)sa * (double)s2;
#endif
        y[h] = mirrored ? rb(s) : s;
    }
}

/* The NVFP4 layer for n_sel tokens: as oracle_moe_tokens, with NVFP4 expert
 * weights (codes, block scales and tensor scales per expert; shared_* for the
 * shared expert, whose w13 may be NULL).  H and I are multiples of 16.  In
 * strict mode (mirrored == 0) a is quantized from its fp64 value rounded once
 * to binary32. */
void oracle_moe_tokens_nvfp4(const uint16_t* x, int64_t H, int64_t I, int64_t k, const int64_t* tok,
                             int64_t n_sel, const int32_t* ids, const double* w, const uint8_t* const* w13,
                             const uint8_t* const* w13sf, const float* s13, const uint8_t* const* w2,
                             const uint8_t* const* w2sf, const float* s2, const uint8_t* shared_w13,
                             const uint8_t* shared_w13sf, float shared_s13, const uint8_t* shared_w2,
                             const uint8_t* shared_w2sf, float shared_s2, int mirrored, double* out) {
#pragma omp parallel
    {
        float* xr = (float*)malloc((size_t)H * sizeof(float));
        uint8_t* xq = (uint8_t*)malloc((size_t)H);
        uint8_t* xsf = (uint8_t*)malloc((size_t)H / 16 + 1);
        float* a = (float*)malloc((size_t)I * sizeof(float));
        uint8_t* aq = (uint8_t*)malloc((size_t)I);
        uint8_t* asf = (uint8_t*)malloc((size_t)I / 16 + 1);
        double* y = (double*)malloc((size_t)H * sizeof(double));
        double* acc = (double*)malloc((size_t)H * sizeof(double));
#pragma omp for schedule(dynamic, 1)
        for (int64_t s = 0; s < n_sel; ++s) {
            int64_t t = tok[s];
            for (int64_t h = 0; h < H; ++h) xr[h] = (float)oracle_bf16_to_double(x[t * H + h]);
            float sx;
            oracle_quantize_row_nvfp4(xr, H, xq, xsf, &sx);
            for (int64_t h = 0; h < H; ++h) acc[h] = 0.0;
            for (int64_t j = 0; j < k; ++j) {
                int32_t e = ids[t * k + j];
                expert_ffn_nvfp4(xq, xsf, sx, H, I, w13[e], w13sf[e], s13[e], w2[e], w2sf[e], s2[e], mirrored, a,
                                 aq, asf, y);
                for (int64_t h = 0; h < H; ++h) acc[h] += w[t * k + j] * y[h];
            }
            if (shared_w13) {
                expert_ffn_nvfp4(xq, xsf, sx, H, I, shared_w13, shared_w13sf, shared_s13, shared_w2, shared_w2sf,
                                 shared_s2, mirrored, a, aq, asf, y);
                for (int64_t h = 0; h < H; ++h) acc[h] += y[h];
            }
            for (int64_t h = 0; h < H; ++h) out[s * H + h] = mirrored ? rb(acc[h]) : acc[h];
        }
        free(xr);
        free(xq);
        free(xsf);
        free(a);
        free(aq);
        free(asf);
        free(y);
        free(acc);
    }
}

/* One NVFP4 linear layer on rows that arrive already quantized (the second
 * half of expert_ffn_nvfp4 on its own, and its first half with
 * epilogue 1), so a caller can check each GEMM of the NVFP4 layer given
 * the codes its input rows really had:
 *   epilogue 0:  out[r][c] = (sum_k A[r][k] W[c][k]) * row_scale[r] * w_scale
 *   epilogue 1:  g = the same with W's row c, u = with W's row N + c,
 *                out[r][c] = SiLU(g) * u                  (W has 2N rows)
 * with A[r][k] = E2M1(codes[r][k]) * E4M3(sf[r][k / 16]) and W likewise
 * (w codes [N or 2N][K], wsf [.][K / 16]); fp64 sums, rounded to bf16 in
 * mirrored mode. */
void oracle_nvfp4_linear(const uint8_t* codes, const uint8_t* sf, const float* row_scale, int64_t n, int64_t K,
                         const uint8_t* w, const uint8_t* wsf, float w_scale, int64_t N, int epilogue, int mirrored,
                         double* out) {
#pragma omp parallel for schedule(dynamic, 1)
    for (int64_t r = 0; r < n; ++r) {
        const uint8_t* a = codes + r * K;
        const uint8_t* as = sf + r * (K / 16);
#if ORACLE_MUTANT == 20
        const double sc = (double)w_scale;                        /* planted: row scale dropped */
#else
        const double sc = (double)row_scale[r] * (double)w_scale;
#endif
        for (int64_t c = 0; c < N; ++c) {
            double s = 0.0;
            for (int64_t k = 0; k < K; ++k) s += nvfp4_elem(a, as, k) * nvfp4_elem(w + c * K, wsf + c * (K / 16), k);
            s *= sc;
            if (epilogue == 1) {
                double u = 0.0;
                const uint8_t* wu = w + (N + c) * K;
                const uint8_t* su = wsf + (N + c) * (K / 16);
                for (int64_t k = 0; k < K; ++k) u += nvfp4_elem(a, as, k) * nvfp4_elem(wu, su, k);
                u *= sc;
                s = s / (1.0 + exp(-s)) * u;
            }
            out[r * N + c] = mirrored ? rb(s) : s;
        }
    }
}

/* One E4M3 linear layer on rows that arrive already quantized (the halves
 * of expert_ffn_fp8 on their own, so a caller can check each GEMM of the
 * E4M3 layer given the codes its input rows really had):
 *   epilogue 0:  out[r][c] = (sum_k E4M3(codes[r][k]) E4M3(w[c][k])) * row_scale[r] * w_scale
 *   epilogue 1:  g = the same with W's row c, u = with W's row N + c,
 *                out[r][c] = SiLU(g) * u                  (w has 2N rows)
 * fp64 sums, rounded to bf16 in mirrored mode. */
void oracle_e4m3_linear(const uint8_t* codes, const float* row_scale, int64_t n, int64_t K, const uint8_t* w,
                        float w_scale, int64_t N, int epilogue, int mirrored, double* out) {
#pragma omp parallel for schedule(dynamic, 1)
    for (int64_t r = 0; r < n; ++r) {
        const uint8_t* a = codes + r * K;
#if ORACLE_MUTANT == 21
        const double sc = (double)row_scale[r];                  /* planted: weight scale dropped */
#else
        const double sc = (double)row_scale[r] * (double)w_scale;
#endif
        for (int64_t c = 0; c < N; ++c) {
            double s = 0.0, u = 0.0;
            for (int64_t k = 0; k < K; ++k) {
                const double av = oracle_e4m3_to_double(a[k]);
                s += av * oracle_e4m3_to_double(w[c * K + k]);
                if (epilogue == 1) u += av * oracle_e4m3_to_double(w[(N + c) * K + k]);
            }
            s *= sc;
            if (epilogue == 1) {
                u *= sc;
                s = s / (1.0 + exp(-s)) * u;
            }
            out[r * N + c] = mirrored ? rb(s) : s;
        }
    }
}
