/*
 * Plain CPU oracle for the routing + dispatch + per-expert grouped GEMM path.
 *
 * TEST INFRASTRUCTURE ONLY.  Nothing in the product library links, loads or
 * calls this file.  Only the test suite, the smoke check and the benchmark's
 * CPU-baseline leg use it.  It shares no code, header, table or constant with
 * the CUDA path.
 *
 * What it follows.  The articles on mKernel ("Conozca mKernel ..." on
 * 7minutos.es and its Arabic twin on k7ail.com), table "the five fused
 * kernels", row "MoE Dispatch + GEMM", describe the operation in one
 * sentence: route MoE tokens to their expert ranks (all-to-all) and run the
 * per-expert grouped GEMM in the same kernel, computing on tokens as soon as
 * they land.  The pages fix nothing finer than that.  Every step below is the
 * plain definition under the readings this library adopts (selection on the
 * logits, lower expert index wins ties, softmax over all experts, stable order
 * by token then slot inside each expert, rank-major expert-contiguous receive
 * rows, fp64 accumulation in ascending k order).
 *
 * Floating point: every sum is a plain left-to-right fp64 sum.  Build with
 * -ffp-contract=off so that no compiler fuses a product into an add.
 *
 * bf16 values are passed as their 16-bit patterns (uint16_t); a bf16 pattern
 * b is the fp32 number whose bit pattern is b << 16.
 */
#include <math.h>
#include <stdint.h>
#include <stdlib.h>
#include <string.h>

#define ORACLE_API __attribute__((visibility("default")))

static double bf16_to_double(uint16_t b) {
    uint32_t u = ((uint32_t)b) << 16;
    float f;
    memcpy(&f, &u, sizeof f);
    return (double)f;
}

/*
 * Step A1: top-k over the softmax of each token's router logits.
 *
 * Selection is made on the logits themselves (softmax is strictly increasing,
 * so the order is the same).  The j-th pick is the largest logit not yet
 * picked; between equal logits the lower expert index is picked first.  The
 * comparison is the float comparison, so -0.0 and +0.0 are equal.
 * Logits must be finite; the function returns -1 on a NaN.
 *
 * topk_w[t*k+j] = exp(L[t][e_j] - m_t) / sum_e exp(L[t][e] - m_t), with m_t
 * the row maximum: the softmax over all E experts, in fp64, with no
 * renormalisation over the k picks.
 */
ORACLE_API int oracle_topk(const float* logits, int T, int E, int k,
                           int32_t* topk_idx, double* topk_w) {
    if (T < 0 || E < 1 || k < 1 || k > E) return -2;
    unsigned char* taken = (unsigned char*)malloc((size_t)E);
    if (!taken) return -3;
    for (int t = 0; t < T; ++t) {
        const float* L = logits + (size_t)t * E;
        for (int e = 0; e < E; ++e)
            if (isnan(L[e])) { free(taken); return -1; }
        memset(taken, 0, (size_t)E);
        double m = (double)L[0];
        for (int e = 1; e < E; ++e)
            if ((double)L[e] > m) m = (double)L[e];
        double s = 0.0;
        for (int e = 0; e < E; ++e) s += exp((double)L[e] - m);
        for (int j = 0; j < k; ++j) {
            int best = -1;
            for (int e = 0; e < E; ++e) {
                if (taken[e]) continue;
                if (best < 0 || L[e] > L[best]) best = e;  /* strict: ties keep the lower index */
            }
            taken[best] = 1;
            topk_idx[(size_t)t * k + j] = best;
            topk_w[(size_t)t * k + j] = exp((double)L[best] - m) / s;
        }
    }
    free(taken);
    return 0;
}

/*
 * Step A1, renormalised variant (Mixtral-style gating): the gates are the
 * softmax over the k chosen logits only, so each token's k gates sum to 1.
 *   topk_w[t*k+j] = exp(L[t][e_j] - M_t) / sum_{j'<k} exp(L[t][e_j'] - M_t)
 * with e_j = topk_idx[t*k+j] (the picks of oracle_topk, unchanged) and M_t the
 * largest chosen logit.  fp64, j' ascending.  Returns -1 on an index outside
 * [0, E).
 */
ORACLE_API int oracle_topk_renorm_gates(const float* logits, int T, int E, int k,
                                        const int32_t* topk_idx, double* topk_w) {
    for (int t = 0; t < T; ++t) {
        const float* L = logits + (size_t)t * E;
        const int32_t* sel = topk_idx + (size_t)t * k;
        for (int j = 0; j < k; ++j)
            if (sel[j] < 0 || sel[j] >= E) return -1;
        double M = (double)L[sel[0]];
        for (int j = 1; j < k; ++j)
            if ((double)L[sel[j]] > M) M = (double)L[sel[j]];
        double s = 0.0;
        for (int j = 0; j < k; ++j) s += exp((double)L[sel[j]] - M);
        for (int j = 0; j < k; ++j)
            topk_w[(size_t)t * k + j] = exp((double)L[sel[j]] - M) / s;
    }
    return 0;
}

/*
 * Step A1 with a selection-only bias (the bias that auxiliary-loss-free load
 * balancing, as in DeepSeek-V3, moves between steps).  Expert e of token t is
 * ranked by the key  key[e] = (float)(L[t][e] + bias[e])  -- one fp32 addition,
 * rounded to nearest -- with the rule of oracle_topk on the keys (largest
 * first, lower index between equal keys, -0.0 equal to +0.0).  Only topk_idx
 * is produced; the gates come from the unbiased logits (oracle_gates_at).
 * Returns -1 on a NaN key.
 */
ORACLE_API int oracle_select_biased(const float* logits, const float* bias, int T, int E, int k,
                                    int32_t* topk_idx) {
    if (T < 0 || E < 1 || k < 1 || k > E) return -2;
    float* key = (float*)malloc(sizeof(float) * (size_t)E);
    unsigned char* taken = (unsigned char*)malloc((size_t)E);
    if (!key || !taken) { free(key); free(taken); return -3; }
    int rc = 0;
    for (int t = 0; t < T && rc == 0; ++t) {
        for (int e = 0; e < E; ++e) {
            volatile float sum = logits[(size_t)t * E + e] + bias[e];  /* stored: rounded to fp32 */
            key[e] = sum;
            if (isnan(key[e])) rc = -1;
        }
        memset(taken, 0, (size_t)E);
        for (int j = 0; j < k; ++j) {
            int best = -1;
            for (int e = 0; e < E; ++e) {
                if (taken[e]) continue;
                if (best < 0 || key[e] > key[best]) best = e;
            }
            taken[best] = 1;
            topk_idx[(size_t)t * k + j] = best;
        }
    }
    free(key);
    free(taken);
    return rc;
}

/*
 * Gates of given picks, from the unbiased logits, in fp64.
 *   sigmoid = 0: softmax over all E logits evaluated at the pick,
 *                exp(L[e_j] - m) / sum_e exp(L[e] - m), m the row maximum;
 *   sigmoid = 1: the logistic 1 / (1 + exp(-L[e_j])).
 *   renorm  = 1: then each token's k gates are divided by their sum
 *                (j ascending).
 * Returns -1 on an index outside [0, E).
 */
ORACLE_API int oracle_gates_at(const float* logits, const int32_t* topk_idx, int T, int E, int k,
                               int sigmoid, int renorm, double* topk_w) {
    for (int t = 0; t < T; ++t) {
        const float* L = logits + (size_t)t * E;
        const int32_t* sel = topk_idx + (size_t)t * k;
        double* w = topk_w + (size_t)t * k;
        for (int j = 0; j < k; ++j)
            if (sel[j] < 0 || sel[j] >= E) return -1;
        if (sigmoid) {
            for (int j = 0; j < k; ++j) w[j] = 1.0 / (1.0 + exp(-(double)L[sel[j]]));
        } else {
            double m = (double)L[0];
            for (int e = 1; e < E; ++e)
                if ((double)L[e] > m) m = (double)L[e];
            double s = 0.0;
            for (int e = 0; e < E; ++e) s += exp((double)L[e] - m);
            for (int j = 0; j < k; ++j) w[j] = exp((double)L[sel[j]] - m) / s;
        }
        if (renorm) {
            double z = 0.0;
            for (int j = 0; j < k; ++j) z += w[j];
            for (int j = 0; j < k; ++j) w[j] /= z;
        }
    }
    return 0;
}

/*
 * Step A2: per-expert histogram and its exclusive prefix sum.
 * counts[e] = number of (t, j) with topk_idx[t*k+j] == e;
 * offsets[0] = 0, offsets[e+1] = offsets[e] + counts[e].
 * Returns -1 if an index is outside [0, E).
 */
ORACLE_API int oracle_histogram(const int32_t* topk_idx, int T, int k, int E,
                                int32_t* counts, int32_t* offsets) {
    for (int e = 0; e < E; ++e) counts[e] = 0;
    for (long s = 0; s < (long)T * k; ++s) {
        int e = topk_idx[s];
        if (e < 0 || e >= E) return -1;
        counts[e] += 1;
    }
    offsets[0] = 0;
    for (int e = 0; e < E; ++e) offsets[e + 1] = offsets[e] + counts[e];
    return 0;
}

/*
 * Step A3: the stable permutation.  Destination rows are filled expert by
 * expert (ascending); inside one expert, by token (ascending) and then by
 * slot (ascending).  perm[row] = source slot t*k+j, dest[t*k+j] = row.
 */
ORACLE_API int oracle_permutation(const int32_t* topk_idx, int T, int k, int E,
                                  int32_t* perm, int32_t* dest) {
    long pos = 0;
    for (int e = 0; e < E; ++e)
        for (int t = 0; t < T; ++t)
            for (int j = 0; j < k; ++j)
                if (topk_idx[(size_t)t * k + j] == e) {
                    perm[pos] = t * k + j;
                    dest[(size_t)t * k + j] = (int32_t)pos;
                    ++pos;
                }
    return pos == (long)T * k ? 0 : -1;
}

/*
 * Receive-buffer split over R simulated expert ranks.  Rank r owns experts
 * [r*E/R, (r+1)*E/R); its rows are the global destination rows
 * [offsets[r*E/R], offsets[(r+1)*E/R]) in the same order, so row i of rank r's
 * buffer is global destination row rank_base[r] + i.  rank_base has R+1
 * entries; rank_base[R] = T*k.
 */
ORACLE_API int oracle_rank_base(const int32_t* offsets, int E, int R, int32_t* rank_base) {
    if (R < 1 || E % R != 0) return -1;
    for (int r = 0; r <= R; ++r) rank_base[r] = offsets[(size_t)r * (E / R)];
    return 0;
}

/*
 * Step A4: dispatch.  Destination row `row` receives a bit copy of the
 * token row x[perm[row] / k].  Rows are written in global destination order
 * (rank 0's rows first); the caller slices per rank with oracle_rank_base.
 */
ORACLE_API void oracle_gather(const uint16_t* x, int T, int d, int k,
                              const int32_t* perm, long S, uint16_t* rows) {
    (void)T;
    for (long row = 0; row < S; ++row) {
        int t = perm[row] / k;
        for (int i = 0; i < d; ++i) rows[(size_t)row * d + i] = x[(size_t)t * d + i];
    }
}

/*
 * Step A5: per-expert grouped GEMM on the destination rows.
 * For each expert e and each row in its segment [offsets[e], offsets[e+1]):
 *   Y[row][n] = sum_{i=0}^{d-1} rows[row][i] * W[e][i][n]
 * summed in fp64, i ascending.  W is [E][d][N] (N contiguous).
 * The loop visits i in the outer position with one fp64 accumulator per
 * output column; each Y element still sees its terms in ascending i.
 */
ORACLE_API int oracle_grouped_gemm(const uint16_t* rows, const uint16_t* W,
                                   const int32_t* offsets, int E, int d, int N,
                                   double* Y) {
    double* acc = (double*)malloc(sizeof(double) * (size_t)N);
    if (!acc) return -3;
    for (int e = 0; e < E; ++e) {
        const uint16_t* We = W + (size_t)e * d * N;
        for (long row = offsets[e]; row < offsets[e + 1]; ++row) {
            for (int n = 0; n < N; ++n) acc[n] = 0.0;
            for (int i = 0; i < d; ++i) {
                double a = bf16_to_double(rows[(size_t)row * d + i]);
                const uint16_t* wrow = We + (size_t)i * N;
                for (int n = 0; n < N; ++n) acc[n] += a * bf16_to_double(wrow[n]);
            }
            for (int n = 0; n < N; ++n) Y[(size_t)row * N + n] = acc[n];
        }
    }
    free(acc);
    return 0;
}

/*
 * One element of step A5, for sampled checks at full size:
 *   sum_{i<d} row[i] * We[i][n]   (fp64, i ascending)
 * `row` is one destination row (d values), `We` one expert's [d][N] matrix.
 */
ORACLE_API double oracle_gemm_entry(const uint16_t* row, const uint16_t* We,
                                    int d, int N, int n) {
    double acc = 0.0;
    for (int i = 0; i < d; ++i)
        acc += bf16_to_double(row[i]) * bf16_to_double(We[(size_t)i * N + n]);
    return acc;
}

/*
 * Gated expert activation (SwiGLU), applied to the up-projection output of
 * one destination row: G is [S][2F] with the gate projection in columns
 * [0, F) and the up projection in [F, 2F);
 *   H[i][f] = silu(G[i][f]) * G[i][F + f],   silu(g) = g / (1 + exp(-g)),
 * in fp64.
 */
ORACLE_API void oracle_swiglu(const double* G, long S, int F, double* H) {
    for (long i = 0; i < S; ++i)
        for (int f = 0; f < F; ++f) {
            const double g = G[(size_t)i * 2 * F + f];
            const double u = G[(size_t)i * 2 * F + F + f];
            H[(size_t)i * F + f] = g / (1.0 + exp(-g)) * u;
        }
}

/*
 * Rounding to bf16, round to nearest with ties to even, from fp64: the bf16
 * value is the nearest number of the form m * 2^q with |m| < 2^8 (8
 * significant bits) in bf16's exponent range; between two equally near, the
 * one with even m.  Values beyond the largest finite bf16 (after rounding)
 * become infinities; NaN becomes the quiet NaN 0x7FC0.  Subnormal bf16
 * results (|v| < 2^-126) are rounded on the fixed grid of spacing 2^-133.
 */
ORACLE_API void oracle_round_bf16(const double* v, long n, uint16_t* out) {
    for (long i = 0; i < n; ++i) {
        const double x = v[i];
        if (isnan(x)) { out[i] = 0x7FC0; continue; }
        const uint16_t sign = signbit(x) ? 0x8000 : 0;
        const double a = fabs(x);
        if (a == 0.0) { out[i] = sign; continue; }
        int q;
        (void)frexp(a, &q);            /* a = f * 2^q, 0.5 <= f < 1 */
        int e = q - 1;                 /* 2^e <= a < 2^(e+1) */
        if (e < -126) e = -126;        /* subnormal range: fixed spacing */
        const double ulp = ldexp(1.0, e - 7);
        double m = a / ulp;            /* exact: a power-of-two scaling */
        double r = floor(m);
        const double frac = m - r;
        if (frac > 0.5 || (frac == 0.5 && fmod(r, 2.0) != 0.0)) r += 1.0;
        const double y = r * ulp;      /* may reach 2^(e+1): still exact */
        if (y == 0.0) { out[i] = sign; continue; }  /* below half the smallest subnormal */
        if (y > 3.3895313892515355e38) { out[i] = sign | 0x7F80; continue; }  /* above bf16 max */
        /* encode y: exponent and 7 fraction bits */
        int qy;
        const double fy = frexp(y, &qy);
        int ey = qy - 1;
        uint16_t bits;
        if (ey < -126) {
            bits = (uint16_t)(y / ldexp(1.0, -133));      /* subnormal: m * 2^-133 */
        } else {
            const double mant = fy * 2.0 - 1.0;           /* in [0, 1) */
            bits = (uint16_t)(((ey + 127) << 7) | (int)(mant * 128.0));
        }
        out[i] = sign | bits;
    }
}

/*
 * Expert that owns destination row `row`: the e with
 * offsets[e] <= row < offsets[e+1] (a linear scan; empty experts are skipped
 * because their segment is empty).
 */
ORACLE_API int oracle_expert_of_row(const int32_t* offsets, int E, long row) {
    for (int e = 0; e < E; ++e)
        if (offsets[e] <= row && row < offsets[e + 1]) return e;
    return -1;
}

/*
 * Combine (the step after the path): undo the permutation and weight each
 * token's k expert outputs by its gates.
 *   out[t][n] = sum_{j<k} w[t*k+j] * Y[dest[t*k+j]][n]
 * summed in fp64, j ascending.  Y is [S][N] in destination order.
 */
ORACLE_API void oracle_combine(const double* Y, const double* w, const int32_t* dest,
                               int T, int k, int N, double* out) {
    for (int t = 0; t < T; ++t)
        for (int n = 0; n < N; ++n) {
            double acc = 0.0;
            for (int j = 0; j < k; ++j) {
                const long s = (long)t * k + j;
                acc += w[s] * Y[(size_t)dest[s] * N + n];
            }
            out[(size_t)t * N + n] = acc;
        }
}

/*
 * Router logits as this library's GPU router computes them (the step before
 * the path): for each token t and expert e,
 *   acc = 0; for i = 0..d-1 ascending: acc = fmaf(x[t][i], W_r[i][e], acc)
 *   L[t][e] = acc + bias[e]          (fp32 add; bias may be NULL)
 * fmaf is the correctly rounded fused multiply-add of C99 / IEEE 754, the
 * same operation as the GPU's; a bf16 x bf16 product is exact in fp32, so
 * each step is one rounding of (exact product + acc).
 */
ORACLE_API void oracle_router_logits(const uint16_t* x, const uint16_t* Wr, const float* bias,
                                     int T, int d, int E, float* L) {
    for (int t = 0; t < T; ++t)
        for (int e = 0; e < E; ++e) {
            float acc = 0.0f;
            for (int i = 0; i < d; ++i)
                acc = fmaf((float)bf16_to_double(x[(size_t)t * d + i]),
                           (float)bf16_to_double(Wr[(size_t)i * E + e]), acc);
            L[(size_t)t * E + e] = bias ? acc + bias[e] : acc;
        }
}
