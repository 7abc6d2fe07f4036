/*
 * moe_oracle.c -- plain, slow CPU oracle for the forward pass of one
 * top-k-routed SwiGLU mixture-of-experts layer.
 *
 * TEST INFRASTRUCTURE ONLY.  Nothing on the product path links, loads or
 * calls this file: only the test suite, the smoke check and the bench's CPU
 * baseline leg use it.  It shares no code, header, table or helper with the
 * CUDA library; the two meet only through the seeded input tensors.
 *
 * Sources (web pages; section names as printed there):
 *   [MoE-vLLM]  "Mixture of Experts in vLLM - From First Principles to
 *               fused_moe": sections "An expert is a small SwiGLU MLP",
 *               "One token uses only 8 experts", "A batch: (token, expert)
 *               pairs", "Group by expert", "The two index lists",
 *               "Put the results back, and combine them per token",
 *               "The rest of the layer stays in pair order".
 *
 * Arithmetic: every sum and product is taken in IEEE double; values are
 * rounded to bfloat16 (round to nearest, ties to even) at the four points the
 * layer stores in bf16: router logits, the GEMM-1 output h, the activation a
 * and the layer output y.  The pages fix no accumulation precision; a double
 * sum of products of bf16 values is the exact sum up to 2^-53 relative in any
 * order, so this oracle does not depend on how a device orders or splits its
 * sums, and a comparison measures the device's own rounding alone.  The GEMM-2 output o is not rounded.  Top-k is
 * decided on the bf16 logits themselves (softmax is monotone), ties going to
 * the lower expert id.
 *
 * Parity status: every function here is pinned by the CPU tests (bf16
 * rounding against a brute-force nearest search and torch casts, top-k
 * against a stable lexsort, align against the worked example on the vLLM
 * page and a stable argsort, the expert MLP against dense expansions and
 * closed forms).  The output values y of a full layer carry no worked
 * numbers on the pages; they are pinned only through those reductions.
 *
 * Data types: bf16 tensors are passed as their raw 16-bit patterns
 * (uint16_t).  All tensors are dense and row-major.
 */
#include <math.h>
#include <stdint.h>
#include <stdlib.h>
#include <string.h>
#ifdef _OPENMP
#include <omp.h>
#endif

typedef uint16_t bf16_t;

/* ---------------------------------------------------------------- bf16 -- */

/* A bf16 pattern is the upper half of an IEEE binary32 pattern. */
double oracle_bf16_to_double(bf16_t b)
{
    uint32_t u = (uint32_t)b << 16;
    float f;
    memcpy(&f, &u, sizeof f);
    return (double)f;
}

/* Round a double to the nearest bf16 value, ties to the even significand.
 * bf16 has 8 significant bits and the binary32 exponent range, so in the
 * binade [2^(ex-1), 2^ex) the spacing of bf16 values is 2^(ex-8); below the
 * smallest normal (2^-126) the spacing is the subnormal step 2^-133.  The
 * value is scaled by a power of two (exact), rounded to an integer with
 * nearbyint (ties to even in the default rounding mode) and scaled back. */
bf16_t oracle_bf16_round(double v)
{
    if (isnan(v))
        return 0x7FC0;
    if (isinf(v))
        return v > 0 ? 0x7F80 : 0xFF80;
    const int neg = signbit(v) ? 1 : 0;
    const double a = fabs(v);
    if (a == 0.0)
        return neg ? 0x8000 : 0x0000;
    int ex;
    (void)frexp(a, &ex);                 /* a in [2^(ex-1), 2^ex) */
    int q = ex - 8;                      /* exponent of one bf16 ulp here */
    if (q < -133)
        q = -133;
    const double r = ldexp(nearbyint(ldexp(a, -q)), q);
    if (r > 3.3895313892515355e38)       /* (2 - 2^-7) * 2^127, largest finite bf16 */
        return neg ? 0xFF80 : 0x7F80;
    const float f = (float)r;            /* exact: r has <= 8 significant bits */
    uint32_t u;
    memcpy(&u, &f, sizeof u);
    return (bf16_t)((u >> 16) | (neg ? 0x8000u : 0u));
}

/* Element-wise oracle_bf16_round over an array. */
void oracle_bf16_round_array(const double *v, long n, bf16_t *out)
{
    for (long i = 0; i < n; ++i)
        out[i] = oracle_bf16_round(v[i]);
}

static double bf(bf16_t b) { return oracle_bf16_to_double(b); }

/* ------------------------------------------------------------- threads -- */

void oracle_set_threads(int n)
{
#ifdef _OPENMP
    if (n > 0)
        omp_set_num_threads(n);
#else
    (void)n;
#endif
}

int oracle_get_threads(void)
{
#ifdef _OPENMP
    return omp_get_max_threads();
#else
    return 1;
#endif
}

/* ------------------------------------------------------- router logits -- */

/* [MoE-vLLM] "One token uses only 8 experts": the router is one linear layer
 * W_r [E, H] giving one score per expert.
 *   logits[t, e] = bf16( sum_h x[t, h] * W_r[e, h]  + bias[e] )
 * bias (nullable, fp32 [E]) is a per-expert offset added before rounding. */
void oracle_router_logits(const bf16_t *x, const bf16_t *w_r, const float *bias,
                          int M, int E, int H, bf16_t *logits)
{
#pragma omp parallel for schedule(static)
    for (int t = 0; t < M; ++t) {
        for (int e = 0; e < E; ++e) {
            double acc = 0.0;
            for (int h = 0; h < H; ++h)
                acc += bf(x[(size_t)t * H + h]) * bf(w_r[(size_t)e * H + h]);
            if (bias)
                acc += (double)bias[e];
            logits[(size_t)t * E + e] = oracle_bf16_round(acc);
        }
    }
}

/* ---------------------------------------------- softmax, top-k, renorm -- */

/* [MoE-vLLM] "One token uses only 8 experts", steps 1-3: softmax over the E
 * scores, keep the top_k largest, and (renormalize) rescale the kept weights
 * so that they add up to 1.
 *   slot j of token t holds the j-th largest logit (slot 0 = largest); equal
 *   logits are ordered by ascending expert id.
 *   p_e = exp(l_e - max l) / sum_e' exp(l_e' - max l)     over all E experts
 *   w_j = p_{id_j} / sum_j' p_{id_j'}   if renormalize,   else w_j = p_{id_j}
 * The weights are returned as float (the layer's topk_weights dtype).
 * Inputs are assumed finite. */
void oracle_topk_softmax(const bf16_t *logits, int M, int E, int top_k,
                         int renormalize, int32_t *topk_ids, float *topk_weights)
{
#pragma omp parallel
    {
        char *taken = (char *)malloc((size_t)E);
        double *p = (double *)malloc(sizeof(double) * (size_t)E);
#pragma omp for schedule(static)
        for (int t = 0; t < M; ++t) {
            const bf16_t *l = logits + (size_t)t * E;
            memset(taken, 0, (size_t)E);
            for (int j = 0; j < top_k; ++j) {
                int best = -1;
                for (int e = 0; e < E; ++e) {
                    if (taken[e])
                        continue;
                    /* strict '>' keeps the lower id among equal values */
                    if (best < 0 || bf(l[e]) > bf(l[best]))
                        best = e;
                }
                taken[best] = 1;
                topk_ids[(size_t)t * top_k + j] = best;
            }
            double m = bf(l[0]);
            for (int e = 1; e < E; ++e)
                if (bf(l[e]) > m)
                    m = bf(l[e]);
            double den = 0.0;
            for (int e = 0; e < E; ++e) {
                p[e] = exp(bf(l[e]) - m);
                den += p[e];
            }
            for (int e = 0; e < E; ++e)
                p[e] /= den;
            double kept = 0.0;
            for (int j = 0; j < top_k; ++j)
                kept += p[topk_ids[(size_t)t * top_k + j]];
            for (int j = 0; j < top_k; ++j) {
                double w = p[topk_ids[(size_t)t * top_k + j]];
                if (renormalize)
                    w /= kept;
                topk_weights[(size_t)t * top_k + j] = (float)w;
            }
        }
        free(p);
        free(taken);
    }
}

/* --------------------------------------------------------------- align -- */

/* Padded capacity of sorted_token_ids: every expert can add at most B-1 pad
 * entries, rounded up to whole blocks. */
long oracle_align_capacity(int M, int top_k, int E, int B)
{
    long P = (long)M * top_k;
    long cap = P + (long)E * (B - 1);
    return (cap + B - 1) / B * B;
}

/* [MoE-vLLM] "A batch: (token, expert) pairs": pair id p = t * top_k + j.
 * "Group by expert" and "The two index lists": sorted_token_ids holds the pair
 * ids grouped by expert; each expert's group is padded up to a multiple of
 * BLOCK_SIZE_M (B) with the id P = M * top_k, which is no real pair;
 * expert_ids holds one expert id per block of B entries.
 * Readings where the page leaves a choice: experts are laid out in ascending
 * id; inside a group the pairs are in ascending pair id (the page says the
 * order is not fixed); an expert with no pairs gets no block.
 * Outputs: sorted_token_ids [cap] (entries from n_post on are set to P),
 * expert_ids [cap / B] (blocks from n_post / B on are set to -1),
 * expert_offsets [E + 1] (start of each expert's padded group; the last entry
 * is n_post), *num_tokens_post_padded = n_post.
 * Returns 0, or -1 if some id lies outside [0, E). */
int oracle_align_block_size(const int32_t *topk_ids, int M, int top_k, int E, int B,
                            int32_t *sorted_token_ids, int32_t *expert_ids,
                            int32_t *expert_offsets, int32_t *num_tokens_post_padded)
{
    const long P = (long)M * top_k;
    const long cap = oracle_align_capacity(M, top_k, E, B);
    for (long p = 0; p < P; ++p)
        if (topk_ids[p] < 0 || topk_ids[p] >= E)
            return -1;
    for (long i = 0; i < cap; ++i)
        sorted_token_ids[i] = (int32_t)P;
    for (long b = 0; b < cap / B; ++b)
        expert_ids[b] = -1;
    long out = 0;
    for (int e = 0; e < E; ++e) {
        expert_offsets[e] = (int32_t)out;
        long n_e = 0;
        for (long p = 0; p < P; ++p) {
            if (topk_ids[p] == e) {
                sorted_token_ids[out + n_e] = (int32_t)p;
                ++n_e;
            }
        }
        const long padded = (n_e + B - 1) / B * B;
        for (long b = out / B; b < (out + padded) / B; ++b)
            expert_ids[b] = e;
        out += padded;
    }
    expert_offsets[E] = (int32_t)out;
    *num_tokens_post_padded = (int32_t)out;
    return 0;
}

/* ---------------------------------------------------------- expert MLP -- */

/* [MoE-vLLM] "An expert is a small SwiGLU MLP": W13 [2I, H] stacks the gate
 * rows (first I) over the up rows (last I); h = W13 x; a = SiLU(h_gate) * h_up.
 * "The rest of the layer stays in pair order": row p of the activation
 * belongs to pair p.  For every pair p = t * top_k + j with e = topk_ids[p]:
 *   h[n] = bf16( sum_k x[t, k] * W13[e][n][k] )            n < 2I
 *   a[p, i] = bf16( SiLU(h[i]) * h[I + i] ),   SiLU(z) = z / (1 + exp(-z))
 * w13 is [E, 2I, H]; a is [M * top_k, I]. */
void oracle_expert_act(const bf16_t *x, const bf16_t *w13, const int32_t *topk_ids,
                       int M, int top_k, int E, int H, int I, bf16_t *a)
{
    (void)E;
#pragma omp parallel
    {
        double *h = (double *)malloc(sizeof(double) * 2 * (size_t)I);
#pragma omp for schedule(static)
        for (long p = 0; p < (long)M * top_k; ++p) {
            const long t = p / top_k;
            const int e = topk_ids[p];
            const bf16_t *W = w13 + (size_t)e * 2 * I * H;
            for (int n = 0; n < 2 * I; ++n) {
                double acc = 0.0;
                for (int k = 0; k < H; ++k)
                    acc += bf(x[(size_t)t * H + k]) * bf(W[(size_t)n * H + k]);
                h[n] = bf(oracle_bf16_round(acc));
            }
            for (int i = 0; i < I; ++i) {
                const double g = h[i];
                const double silu = g / (1.0 + exp(-g));
                a[(size_t)p * I + i] = oracle_bf16_round(silu * h[I + i]);
            }
        }
        free(h);
    }
}

/* [MoE-vLLM] "An expert is a small SwiGLU MLP" step 3 (o = W2 a, W2 [H, I]),
 * "One token uses only 8 experts" step 5 and "Put the results back, and
 * combine them per token": y = sum_j w_j f_{id_j}(x), one row per token.
 *   o_{p}[n] = sum_i a[p, i] * W2[e][n][i]           (not rounded)
 *   y[t, n]  = bf16( sum_j topk_weights[t, j] * o_{t*top_k + j}[n]
 *                    + residual[t, n] )               (residual nullable)
 * w2 is [E, H, I]; y is [M, H]. */
void oracle_expert_down_combine(const bf16_t *a, const bf16_t *w2, const int32_t *topk_ids,
                                const float *topk_weights, const bf16_t *residual,
                                int M, int top_k, int E, int H, int I, bf16_t *y)
{
    (void)E;
#pragma omp parallel for schedule(static)
    for (int t = 0; t < M; ++t) {
        for (int n = 0; n < H; ++n) {
            double acc = 0.0;
            for (int j = 0; j < top_k; ++j) {
                const long p = (long)t * top_k + j;
                const bf16_t *W = w2 + (size_t)topk_ids[p] * H * I + (size_t)n * I;
                double o = 0.0;
                for (int i = 0; i < I; ++i)
                    o += bf(a[(size_t)p * I + i]) * bf(W[i]);
                acc += (double)topk_weights[p] * o;
            }
            if (residual)
                acc += bf(residual[(size_t)t * H + n]);
            y[(size_t)t * H + n] = oracle_bf16_round(acc);
        }
    }
}

/* ----------------------------------------------------------- the layer -- */

/* The whole layer, token by token: router logits (or the given logits),
 * softmax / top-k / renormalize, the chosen experts' SwiGLU MLPs and the
 * weighted combine.  Exactly one of w_router and router_logits is non-NULL.
 * topk_ids_out / topk_weights_out / logits_out are optional outputs.
 * The grouping by expert changes only the order of the work, not the
 * result ([MoE-vLLM] "Put the results back"), so the oracle skips it.
 * Returns 0, or -1 on bad arguments. */
int oracle_moe_forward(const bf16_t *x, const bf16_t *w_router, const bf16_t *router_logits,
                       const float *router_bias, const bf16_t *w13, const bf16_t *w2,
                       const bf16_t *residual, int M, int E, int top_k, int H, int I,
                       int renormalize, bf16_t *y, int32_t *topk_ids_out,
                       float *topk_weights_out, bf16_t *logits_out)
{
    if ((w_router == NULL) == (router_logits == NULL))
        return -1;
    if (M < 0 || E < 1 || top_k < 1 || top_k > E || H < 1 || I < 1)
        return -1;
    if (M == 0)
        return 0;
    const size_t P = (size_t)M * top_k;
    bf16_t *logits = (bf16_t *)malloc(sizeof(bf16_t) * (size_t)M * E);
    int32_t *ids = (int32_t *)malloc(sizeof(int32_t) * P);
    float *w = (float *)malloc(sizeof(float) * P);
    bf16_t *a = (bf16_t *)malloc(sizeof(bf16_t) * P * I);
    if (!logits || !ids || !w || !a) {
        free(logits); free(ids); free(w); free(a);
        return -1;
    }
    if (w_router)
        oracle_router_logits(x, w_router, router_bias, M, E, H, logits);
    else
        memcpy(logits, router_logits, sizeof(bf16_t) * (size_t)M * E);
    oracle_topk_softmax(logits, M, E, top_k, renormalize, ids, w);
    oracle_expert_act(x, w13, ids, M, top_k, E, H, I, a);
    oracle_expert_down_combine(a, w2, ids, w, residual, M, top_k, E, H, I, y);
    if (topk_ids_out)
        memcpy(topk_ids_out, ids, sizeof(int32_t) * P);
    if (topk_weights_out)
        memcpy(topk_weights_out, w, sizeof(float) * P);
    if (logits_out)
        memcpy(logits_out, logits, sizeof(bf16_t) * (size_t)M * E);
    free(logits); free(ids); free(w); free(a);
    return 0;
}


/* ------------------------------------------------------ FP8 (E4M3) path -- */

/* [MoE-vLLM] "fused_experts_impl": for FP8 models the GEMM-1 input is the
 * quantized copy of x (qhidden_states), and one kernel serves bf16 and FP8
 * weights.  The page gives no format details; the readings taken here (the
 * same on the device):
 *   - FP8 is E4M3 (1 sign, 4 exponent bits with bias 7, 3 mantissa bits; no
 *     infinities; 0x7F / 0xFF are NaN; largest finite 448), converted from a
 *     value by rounding to nearest, ties to even, saturating at +-448;
 *   - weights are stored as E4M3 codes with one fp32 scale per output row
 *     (per output channel): W[e][n][k] ~ s_w[e][n] * q_w[e][n][k];
 *   - activations are quantized per row (per token for x, per pair for the
 *     GEMM-1 output a) with a dynamic scale s = amax / 448 (1 for an all-zero
 *     row) and codes q = e4m3(v / s); amax, the scale and v / s are taken in
 *     fp32 with correctly rounded division, the precision the device uses,
 *     so that both sides decide every code the same way;
 *   - dequantization happens after the sums:
 *       h[n] = bf16( s_x[t] * s_w[e][n] * sum_k e4m3(q_x[t,k]) e4m3(q_w[e][n,k]) )
 *       o[n] =       s_a[p] * s_w2[e][n] * sum_i e4m3(q_a[p,i]) e4m3(q_w2[e][n,i])
 *     with the bf16 rounding points of the bf16 layer (h, a, y).  */

/* Value of an E4M3 code. */
double oracle_e4m3_to_double(uint8_t c)
{
    const int neg = (c >> 7) & 1, ex = (c >> 3) & 15, m = c & 7;
    double v;
    if (ex == 15 && m == 7)
        return NAN;
    if (ex == 0)
        v = ldexp((double)m, -9);               /* subnormal: m/8 * 2^-6 */
    else
        v = ldexp(8.0 + m, ex - 7 - 3);         /* (1 + m/8) * 2^(ex-7) */
    return neg ? -v : v;
}

/* The E4M3 code nearest to v (ties to the even code), saturating at +-448. */
uint8_t oracle_e4m3_round(double v)
{
    if (isnan(v))
        return 0x7F;
    const int neg = signbit(v) ? 1 : 0;
    double a = fabs(v);
    uint8_t code;
    if (a >= 448.0) {
        code = 0x7E;                            /* 448 = 1.75 * 2^8 */
    } else if (a < ldexp(1.0, -6)) {
        const double m = nearbyint(ldexp(a, 9)); /* steps of 2^-9 below 2^-6 */
        code = (uint8_t)m;                      /* m = 8 is 2^-6, the first normal code */
    } else {
        int ex;
        (void)frexp(a, &ex);                    /* a in [2^(ex-1), 2^ex) */
        const int e = ex - 1;                   /* a in [2^e, 2^(e+1)), -6 <= e <= 8 */
        double m = nearbyint(ldexp(a, 3 - e));  /* 8 .. 16 in steps of one code */
        int E = e + 7;
        if (m >= 16.0) {                        /* rounded up into the next binade */
            m = 8.0;
            E += 1;
        }
        if (E > 15 || (E == 15 && m > 14.0))    /* above 448 after rounding */
            code = 0x7E;
        else
            code = (uint8_t)((E << 3) | ((int)m - 8));
    }
    return (uint8_t)(code | (neg ? 0x80 : 0));
}

/* Element-wise oracle_e4m3_round / oracle_e4m3_to_double over arrays. */
void oracle_e4m3_round_array(const double *v, long n, uint8_t *out)
{
    for (long i = 0; i < n; ++i)
        out[i] = oracle_e4m3_round(v[i]);
}

void oracle_e4m3_to_double_array(const uint8_t *c, long n, double *out)
{
    for (long i = 0; i < n; ++i)
        out[i] = oracle_e4m3_to_double(c[i]);
}

/* Per-row dynamic E4M3 quantization of a bf16 matrix [R, K]:
 *   amax = max_k |src[r, k]|;  s[r] = amax / 448 (fp32; 1 if amax == 0)
 *   q[r, k] = e4m3( float(src[r, k]) / s[r] )   (fp32 division)         */
void oracle_quant_rows(const bf16_t *src, int R, int K, uint8_t *q, float *s)
{
#pragma omp parallel for schedule(static)
    for (int r = 0; r < R; ++r) {
        float amax = 0.0f;
        for (int k = 0; k < K; ++k) {
            const float v = (float)fabs(bf(src[(size_t)r * K + k]));
            if (v > amax)
                amax = v;
        }
        const float sc = amax > 0.0f ? amax / 448.0f : 1.0f;
        s[r] = sc;
        for (int k = 0; k < K; ++k) {
            const float v = (float)bf(src[(size_t)r * K + k]) / sc;
            q[(size_t)r * K + k] = oracle_e4m3_round((double)v);
        }
    }
}

static double f8(uint8_t c) { return oracle_e4m3_to_double(c); }

/* oracle_expert_act on E4M3 operands: for every pair p = t * top_k + j with
 * e = topk_ids[p]
 *   h[n] = bf16( s_x[t] * s_w13[e][n] * sum_k q_x[t,k] q_w13[e][n][k] )   n < 2I
 *   a[p, i] = bf16( SiLU(h[i]) * h[I + i] )
 * q_x [M, H], s_x [M]; q_w13 [E, 2I, H], s_w13 [E, 2I]; a [M * top_k, I]. */
void oracle_expert_act_fp8(const uint8_t *qx, const float *sx, const uint8_t *qw13,
                           const float *sw13, const int32_t *topk_ids, int M, int top_k,
                           int E, int H, int I, bf16_t *a)
{
    (void)E;
#pragma omp parallel
    {
        double *h = (double *)malloc(sizeof(double) * 2 * (size_t)I);
#pragma omp for schedule(static)
        for (long p = 0; p < (long)M * top_k; ++p) {
            const long t = p / top_k;
            const int e = topk_ids[p];
            const uint8_t *W = qw13 + (size_t)e * 2 * I * H;
            for (int n = 0; n < 2 * I; ++n) {
                double acc = 0.0;
                for (int k = 0; k < H; ++k)
                    acc += f8(qx[(size_t)t * H + k]) * f8(W[(size_t)n * H + k]);
                acc *= (double)sx[t] * (double)sw13[(size_t)e * 2 * I + n];
                h[n] = bf(oracle_bf16_round(acc));
            }
            for (int i = 0; i < I; ++i) {
                const double g = h[i];
                const double silu = g / (1.0 + exp(-g));
                a[(size_t)p * I + i] = oracle_bf16_round(silu * h[I + i]);
            }
        }
        free(h);
    }
}

/* oracle_expert_down_combine on E4M3 operands:
 *   o_p[n] = s_a[p] * s_w2[e][n] * sum_i q_a[p,i] q_w2[e][n][i]     (not rounded)
 *   y[t, n] = bf16( sum_j topk_weights[t, j] * o_{t*top_k + j}[n] + residual[t, n] )
 * q_a [M * top_k, I], s_a [M * top_k]; q_w2 [E, H, I], s_w2 [E, H]. */
void oracle_expert_down_combine_fp8(const uint8_t *qa, const float *sa, const uint8_t *qw2,
                                    const float *sw2, const int32_t *topk_ids,
                                    const float *topk_weights, const bf16_t *residual, int M,
                                    int top_k, int E, int H, int I, bf16_t *y)
{
    (void)E;
#pragma omp parallel for schedule(static)
    for (int t = 0; t < M; ++t) {
        for (int n = 0; n < H; ++n) {
            double acc = 0.0;
            for (int j = 0; j < top_k; ++j) {
                const long p = (long)t * top_k + j;
                const int e = topk_ids[p];
                const uint8_t *W = qw2 + (size_t)e * H * I + (size_t)n * I;
                double o = 0.0;
                for (int i = 0; i < I; ++i)
                    o += f8(qa[(size_t)p * I + i]) * f8(W[i]);
                o *= (double)sa[p] * (double)sw2[(size_t)e * H + n];
                acc += (double)topk_weights[p] * o;
            }
            if (residual)
                acc += bf(residual[(size_t)t * H + n]);
            y[(size_t)t * H + n] = oracle_bf16_round(acc);
        }
    }
}

/* The layer with E4M3 expert weights: the router stays bf16 (logits, top-k
 * as in oracle_moe_forward); x is quantized per token, GEMM 1 runs on codes,
 * its bf16 output a is quantized per pair, GEMM 2 runs on codes, and the
 * combine is the bf16 layer's.  qx_out / sx_out / qa_out / sa_out (nullable)
 * receive the intermediate codes and scales.  Returns 0, or -1 on bad
 * arguments. */
int oracle_moe_forward_fp8(const bf16_t *x, const bf16_t *w_router, const bf16_t *router_logits,
                           const float *router_bias, const uint8_t *qw13, const float *sw13,
                           const uint8_t *qw2, const float *sw2, const bf16_t *residual, int M,
                           int E, int top_k, int H, int I, int renormalize, bf16_t *y,
                           int32_t *topk_ids_out, float *topk_weights_out, bf16_t *logits_out)
{
    if ((w_router == NULL) == (router_logits == NULL))
        return -1;
    if (M < 0 || E < 1 || top_k < 1 || top_k > E || H < 1 || I < 1)
        return -1;
    if (M == 0)
        return 0;
    const size_t P = (size_t)M * top_k;
    bf16_t *logits = (bf16_t *)malloc(sizeof(bf16_t) * (size_t)M * E);
    int32_t *ids = (int32_t *)malloc(sizeof(int32_t) * P);
    float *w = (float *)malloc(sizeof(float) * P);
    bf16_t *a = (bf16_t *)malloc(sizeof(bf16_t) * P * I);
    uint8_t *qx = (uint8_t *)malloc((size_t)M * H);
    float *sx = (float *)malloc(sizeof(float) * (size_t)M);
    uint8_t *qa = (uint8_t *)malloc(P * I);
    float *sa = (float *)malloc(sizeof(float) * P);
    if (!logits || !ids || !w || !a || !qx || !sx || !qa || !sa) {
        free(logits); free(ids); free(w); free(a); free(qx); free(sx); free(qa); free(sa);
        return -1;
    }
    if (w_router)
        oracle_router_logits(x, w_router, router_bias, M, E, H, logits);
    else
        memcpy(logits, router_logits, sizeof(bf16_t) * (size_t)M * E);
    oracle_topk_softmax(logits, M, E, top_k, renormalize, ids, w);
    oracle_quant_rows(x, M, H, qx, sx);
    oracle_expert_act_fp8(qx, sx, qw13, sw13, ids, M, top_k, E, H, I, a);
    oracle_quant_rows(a, (int)P, I, qa, sa);
    oracle_expert_down_combine_fp8(qa, sa, qw2, sw2, ids, w, residual, M, top_k, E, H, I, y);
    if (topk_ids_out)
        memcpy(topk_ids_out, ids, sizeof(int32_t) * P);
    if (topk_weights_out)
        memcpy(topk_weights_out, w, sizeof(float) * P);
    if (logits_out)
        memcpy(logits_out, logits, sizeof(bf16_t) * (size_t)M * E);
    free(logits); free(ids); free(w); free(a); free(qx); free(sx); free(qa); free(sa);
    return 0;
}
