/*
 * moe_oracle.c -- plain, slow fp64 CPU oracle for the routed-expert block of a
 * 4-bit sparse-MoE decode step.
 *
 * TEST INFRASTRUCTURE ONLY.  Nothing in the product library links, includes or
 * calls this file; only the tests, the smoke check and the benchmark's
 * CPU-baseline leg load it (through oracle/__init__.py).  It shares no code,
 * header, table or constant with the CUDA path.
 *
 * What it computes, and where that is stated:
 *  - The block itself (router top-k, softmax over the selected experts, per
 *    expert a dequantised gate_up GEMV, SwiGLU, a dequantised down GEMV, the
 *    routing-weighted sum into the residual): "Sovereign gpt-oss-20B (MXFP4)
 *    on Apple Silicon", sections 1 and 3 (4 sequential experts x 2 small-block
 *    GEMVs per layer, top-4 routing, 2880-wide experts).
 *  - Dequantise-then-multiply is the definition: the fused int4 kernel on the
 *    TinyTitan tracker (entry D108) is bit-identical to dequantising followed
 *    by an ordered matmul, so the oracle dequantises each weight and then
 *    multiplies.
 *  - MXFP4 element and scale formats (FP4 E2M1 codes, 32 per block, one E8M0
 *    power-of-two scale): OCP Microscaling Formats (MX) v1.0, element type
 *    FP4 E2M1 and scale type E8M0.  The pages name the format ("MXFP4 reader",
 *    section 3 of the gpt-oss page) but do not print its bit layout.
 *  - Packed int4 with one fp16 scale per group: "Single-stream int4 decode of
 *    a 30B MoE on Apple Silicon", sections 1 and 6 (the int4 path dequantises
 *    on chip from packed int4); symmetric code-8 with fp16 group scales.
 *
 * Readings where the pages are silent (each also listed in the design notes):
 *  - Top-k order: logit descending, lower expert index first on ties; a NaN
 *    logit orders as -inf.
 *  - Softmax is over the k selected logits only.
 *  - Nibble order: the low nibble of byte b holds element 2b, the high nibble
 *    element 2b+1; weights are row-major [N_out][K] with blocks along K.
 *  - gate_up rows [0, I) are gate, rows [I, 2I) are up; SwiGLU is
 *    silu(gate) * up with silu(g) = g / (1 + exp(-g)) by default; the
 *    clamped, alpha-scaled form of the public gpt-oss model is a setting
 *    (moe_oracle_set_swiglu, below).
 *  - Stack coupling: x_l = bf16(r_l / sqrt(mean(r_l^2) + 1e-6)),
 *    r_{l+1} = bf16(r_l + MoE_l(x_l)), both roundings to nearest-even.
 *  - Batched path: x and h are quantised to MXFP4 per 32 elements along K
 *    with the OCP MX conversion (shared exponent floor(log2 amax) - 2,
 *    elements rounded to nearest-even E2M1, saturating at +-6).
 *
 * Everything is fp64.  Loops are the textbook ones; the only parallelism is an
 * OpenMP split over independent output rows, each row summed in index order.
 */
#include <math.h>
#include <stdint.h>
#include <stdlib.h>
#include <string.h>
#ifdef _OPENMP
#include <omp.h>
#endif

enum { FMT_MXFP4 = 1, FMT_INT4 = 2 };

/* ------------------------------------------------------------------------ */
/* Scalar formats                                                            */
/* ------------------------------------------------------------------------ */

/* FP4 E2M1: sign bit 3, exponent bits 2..1 (bias 1), mantissa bit 0.
 * Exponent field 0 is subnormal: value = mantissa * 2^(1-1) * 0.5. */
double moe_oracle_e2m1(int code)
{
    int sign = (code >> 3) & 1;
    int e = (code >> 1) & 3;
    int m = code & 1;
    double mag;
    if (e == 0)
        mag = 0.5 * m;
    else
        mag = ldexp(1.0 + 0.5 * m, e - 1);
    return sign ? -mag : mag;
}

/* E8M0: an unsigned biased exponent, value 2^(e-127); 0xFF is NaN. */
double moe_oracle_e8m0(int byte)
{
    if (byte == 255)
        return NAN;
    return ldexp(1.0, byte - 127);
}

/* IEEE 754 binary16: sign, 5 exponent bits (bias 15), 10 fraction bits. */
double moe_oracle_fp16(uint16_t bits)
{
    int sign = bits >> 15;
    int e = (bits >> 10) & 0x1f;
    int f = bits & 0x3ff;
    double mag;
    if (e == 0)
        mag = ldexp((double)f, -24);              /* subnormal: f * 2^-14 * 2^-10 */
    else if (e == 31)
        mag = f ? NAN : INFINITY;
    else
        mag = ldexp(1.0 + f / 1024.0, e - 15);
    return sign ? -mag : mag;
}

/* bfloat16: sign, 8 exponent bits (bias 127), 7 fraction bits. */
double moe_oracle_bf16(uint16_t bits)
{
    int sign = bits >> 15;
    int e = (bits >> 7) & 0xff;
    int f = bits & 0x7f;
    double mag;
    if (e == 0)
        mag = ldexp((double)f, -133);             /* subnormal: f * 2^-126 * 2^-7 */
    else if (e == 255)
        mag = f ? NAN : INFINITY;
    else
        mag = ldexp(1.0 + f / 128.0, e - 127);
    return sign ? -mag : mag;
}

/* Round an fp64 value to the nearest bfloat16 (ties to even), as bits. */
uint16_t moe_oracle_to_bf16(double v)
{
    if (isnan(v))
        return 0x7fc0;
    uint16_t sign = signbit(v) ? 0x8000 : 0;
    double a = fabs(v);
    if (a == 0.0)
        return sign;
    if (isinf(a))
        return sign | 0x7f80;
    int e;
    frexp(a, &e);                 /* a in [2^(e-1), 2^e) */
    int exp2 = e - 1;             /* a in [2^exp2, 2^(exp2+1)) */
    if (exp2 < -126)
        exp2 = -126;              /* subnormal range: fixed spacing 2^-133 */
    double ulp = ldexp(1.0, exp2 - 7);
    double q = nearbyint(a / ulp);            /* default rounding mode: ties to even */
    double r = q * ulp;
    if (r >= ldexp(1.0, 128))
        return sign | 0x7f80;
    /* encode r exactly */
    if (r < ldexp(1.0, -126)) {
        return sign | (uint16_t)q;            /* subnormal: fraction = q */
    }
    int er;
    double fr = frexp(r, &er);                /* r = fr * 2^er, fr in [0.5, 1) */
    int biased = er - 1 + 127;
    int frac = (int)((fr * 2.0 - 1.0) * 128.0);
    return sign | (uint16_t)(biased << 7) | (uint16_t)frac;
}

/* ------------------------------------------------------------------------ */
/* Weights                                                                   */
/* ------------------------------------------------------------------------ */

/* The 4-bit code of element (n, k) of a row-major [N][K] packed matrix. */
static int nibble(const uint8_t* codes, int K, int64_t n, int64_t k)
{
    uint8_t byte = codes[n * (K / 2) + k / 2];
    return (k % 2 == 0) ? (byte & 0xf) : (byte >> 4);
}

/* W[n][k] of one expert projection.
 *  MXFP4: e2m1(code) * 2^(scale[n][k/32] - 127), scales u8 [N][K/32].
 *  int4 : (code - 8) * fp16(scale[n][k/group]), scales fp16 [N][K/group]. */
double moe_oracle_weight(int fmt, const uint8_t* codes, const void* scales,
                         int K, int group, int64_t n, int64_t k)
{
    int q = nibble(codes, K, n, k);
    if (fmt == FMT_MXFP4) {
        const uint8_t* s = (const uint8_t*)scales;
        return moe_oracle_e2m1(q) * moe_oracle_e8m0(s[n * (K / 32) + k / 32]);
    } else {
        const uint16_t* s = (const uint16_t*)scales;
        return (double)(q - 8) * moe_oracle_fp16(s[n * (K / group) + k / group]);
    }
}

void moe_oracle_dequant(int fmt, const uint8_t* codes, const void* scales,
                        int N, int K, int group, double* out)
{
    for (int64_t n = 0; n < N; ++n)
        for (int64_t k = 0; k < K; ++k)
            out[n * K + k] = moe_oracle_weight(fmt, codes, scales, K, group, n, k);
}

/* y[n] = sum_k W[n][k] * v[k] + bias[n]   (bias may be NULL) */
static void gemv(int fmt, const uint8_t* codes, const void* scales, const uint16_t* bias,
                 int N, int K, int group, const double* v, double* y, int nthreads)
{
    (void)nthreads;
#ifdef _OPENMP
#pragma omp parallel for schedule(static) num_threads(nthreads > 0 ? nthreads : 1)
#endif
    for (int64_t n = 0; n < N; ++n) {
        double acc = 0.0;
        for (int64_t k = 0; k < K; ++k)
            acc += moe_oracle_weight(fmt, codes, scales, K, group, n, k) * v[k];
        if (bias)
            acc += moe_oracle_bf16(bias[n]);
        y[n] = acc;
    }
}

/* ------------------------------------------------------------------------ */
/* Router                                                                    */
/* ------------------------------------------------------------------------ */

/* Per token: the k experts with the largest logits (ties: lower index first;
 * NaN orders as -inf), then w_s = exp(l_s - l_max) / sum_j exp(l_j - l_max)
 * over the k selected.  idx [M][k] in selection order, w [M][k]. */
void moe_oracle_route(const float* logits, int M, int E, int k, int32_t* idx, double* w)
{
    for (int m = 0; m < M; ++m) {
        const float* l = logits + (int64_t)m * E;
        char* taken = (char*)calloc((size_t)E, 1);
        for (int s = 0; s < k; ++s) {
            int best = -1;
            double bv = 0.0;
            for (int e = 0; e < E; ++e) {
                if (taken[e])
                    continue;
                double v = isnan(l[e]) ? -INFINITY : (double)l[e];
                if (best < 0 || v > bv) {     /* strict: the lower index keeps a tie */
                    best = e;
                    bv = v;
                }
            }
            taken[best] = 1;
            idx[m * k + s] = best;
        }
        free(taken);
        double lmax = -INFINITY;
        for (int s = 0; s < k; ++s) {
            double v = isnan(l[idx[m * k + s]]) ? -INFINITY : (double)l[idx[m * k + s]];
            if (v > lmax)
                lmax = v;
        }
        double den = 0.0;
        for (int s = 0; s < k; ++s) {
            double v = isnan(l[idx[m * k + s]]) ? -INFINITY : (double)l[idx[m * k + s]];
            w[m * k + s] = exp(v - lmax);
            den += w[m * k + s];
        }
        for (int s = 0; s < k; ++s)
            w[m * k + s] /= den;
    }
}

/* ------------------------------------------------------------------------ */
/* One routed-expert MoE layer                                               */
/* ------------------------------------------------------------------------ */

/* SwiGLU form: h = gc * sigmoid(alpha * gc) * (uc + beta), gc = min(g, limit),
 * uc = clamp(u, -limit, limit) (a NaN stays NaN).  alpha = 1, limit = +inf,
 * beta = 0 is the plain silu(g) * u.  The gpt-oss model's expert activation
 * (its public reference implementation) is alpha = 1.702, limit = 7, beta = 1;
 * the pages name the model but not its activation's constants. */
static double sw_alpha = 1.0, sw_limit = INFINITY, sw_beta = 0.0;

void moe_oracle_set_swiglu(double alpha, double limit, double beta)
{
    sw_alpha = alpha;
    sw_limit = limit;
    sw_beta = beta;
}

static double swiglu(double g, double u)
{
    if (g > sw_limit)
        g = sw_limit;
    if (u > sw_limit)
        u = sw_limit;
    if (u < -sw_limit)
        u = -sw_limit;
    return g / (1.0 + exp(-(sw_alpha * g))) * (u + sw_beta);
}

/* Sizes of one expert's tensors in elements / bytes. */
static int64_t codes_bytes(int N, int K) { return (int64_t)N * K / 2; }
static int64_t scale_count(int fmt, int N, int K, int group)
{
    return fmt == FMT_MXFP4 ? (int64_t)N * (K / 32) : (int64_t)N * (K / group);
}
static int64_t scale_bytes(int fmt, int N, int K, int group)
{
    return scale_count(fmt, N, K, group) * (fmt == FMT_MXFP4 ? 1 : 2);
}

/* out_delta[m][:] = sum_s w[m][s] * expert_{idx[m][s]}(x[m]) for the given
 * (already routed) token, with x given in fp64.  Helper shared by the decode
 * and stack entry points. */
static void expert_mix(int fmt, int H, int I, int group, int k,
                       const uint8_t* gu_codes, const void* gu_scales, const uint16_t* gu_bias,
                       const uint8_t* dn_codes, const void* dn_scales, const uint16_t* dn_bias,
                       const int32_t* idx, const double* w, const double* x, double* delta,
                       int nthreads)
{
    double* a = (double*)malloc(sizeof(double) * 2 * (size_t)I);
    double* h = (double*)malloc(sizeof(double) * (size_t)I);
    double* y = (double*)malloc(sizeof(double) * (size_t)H);
    for (int j = 0; j < H; ++j)
        delta[j] = 0.0;
    for (int s = 0; s < k; ++s) {
        int64_t e = idx[s];
        const uint8_t* guc = gu_codes + e * codes_bytes(2 * I, H);
        const uint8_t* gus = (const uint8_t*)gu_scales + e * scale_bytes(fmt, 2 * I, H, group);
        const uint16_t* gub = gu_bias ? gu_bias + e * 2 * I : NULL;
        const uint8_t* dnc = dn_codes + e * codes_bytes(H, I);
        const uint8_t* dns = (const uint8_t*)dn_scales + e * scale_bytes(fmt, H, I, group);
        const uint16_t* dnb = dn_bias ? dn_bias + e * H : NULL;
        gemv(fmt, guc, gus, gub, 2 * I, H, group, x, a, nthreads);      /* a = W_gu x + b_gu */
        for (int i = 0; i < I; ++i)
            h[i] = swiglu(a[i], a[I + i]);                             /* SwiGLU */
        gemv(fmt, dnc, dns, dnb, H, I, group, h, y, nthreads);          /* y = W_d h + b_d */
        for (int j = 0; j < H; ++j)
            delta[j] += w[s] * y[j];                                   /* weighted combine */
    }
    free(a);
    free(h);
    free(y);
}

/* Decode layer: out[m][j] = r[m][j] + sum_s w[m][s] * y_{m,s}[j]  (fp64).
 * Tensor layouts (one layer, all E experts):
 *   gu_codes  u8   [E][2I][H/2]     gu_scales u8 [E][2I][H/32] or fp16 [E][2I][H/group]
 *   gu_bias   bf16 [E][2I] or NULL
 *   dn_codes  u8   [E][H][I/2]      dn_scales u8 [E][H][I/32]  or fp16 [E][H][I/group]
 *   dn_bias   bf16 [E][H]  or NULL
 *   x bf16 [M][H], logits fp32 [M][E], r bf16 [M][H] or NULL (zero residual)
 * idx_out [M][k] / w_out [M][k] receive the routing if non-NULL. */
int moe_oracle_layer(int fmt, int H, int I, int E, int group, int M, int k,
                     const uint8_t* gu_codes, const void* gu_scales, const uint16_t* gu_bias,
                     const uint8_t* dn_codes, const void* dn_scales, const uint16_t* dn_bias,
                     const uint16_t* x, const float* logits, const uint16_t* r,
                     double* out, int32_t* idx_out, double* w_out, int nthreads)
{
    if (k < 1 || k > E || M < 0)
        return -1;
    int32_t* idx = (int32_t*)malloc(sizeof(int32_t) * (size_t)(M * k + 1));
    double* w = (double*)malloc(sizeof(double) * (size_t)(M * k + 1));
    double* xv = (double*)malloc(sizeof(double) * (size_t)H);
    double* delta = (double*)malloc(sizeof(double) * (size_t)H);
    moe_oracle_route(logits, M, E, k, idx, w);
    for (int m = 0; m < M; ++m) {
        for (int j = 0; j < H; ++j)
            xv[j] = moe_oracle_bf16(x[(int64_t)m * H + j]);
        expert_mix(fmt, H, I, group, k, gu_codes, gu_scales, gu_bias, dn_codes, dn_scales,
                   dn_bias, idx + m * k, w + m * k, xv, delta, nthreads);
        for (int j = 0; j < H; ++j)
            out[(int64_t)m * H + j] = (r ? moe_oracle_bf16(r[(int64_t)m * H + j]) : 0.0) + delta[j];
    }
    if (idx_out)
        memcpy(idx_out, idx, sizeof(int32_t) * (size_t)(M * k));
    if (w_out)
        memcpy(w_out, w, sizeof(double) * (size_t)(M * k));
    free(idx);
    free(w);
    free(xv);
    free(delta);
    return 0;
}

/* Router GEMV, the plain definition in fp64:
 *   logits[m][e] = b[e] + sum_h x[m][h] * W[e][h]
 * x bf16 [M][H] (the layer input the experts see), W bf16 [E][H], b bf16 [E]
 * or NULL.  The router is the MoE block's gate: a linear map of the
 * normalised hidden state to one logit per expert, whose top-k picks the
 * experts ("Sovereign gpt-oss-20B (MXFP4) on Apple Silicon", section 1, top-4
 * of 32; "Amortizing the per-token host-sync setup tax in fused all-layer q4
 * decode on Apple M1 Ultra", section 3, the top-k on the GPU). */
void moe_oracle_router(int H, int E, int M, const uint16_t* x, const uint16_t* w, const uint16_t* b,
                       double* out)
{
    for (int m = 0; m < M; ++m)
        for (int e = 0; e < E; ++e) {
            double acc = 0.0;
            for (int j = 0; j < H; ++j)
                acc += moe_oracle_bf16(x[(int64_t)m * H + j]) * moe_oracle_bf16(w[(int64_t)e * H + j]);
            out[(int64_t)m * E + e] = (b ? moe_oracle_bf16(b[e]) : 0.0) + acc;
        }
}

/* Expert stack: for l = 0..L-1, per token
 *   x_l     = bf16( r_l / sqrt(mean(r_l^2) + 1e-6) )
 *   r_{l+1} = bf16( r_l + MoE_l(x_l) )
 * layer l's tensors are passed as arrays of L pointers; logits fp32 [L][M][E];
 * resid bf16 [M][H] is read as r_0 and overwritten with r_L.
 * With router weights rw (L pointers to bf16 [E][H]; rb: L pointers to bf16
 * [E] or NULL), layer l's logits are instead the router GEMV of x_l, rounded
 * to fp32 (the precision the top-k is taken in), and `logits` is not read. */
int moe_oracle_stack(int fmt, int H, int I, int E, int group, int L, int M, int k,
                     const uint8_t* const* gu_codes, const void* const* gu_scales,
                     const uint16_t* const* gu_bias,
                     const uint8_t* const* dn_codes, const void* const* dn_scales,
                     const uint16_t* const* dn_bias,
                     const float* logits, uint16_t* resid,
                     const uint16_t* const* rw, const uint16_t* const* rb, int nthreads)
{
    if (k < 1 || k > E || M < 0 || L < 0)
        return -1;
    int32_t* idx = (int32_t*)malloc(sizeof(int32_t) * (size_t)(M * k + 1));
    double* w = (double*)malloc(sizeof(double) * (size_t)(M * k + 1));
    double* xv = (double*)malloc(sizeof(double) * (size_t)H);
    double* rv = (double*)malloc(sizeof(double) * (size_t)H);
    double* delta = (double*)malloc(sizeof(double) * (size_t)H);
    uint16_t* xb = (uint16_t*)malloc(sizeof(uint16_t) * (size_t)H);
    double* lg64 = (double*)malloc(sizeof(double) * (size_t)E);
    float* lg32 = (float*)malloc(sizeof(float) * (size_t)E);
    for (int l = 0; l < L; ++l) {
        if (!rw)
            moe_oracle_route(logits + (int64_t)l * M * E, M, E, k, idx, w);
        for (int m = 0; m < M; ++m) {
            uint16_t* rm = resid + (int64_t)m * H;
            double ss = 0.0;
            for (int j = 0; j < H; ++j) {
                rv[j] = moe_oracle_bf16(rm[j]);
                ss += rv[j] * rv[j];
            }
            double inv = 1.0 / sqrt(ss / H + 1e-6);
            for (int j = 0; j < H; ++j) {
                xb[j] = moe_oracle_to_bf16(rv[j] * inv);
                xv[j] = moe_oracle_bf16(xb[j]);
            }
            if (rw) {
                moe_oracle_router(H, E, 1, xb, rw[l], rb ? rb[l] : NULL, lg64);
                for (int e = 0; e < E; ++e)
                    lg32[e] = (float)lg64[e];
                moe_oracle_route(lg32, 1, E, k, idx + m * k, w + m * k);
            }
            expert_mix(fmt, H, I, group, k, gu_codes[l], gu_scales[l],
                       gu_bias ? gu_bias[l] : NULL, dn_codes[l], dn_scales[l],
                       dn_bias ? dn_bias[l] : NULL, idx + m * k, w + m * k, xv, delta,
                       nthreads);
            for (int j = 0; j < H; ++j)
                rm[j] = moe_oracle_to_bf16(rv[j] + delta[j]);
        }
    }
    free(idx);
    free(w);
    free(xv);
    free(rv);
    free(delta);
    free(xb);
    free(lg64);
    free(lg32);
    return 0;
}

/* ------------------------------------------------------------------------ */
/* Batched path: MX quantisation of activations                              */
/* ------------------------------------------------------------------------ */

/* Nearest E2M1 code to v (ties to the even mantissa), saturating at +-6.
 * Sign is kept, so a negative value that rounds to zero gives code 8 (-0). */
static int e2m1_round(double v)
{
    int sign = signbit(v) ? 8 : 0;
    double a = fabs(v);
    if (isnan(v))
        return 7 | sign;        /* not produced for finite inputs; saturate */
    int best = 0;
    double bd = INFINITY;
    for (int c = 0; c < 8; ++c) {
        double d = fabs(a - moe_oracle_e2m1(c));
        if (d < bd || (d == bd && (c & 1) == 0 && (best & 1) == 1)) {
            best = c;
            bd = d;
        }
    }
    return best | sign;
}

/* OCP MX conversion of n values (n a multiple of 32) to MXFP4:
 *   per block: amax = max |v|; amax == 0 -> scale byte 0, codes +0;
 *   else shared exponent X = floor(log2(amax)) - 2 (2 = largest E2M1 exponent),
 *   clamped to [-127, 127]; scale byte = X + 127; code_i = e2m1_round(v_i / 2^X).
 * codes are packed two per byte, low nibble first. */
void moe_oracle_mx_quantize(const double* v, int64_t n, uint8_t* codes, uint8_t* scales)
{
    for (int64_t b = 0; b < n / 32; ++b) {
        double amax = 0.0;
        for (int i = 0; i < 32; ++i) {
            double a = fabs(v[b * 32 + i]);
            if (a > amax)
                amax = a;
        }
        int X;
        if (amax == 0.0) {
            X = -127;
        } else {
            int e;
            frexp(amax, &e);            /* amax in [2^(e-1), 2^e) */
            X = (e - 1) - 2;
            if (X < -127)
                X = -127;
            if (X > 127)
                X = 127;
        }
        scales[b] = (uint8_t)(X + 127);
        for (int i = 0; i < 32; i += 2) {
            int c0 = amax == 0.0 ? 0 : e2m1_round(ldexp(v[b * 32 + i], -X));
            int c1 = amax == 0.0 ? 0 : e2m1_round(ldexp(v[b * 32 + i + 1], -X));
            codes[(b * 32 + i) / 2] = (uint8_t)(c0 | (c1 << 4));
        }
    }
}

/* Batched MXFP4 layer with MX-quantised activations (the tensor-core path):
 *   x_q = MX(x)                          per token, blocks of 32 along H
 *   a   = W_gu x_q + b_gu;  h = SwiGLU(a[0:I], a[I:2I]) (the form set above)
 *   h_q = MX(h)                          blocks of 32 along I
 *   y   = W_d h_q + b_d;    out = r + sum_s w_s y_s
 * If h_codes_in / h_scales_in are non-NULL they replace the oracle's own h_q
 * (layout [M][k][I/2] and [M][k][I/32], slot order of the routing); this lets
 * a test check the down stage on a given quantised h.  h_codes_out /
 * h_scales_out, if non-NULL, receive the oracle's h_q. */
int moe_oracle_layer_batched(int H, int I, int E, int M, int k,
                             const uint8_t* gu_codes, const uint8_t* gu_scales,
                             const uint16_t* gu_bias,
                             const uint8_t* dn_codes, const uint8_t* dn_scales,
                             const uint16_t* dn_bias,
                             const uint16_t* x, const float* logits, const uint16_t* r,
                             const uint8_t* h_codes_in, const uint8_t* h_scales_in,
                             uint8_t* h_codes_out, uint8_t* h_scales_out,
                             double* out, int nthreads)
{
    if (k < 1 || k > E || M < 0 || H % 32 || I % 32)
        return -1;
    int32_t* idx = (int32_t*)malloc(sizeof(int32_t) * (size_t)(M * k + 1));
    double* w = (double*)malloc(sizeof(double) * (size_t)(M * k + 1));
    double* xv = (double*)malloc(sizeof(double) * (size_t)H);
    double* xq = (double*)malloc(sizeof(double) * (size_t)H);
    uint8_t* xc = (uint8_t*)malloc((size_t)H / 2);
    uint8_t* xs = (uint8_t*)malloc((size_t)H / 32);
    double* a = (double*)malloc(sizeof(double) * 2 * (size_t)I);
    double* h = (double*)malloc(sizeof(double) * (size_t)I);
    double* hq = (double*)malloc(sizeof(double) * (size_t)I);
    uint8_t* hc = (uint8_t*)malloc((size_t)I / 2);
    uint8_t* hs = (uint8_t*)malloc((size_t)I / 32);
    double* y = (double*)malloc(sizeof(double) * (size_t)H);
    moe_oracle_route(logits, M, E, k, idx, w);
    for (int m = 0; m < M; ++m) {
        for (int j = 0; j < H; ++j)
            xv[j] = moe_oracle_bf16(x[(int64_t)m * H + j]);
        moe_oracle_mx_quantize(xv, H, xc, xs);
        for (int j = 0; j < H; ++j)
            xq[j] = moe_oracle_e2m1(nibble(xc, H, 0, j)) * moe_oracle_e8m0(xs[j / 32]);
        double* o = out + (int64_t)m * H;
        for (int j = 0; j < H; ++j)
            o[j] = r ? moe_oracle_bf16(r[(int64_t)m * H + j]) : 0.0;
        for (int s = 0; s < k; ++s) {
            int64_t e = idx[m * k + s];
            gemv(FMT_MXFP4, gu_codes + e * codes_bytes(2 * I, H),
                 gu_scales + e * scale_bytes(FMT_MXFP4, 2 * I, H, 32),
                 gu_bias ? gu_bias + e * 2 * I : NULL, 2 * I, H, 32, xq, a, nthreads);
            for (int i = 0; i < I; ++i)
                h[i] = swiglu(a[i], a[I + i]);
            int64_t slot = (int64_t)m * k + s;
            const uint8_t* hcu = hc;
            const uint8_t* hsu = hs;
            if (h_codes_in && h_scales_in) {
                hcu = h_codes_in + slot * (I / 2);
                hsu = h_scales_in + slot * (I / 32);
            } else {
                moe_oracle_mx_quantize(h, I, hc, hs);
            }
            if (h_codes_out)
                memcpy(h_codes_out + slot * (I / 2), hcu, (size_t)I / 2);
            if (h_scales_out)
                memcpy(h_scales_out + slot * (I / 32), hsu, (size_t)I / 32);
            for (int i = 0; i < I; ++i)
                hq[i] = moe_oracle_e2m1(nibble(hcu, I, 0, i)) * moe_oracle_e8m0(hsu[i / 32]);
            gemv(FMT_MXFP4, dn_codes + e * codes_bytes(H, I),
                 dn_scales + e * scale_bytes(FMT_MXFP4, H, I, 32),
                 dn_bias ? dn_bias + e * H : NULL, H, I, 32, hq, y, nthreads);
            for (int j = 0; j < H; ++j)
                o[j] += w[m * k + s] * y[j];
        }
    }
    free(idx); free(w); free(xv); free(xq); free(xc); free(xs);
    free(a); free(h); free(hq); free(hc); free(hs); free(y);
    return 0;
}

int moe_oracle_max_threads(void)
{
#ifdef _OPENMP
    return omp_get_max_threads();
#else
    return 1;
#endif
}
