/*
 * Oracle for the fused rank-sum + residual add + RMSNorm operator.
 *
 * TEST INFRASTRUCTURE ONLY.  This file is the plain, slow, single-threaded
 * CPU statement of what the operator computes.  Only the tests, the smoke
 * check and the benchmark's CPU-baseline leg load it; the product path
 * (the CUDA library and its Python binding) never does, and shares no code,
 * header or constant with it.
 *
 * Source of the method: FlagTree pull request "[TLERaw] Add NVSHMEM
 * allreduce RMSNorm tutorial".
 *   - Summary: the contract
 *         reduced      = AllReduce_SUM(x)
 *         residual_out = reduced + residual
 *         norm_out     = RMSNorm(residual_out, weight, eps)
 *   - Implementation section 3, "Residual + RMSNorm epilogue": the epilogue
 *     runs after the reduction is complete, on `reduced`, with FP32
 *     accumulation for the normalisation.
 *   - Correctness section: all tensors are BF16.
 *
 * Readings where the page is silent (each one is listed with its reason in
 * the design notes of this repository):
 *   1. The W partials are summed in FP32, strictly in rank order 0..W-1,
 *      with the accumulator seeded from the widened x[0] (not from +0.0,
 *      which would turn an all -0 column into +0).
 *   2. `reduced` is rounded to bf16 before the residual is added (the
 *      epilogue consumes the reduced tensor, itself a bf16 output).
 *   3. residual_out = bf16(f32(reduced) + f32(residual)).
 *   4. RMSNorm over the bf16 residual_out of one row (H elements):
 *         ss   = sum over h of ro[h]*ro[h]   (fp32, sequential in h)
 *         mean = ss / H                      (fp32 division)
 *         rstd = 1 / sqrt(mean + eps)        (fp32, eps inside the root)
 *         norm_out[h] = bf16((ro[h] * rstd) * weight[h])
 *      i.e. the weight multiplies the fp32 normalised value and the result
 *      is rounded once.
 *   5. Every fp32 -> bf16 conversion rounds to nearest, ties to even.
 *      Subnormals are kept.  NaN stays NaN (quiet, sign kept).
 *
 * Build: -O2 -ffp-contract=off, no fast-math, so that every + and * above
 * is one IEEE single-precision operation (no fused multiply-add, no
 * reassociation).  sqrtf and '/' are IEEE correctly rounded.
 *
 * bf16 values travel as their 16-bit patterns (uint16_t).
 */
#include <math.h>
#include <stdint.h>
#include <string.h>

/* bfloat16 is the upper half of an IEEE binary32 pattern (1 sign bit,
 * 8 exponent bits, 7 fraction bits), so widening is exact: shift the
 * 16 bits into the upper half of a binary32 and zero the rest. */
float oracle_bf16_to_f32(uint16_t b)
{
    uint32_t u = ((uint32_t)b) << 16;
    float f;
    memcpy(&f, &u, sizeof f);
    return f;
}

/* Narrowing binary32 -> bfloat16, round to nearest, ties to even.
 * The 16 dropped low bits decide: above half an ulp rounds up, below
 * rounds down, exactly half rounds to the even kept pattern.  Rounding up
 * adds one to the kept pattern; a carry out of the fraction moves into the
 * exponent, which is the correct next representable value (up to +-inf).
 * NaN is returned as a quiet NaN with the same sign. */
uint16_t oracle_f32_to_bf16(float f)
{
    uint32_t u;
    memcpy(&u, &f, sizeof u);
    uint32_t kept = u >> 16;
    uint32_t dropped = u & 0xFFFFu;
    if (isnan(f))
        return (uint16_t)(kept | 0x0040u);
    if (dropped > 0x8000u || (dropped == 0x8000u && (kept & 1u)))
        kept += 1u;
    return (uint16_t)kept;
}

/* The same narrowing applied to a binary32 given by its bit pattern, so a
 * caller can pass any NaN payload unchanged. */
uint16_t oracle_f32_bits_to_bf16(uint32_t u)
{
    float f;
    memcpy(&f, &u, sizeof f);
    return oracle_f32_to_bf16(f);
}

/* Step a1, rank sum of one element position: FP32 accumulation in rank
 * order, the sum rounded to bf16. */
static uint16_t rank_sum_one(const uint16_t *const *x, int W, int64_t idx)
{
    float acc = oracle_bf16_to_f32(x[0][idx]);
    for (int r = 1; r < W; ++r)
        acc = acc + oracle_bf16_to_f32(x[r][idx]);
    return oracle_f32_to_bf16(acc);
}

/* Step a1 over a [T,H] block: reduced[t,h] = bf16(sum_r x[r][t,h]). */
void oracle_rank_sum(const uint16_t *const *x, int W, int64_t n,
                     uint16_t *reduced)
{
    for (int64_t i = 0; i < n; ++i)
        reduced[i] = rank_sum_one(x, W, i);
}

/* Step a2: residual_out = bf16(f32(reduced) + f32(residual)). */
void oracle_residual_add(const uint16_t *reduced, const uint16_t *residual,
                         int64_t n, uint16_t *residual_out)
{
    for (int64_t i = 0; i < n; ++i) {
        float s = oracle_bf16_to_f32(reduced[i]) + oracle_bf16_to_f32(residual[i]);
        residual_out[i] = oracle_f32_to_bf16(s);
    }
}

/* Steps a3-a4 for one row of H elements: RMSNorm of the bf16 residual_out
 * with FP32 accumulation, scaled by weight, rounded once to bf16.
 * Returns the fp32 rstd it used (the tests read it). */
float oracle_rmsnorm_row(const uint16_t *ro, const uint16_t *weight,
                         float eps, int64_t H, uint16_t *norm_out)
{
    float ss = 0.0f;
    for (int64_t h = 0; h < H; ++h) {
        float v = oracle_bf16_to_f32(ro[h]);
        ss = ss + v * v;
    }
    float mean = ss / (float)H;
    float rstd = 1.0f / sqrtf(mean + eps);
    for (int64_t h = 0; h < H; ++h) {
        float v = oracle_bf16_to_f32(ro[h]);
        float n = v * rstd;
        norm_out[h] = oracle_f32_to_bf16(n * oracle_bf16_to_f32(weight[h]));
    }
    return rstd;
}

/* Step a1 with fp32 partials (the partial sums of a GEMM epilogue, say):
 * the same rank-order FP32 sum, the partials' own fp32 values used as they
 * are (no rounding to bf16 before the sum), the sum rounded once to bf16. */
static uint16_t rank_sum_one_f32(const float *const *x, int W, int64_t idx)
{
    float acc = x[0][idx];
    for (int r = 1; r < W; ++r)
        acc = acc + x[r][idx];
    return oracle_f32_to_bf16(acc);
}

void oracle_rank_sum_f32(const float *const *x, int W, int64_t n, uint16_t *reduced)
{
    for (int64_t i = 0; i < n; ++i)
        reduced[i] = rank_sum_one_f32(x, W, i);
}

/* The whole operator on row-major [T,H] tensors, row after row, in the
 * order of the contract: rank sum, residual add, RMSNorm.
 * x is an array of W pointers, one per rank partial.  Returns 0, or -1 on
 * an argument it cannot process (W < 1, T < 0, H < 1, a null pointer). */
int oracle_forward(const uint16_t *const *x, int W, const uint16_t *residual,
                   const uint16_t *weight, float eps, int64_t T, int64_t H,
                   uint16_t *reduced, uint16_t *residual_out,
                   uint16_t *norm_out)
{
    if (W < 1 || T < 0 || H < 1 || !x || !residual || !weight || !reduced ||
        !residual_out || !norm_out)
        return -1;
    for (int r = 0; r < W; ++r)
        if (!x[r])
            return -1;
    const uint16_t *row_x[256];
    if (W > 256)
        return -1;
    for (int64_t t = 0; t < T; ++t) {
        int64_t off = t * H;
        for (int r = 0; r < W; ++r)
            row_x[r] = x[r] + off;
        oracle_rank_sum(row_x, W, H, reduced + off);
        oracle_residual_add(reduced + off, residual + off, H, residual_out + off);
        oracle_rmsnorm_row(residual_out + off, weight, eps, H, norm_out + off);
    }
    return 0;
}

/* The whole operator with fp32 partials; residual, weight and the three
 * outputs bf16 as in oracle_forward.  Same return convention. */
int oracle_forward_f32(const float *const *x, int W, const uint16_t *residual,
                       const uint16_t *weight, float eps, int64_t T, int64_t H,
                       uint16_t *reduced, uint16_t *residual_out,
                       uint16_t *norm_out)
{
    if (W < 1 || W > 256 || T < 0 || H < 1 || !x || !residual || !weight ||
        !reduced || !residual_out || !norm_out)
        return -1;
    for (int r = 0; r < W; ++r)
        if (!x[r])
            return -1;
    const float *row_x[256];
    for (int64_t t = 0; t < T; ++t) {
        int64_t off = t * H;
        for (int r = 0; r < W; ++r)
            row_x[r] = x[r] + off;
        oracle_rank_sum_f32(row_x, W, H, reduced + off);
        oracle_residual_add(reduced + off, residual + off, H, residual_out + off);
        oracle_rmsnorm_row(residual_out + off, weight, eps, H, norm_out + off);
    }
    return 0;
}

/* ---------------------------------------------------------------------
 * Fused FP8 quantisation of norm_out (an extension the page does not
 * describe: the next layer's GEMM input in the OCP 8-bit E4M3 format).
 *
 * E4M3 ("FN" flavour): 1 sign bit, 4 exponent bits (bias 7), 3 fraction
 * bits; no infinities; S.1111.111 is NaN; the largest finite magnitude is
 * 448 = 1.75 * 2^8; subnormals are multiples of 2^-9.
 *
 * Reading: per row t, amax = the largest |norm_out[t,h]| (NaN ignored, as
 * IEEE maxNum does); the scale written for dequantisation is
 * scale[t] = amax / 448 and the quantised values use the row's fp32
 * inverse inv = 448 / amax (both single fp32 divisions; 1 and 1 if amax is
 * 0): q[t,h] = E4M3(norm_out[t,h] * inv), round to nearest even, any
 * magnitude above 448 (infinity included) saturated to 448; NaN stays NaN.
 * Given the bf16 norm_out row, scale and q are unique.
 * ------------------------------------------------------------------- */
float oracle_e4m3_to_f32(uint8_t b)
{
    float sign = (b & 0x80u) ? -1.0f : 1.0f;
    int e = (b >> 3) & 0xF, m = b & 0x7;
    if (e == 0xF && m == 0x7)
        return NAN;
    if (e == 0)
        return sign * ldexpf((float)m, -9);
    return sign * ldexpf(1.0f + (float)m / 8.0f, e - 7);
}

uint8_t oracle_f32_to_e4m3_sat(float f)
{
    if (isnan(f))
        return 0x7Fu;
    uint8_t sign = signbit(f) ? 0x80u : 0x00u;
    float a = fabsf(f);
    if (a > 448.0f)
        return (uint8_t)(sign | 0x7Eu);          /* saturate to 448 */
    if (a == 0.0f)
        return sign;
    int e2;
    frexpf(a, &e2);                 /* a = m * 2^e2, m in [0.5, 1) */
    int E = e2 - 1;                 /* 2^E <= a < 2^(E+1) */
    if (E < -6)
        E = -6;                     /* subnormal range: step 2^-9 */
    float step = ldexpf(1.0f, E - 3);
    float k = rintf(a / step);      /* exact division; rint: nearest even */
    float v = k * step;
    if (v > 448.0f)
        v = 448.0f;
    if (v == 0.0f)
        return sign;
    if (v < ldexpf(1.0f, -6))       /* subnormal: v = k * 2^-9, k in 1..7 */
        return (uint8_t)(sign | (uint8_t)(v / ldexpf(1.0f, -9)));
    frexpf(v, &e2);
    E = e2 - 1;
    int mant = (int)((v / ldexpf(1.0f, E) - 1.0f) * 8.0f);
    return (uint8_t)(sign | (uint8_t)((E + 7) << 3) | (uint8_t)mant);
}

/* One row: returns the scale, writes q[0..H). */
float oracle_quant_e4m3_row(const uint16_t *norm, int64_t H, uint8_t *q)
{
    float amax = 0.0f;
    for (int64_t h = 0; h < H; ++h) {
        float v = fabsf(oracle_bf16_to_f32(norm[h]));
        if (v > amax)               /* NaN never compares greater */
            amax = v;
    }
    float scale = amax > 0.0f ? amax / 448.0f : 1.0f;
    float inv = amax > 0.0f ? 448.0f / amax : 1.0f;
    for (int64_t h = 0; h < H; ++h)
        q[h] = oracle_f32_to_e4m3_sat(oracle_bf16_to_f32(norm[h]) * inv);
    return scale;
}

/* ---------------------------------------------------------------------
 * Fused NVFP4 quantisation of norm_out (also not described by the page:
 * the 4-bit input of a block-scaled GEMM).
 *
 * E2M1: 1 sign bit, 2 exponent bits (bias 1), 1 fraction bit; magnitudes
 * 0, 0.5 (the one subnormal), 1, 1.5, 2, 3, 4, 6; no infinities, no NaN.
 * NVFP4 groups 16 consecutive elements of a row into a block that shares
 * one positive E4M3 scale, under one fp32 scale for the whole tensor.
 *
 * Reading: the tensor scale g (fp32, finite, > 0) is an input of the call
 * (a calibrated constant: a fused kernel cannot see the whole tensor's
 * amax before it writes the first block).  For block b of row t
 * (elements 16b .. 16b+15):
 *     amax   = the largest |norm_out| of the block (NaN ignored)
 *     s[t,b] = E4M3((amax / 6) * g)            saturating, as above
 *     inv    = g / e4m3_value(s[t,b])           one fp32 division
 *     q[t,h] = E2M1(norm_out[t,h] * inv)        round to nearest even,
 *              magnitudes above 6 (infinity included) saturated to 6
 * and q = 0 for the whole block when e4m3_value(s) is 0 (an all-zero block
 * or one whose scale underflows).  A NaN element, which E2M1 cannot hold,
 * is written as +6 (code 0x7).  The value represented is
 * e2m1_value(q) * e4m3_value(s) / g.
 * Layout: q packs two codes per byte, element 2i in the low nibble and
 * element 2i+1 in the high nibble ([T, H/2] bytes); s is [T, H/16] bytes.
 * ------------------------------------------------------------------- */
float oracle_e2m1_to_f32(uint8_t c)
{
    float sign = (c & 0x8u) ? -1.0f : 1.0f;
    int e = (c >> 1) & 0x3, m = c & 0x1;
    if (e == 0)
        return sign * 0.5f * (float)m;
    return sign * ldexpf(1.0f + 0.5f * (float)m, e - 1);
}

uint8_t oracle_f32_to_e2m1_sat(float f)
{
    if (isnan(f))
        return 0x7u;
    uint8_t sign = signbit(f) ? 0x8u : 0x0u;
    float a = fabsf(f);
    if (a > 6.0f)
        return (uint8_t)(sign | 0x7u);           /* saturate to 6 */
    if (a == 0.0f)
        return sign;
    int e2;
    frexpf(a, &e2);                 /* a = m * 2^e2, m in [0.5, 1) */
    int E = e2 - 1;                 /* 2^E <= a < 2^(E+1) */
    if (E < 0)
        E = 0;                      /* below 1: the subnormal step 0.5 */
    float step = ldexpf(1.0f, E - 1);
    float v = rintf(a / step) * step;   /* exact division; nearest even */
    if (v > 6.0f)
        v = 6.0f;
    if (v == 0.0f)
        return sign;
    if (v < 1.0f)
        return (uint8_t)(sign | 0x1u);           /* 0.5 */
    frexpf(v, &e2);
    E = e2 - 1;
    int mant = (int)((v / ldexpf(1.0f, E) - 1.0f) * 2.0f);
    return (uint8_t)(sign | (uint8_t)((E + 1) << 1) | (uint8_t)mant);
}

/* One row (H a multiple of 16): writes q[0..H/2) and s[0..H/16). */
void oracle_quant_nvfp4_row(const uint16_t *norm, int64_t H, float g, uint8_t *q, uint8_t *s)
{
    for (int64_t b = 0; b < H / 16; ++b) {
        const uint16_t *blk = norm + 16 * b;
        float amax = 0.0f;
        for (int i = 0; i < 16; ++i) {
            float v = fabsf(oracle_bf16_to_f32(blk[i]));
            if (v > amax)           /* NaN never compares greater */
                amax = v;
        }
        s[b] = oracle_f32_to_e4m3_sat((amax / 6.0f) * g);
        float sv = oracle_e4m3_to_f32(s[b]);
        float inv = sv > 0.0f ? g / sv : 0.0f;
        for (int i = 0; i < 16; i += 2) {
            uint8_t lo = 0, hi = 0;
            if (sv > 0.0f) {
                lo = oracle_f32_to_e2m1_sat(oracle_bf16_to_f32(blk[i]) * inv);
                hi = oracle_f32_to_e2m1_sat(oracle_bf16_to_f32(blk[i + 1]) * inv);
            }
            q[8 * b + i / 2] = (uint8_t)(lo | (hi << 4));
        }
    }
}

/* ---------------------------------------------------------------------
 * MoE combine ("local y reduce": the per-token weighted sum of its top-k
 * expert outputs) fused with the same residual add + RMSNorm.  The page
 * names the step but defines neither its weights nor its layout; reading:
 *   expert_out  bf16 [n_slots, H], one row per (token, expert) assignment
 *   index       int32 [T, K], the row of expert_out of token t's k-th
 *               expert; -1 (or any value outside [0, n_slots)) is skipped
 *   gates       fp32 [T, K], the routing weights
 *   reduced[t,h] = bf16(acc), acc = -0; for k in 0..K-1, not skipped:
 *                 acc = acc + (gates[t,k] * f(expert_out[index[t,k], h]))
 *   with the product and the sum each rounded to fp32 (no fused
 *   multiply-add), in k order; then residual_out and norm_out as in
 *   oracle_forward.
 * ------------------------------------------------------------------- */
/* The fp32 accumulator of one element (token row `index_row`/`gates_row`,
 * column h), before its rounding to bf16. */
float oracle_moe_combine_acc(const uint16_t *expert_out, int64_t n_slots,
                             const int32_t *index_row, const float *gates_row, int K,
                             int64_t H, int64_t h)
{
    float acc = -0.0f;
    for (int k = 0; k < K; ++k) {
        int32_t s = index_row[k];
        if (s < 0 || (int64_t)s >= n_slots)
            continue;
        float prod = gates_row[k] * oracle_bf16_to_f32(expert_out[(int64_t)s * H + h]);
        acc = acc + prod;
    }
    return acc;
}

int oracle_moe_combine(const uint16_t *expert_out, int64_t n_slots, const int32_t *index,
                       const float *gates, int K, const uint16_t *residual,
                       const uint16_t *weight, float eps, int64_t T, int64_t H,
                       uint16_t *reduced, uint16_t *residual_out, uint16_t *norm_out)
{
    if (K < 1 || T < 0 || H < 1 || n_slots < 0 || !index || !gates || !residual ||
        !weight || !reduced || !residual_out || !norm_out || (n_slots > 0 && !expert_out))
        return -1;
    for (int64_t t = 0; t < T; ++t) {
        int64_t off = t * H;
        for (int64_t h = 0; h < H; ++h)
            reduced[off + h] = oracle_f32_to_bf16(oracle_moe_combine_acc(
                expert_out, n_slots, index + t * K, gates + t * K, K, H, h));
        oracle_residual_add(reduced + off, residual + off, H, residual_out + off);
        oracle_rmsnorm_row(residual_out + off, weight, eps, H, norm_out + off);
    }
    return 0;
}

