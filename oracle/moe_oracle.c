/*
 * moe_oracle.c -- plain, slow, obviously-correct CPU oracle for the
 * single-GPU MoE layer with router replay and block-scaled FP8.
 *
 * TEST INFRASTRUCTURE ONLY.  Nothing on the product path may call, link or
 * load this file; only the tests, the smoke check and the bench's CPU
 * baseline do.  It shares no code, header or table with the CUDA library.
 *
 * Sources (prime-rl 0.6.0 performance deep dive, "RL at 1T Scale"):
 *   - section "Router replay" (R3): routing decisions made at inference are
 *     captured and replayed on the trainer; the routed-experts payload is a
 *     tensor of shape [num_layers, top_k, seq_len].
 *   - section "FP8 training": block-scaled FP8 as proposed by DeepSeek-V3
 *     (1x128 activation tiles, 128x128 weight blocks, fp32 scales, e4m3).
 *   - section "Parallelism", "Expert parallelism (EP)": tokens are dispatched
 *     to experts and combined back.
 * What the pages leave open (score function, tie-break, SwiGLU, layouts,
 * accumulation order) is fixed by the plainest reading, stated in the
 * comment of the routine that takes it.
 *
 * Every routine below computes the definition directly: no tiling, no
 * fusion, no reordering beyond what the definition states.  Floating point
 * follows C99 IEEE semantics; build with -ffp-contract=off -fno-fast-math so
 * that only the explicit fmaf() calls fuse.
 *
 * Parity status: every function here is pinned by tests/test_oracle_*.py
 * (brute force, closed forms, invariants, library routines).
 */
#include <math.h>
#include <stdint.h>
#include <stdlib.h>
#include <string.h>

#define OR_OK 0
#define OR_ERR_BAD_IDS 5

/* ------------------------------------------------------------------ */
/* scalar formats                                                       */
/* ------------------------------------------------------------------ */

/* bf16 is the upper 16 bits of an IEEE binary32: widening is exact. */
float or_bf16_to_f32(uint16_t h)
{
    uint32_t u = (uint32_t)h << 16;
    float f;
    memcpy(&f, &u, 4);
    return f;
}

/* Round a binary32 to bf16, round-to-nearest-even.  Works on the bit pattern:
 * adding 0x7FFF plus the lowest kept bit rounds the discarded 16 bits to
 * nearest with ties to the even kept value (a carry into the exponent is the
 * correct next binade, and past the largest finite value it gives inf). */
uint16_t or_f32_to_bf16(float f)
{
    uint32_t u;
    memcpy(&u, &f, 4);
    if ((u & 0x7F800000u) == 0x7F800000u && (u & 0x007FFFFFu) != 0)
        return (uint16_t)((u >> 16) | 0x0040u); /* NaN stays a quiet NaN */
    uint32_t keep_lsb = (u >> 16) & 1u;
    u += 0x7FFFu + keep_lsb;
    return (uint16_t)(u >> 16);
}

/* OCP FP8 E4M3 ("e4m3fn"): sign, 4 exponent bits (bias 7), 3 mantissa bits;
 * exponent field 0 is subnormal (m * 2^-9); 0x7F / 0xFF are NaN; no inf;
 * largest finite 0x7E = 1.75 * 2^8 = 448. */
double or_e4m3_decode(uint8_t c)
{
    int sign = (c >> 7) & 1;
    int e = (c >> 3) & 0xF;
    int m = c & 0x7;
    double v;
    if (e == 0xF && m == 0x7)
        return NAN;
    if (e == 0)
        v = ldexp((double)m, -9);
    else
        v = ldexp(1.0 + m / 8.0, e - 7);
    return sign ? -v : v;
}

/* Encode a finite binary32 as E4M3, round-to-nearest-even, saturating to
 * +-448 (the "satfinite" rule: a value whose rounding would leave the finite
 * range becomes the largest finite code).  The sign is kept, so -0 -> 0x80.
 *
 * Rounding: the E4M3 grid spacing in the binade [2^e, 2^(e+1)) is 2^(e-3)
 * for e >= -6 and 2^-9 below 2^-6 (subnormals).  Dividing by that power of
 * two is exact in double, rint() rounds to the nearest integer with ties to
 * even, and multiplying back is exact. */
uint8_t or_e4m3_encode(float v)
{
    uint8_t sign = signbit(v) ? 0x80 : 0x00;
    double a = fabs((double)v);
    if (isnan(v))
        return 0x7F;
    if (a == 0.0)
        return sign;
    int ex;
    frexp(a, &ex);          /* a = f * 2^ex, f in [0.5, 1) -> binade 2^(ex-1) */
    int e = ex - 1;
    int qexp = (e < -6) ? -9 : e - 3;
    double n = rint(ldexp(a, -qexp));
    double r = ldexp(n, qexp);
    if (r > 448.0)
        r = 448.0;
    if (r == 0.0)
        return sign;
    /* r is now an exact E4M3 value; write its bit fields. */
    frexp(r, &ex);
    e = ex - 1;
    uint8_t code;
    if (e < -6) {
        code = (uint8_t)ldexp(r, 9);                  /* subnormal: m = r / 2^-9 */
    } else {
        int m = (int)(ldexp(r, -e) * 8.0) - 8;        /* r = 2^e * (1 + m/8) */
        code = (uint8_t)(((e + 7) << 3) | m);
    }
    return (uint8_t)(sign | code);
}

/* ------------------------------------------------------------------ */
/* block-scaled quantisation (DeepSeek-V3 recipe, "FP8 training")       */
/* ------------------------------------------------------------------ */

/* One block: amax over its elements, s = amax / 448 (IEEE binary32
 * division), code = e4m3(v / s) with IEEE division.  An all-zero block (or a
 * block so small that amax / 448 underflows to zero) takes s = 1. */
static float block_scale(float amax)
{
    float s = amax / 448.0f;
    if (s == 0.0f)
        s = 1.0f;
    return s;
}

/* Activations: 1 x 128 blocks along each row.  src [rows, cols] bf16 with row
 * stride ld_src elements; q [rows, cols] e4m3; s [rows, cols/128] fp32. */
void or_quant_1x128(const uint16_t *src, int64_t rows, int64_t cols, int64_t ld_src,
                    uint8_t *q, float *s)
{
    int64_t nb = cols / 128;
#pragma omp parallel for schedule(static)
    for (int64_t r = 0; r < rows; r++) {
        for (int64_t b = 0; b < nb; b++) {
            const uint16_t *v = src + r * ld_src + b * 128;
            float amax = 0.0f;
            for (int i = 0; i < 128; i++) {
                float a = fabsf(or_bf16_to_f32(v[i]));
                if (a > amax)
                    amax = a;
            }
            float sc = block_scale(amax);
            s[r * nb + b] = sc;
            for (int i = 0; i < 128; i++)
                q[r * cols + b * 128 + i] = or_e4m3_encode(or_bf16_to_f32(v[i]) / sc);
        }
    }
}

/* Weights: 128 x 128 blocks.  src [rows, cols] bf16; q [rows, cols];
 * s [rows/128, cols/128]. */
void or_quant_128x128(const uint16_t *src, int64_t rows, int64_t cols, int64_t ld_src,
                      uint8_t *q, float *s)
{
    int64_t nbr = rows / 128, nbc = cols / 128;
#pragma omp parallel for schedule(static)
    for (int64_t br = 0; br < nbr; br++) {
        for (int64_t bc = 0; bc < nbc; bc++) {
            float amax = 0.0f;
            for (int64_t i = 0; i < 128; i++)
                for (int64_t j = 0; j < 128; j++) {
                    float a = fabsf(or_bf16_to_f32(src[(br * 128 + i) * ld_src + bc * 128 + j]));
                    if (a > amax)
                        amax = a;
                }
            float sc = block_scale(amax);
            s[br * nbc + bc] = sc;
            for (int64_t i = 0; i < 128; i++)
                for (int64_t j = 0; j < 128; j++) {
                    int64_t r = br * 128 + i, c = bc * 128 + j;
                    q[r * cols + c] = or_e4m3_encode(or_bf16_to_f32(src[r * ld_src + c]) / sc);
                }
        }
    }
}

/* Power-of-two (UE8M0) variant of the block scale: s = 2^p with p the
 * smallest integer such that amax <= 448 * 2^p, so that no code saturates;
 * stored as the biased exponent e = p + 127 (one byte, s = 2^(e-127)).  An
 * all-zero block takes e = 127 (s = 1).  p is clamped to [-127, 127]; the
 * upper clamp is never reached by a finite bf16 input. */
static int ue8m0_exponent(float amax)
{
    if (amax == 0.0f)
        return 127;
    int ex;
    frexp((double)amax, &ex);
    int p = ex - 10;                        /* 448 * 2^(ex-10) < 2^(ex-1) <= amax */
    while (ldexp(448.0, p) < (double)amax)
        p++;
    if (p < -127)
        p = -127;
    if (p > 127)
        p = 127;
    return p + 127;
}

/* Block quantisation with power-of-two scales: blocks of block_rows (1 or
 * 128) x 128 elements, code = e4m3(v / 2^(e-127)) (an exact division),
 * e [rows/block_rows, cols/128] biased exponents. */
void or_quant_ue8m0(const uint16_t *src, int64_t rows, int64_t cols, int64_t ld_src, int block_rows,
                    uint8_t *q, uint8_t *e)
{
    int64_t nbr = rows / block_rows, nbc = cols / 128;
#pragma omp parallel for schedule(static)
    for (int64_t br = 0; br < nbr; br++) {
        for (int64_t bc = 0; bc < nbc; bc++) {
            float amax = 0.0f;
            for (int64_t i = 0; i < block_rows; i++)
                for (int64_t j = 0; j < 128; j++) {
                    float a = fabsf(or_bf16_to_f32(src[(br * block_rows + i) * ld_src + bc * 128 + j]));
                    if (a > amax)
                        amax = a;
                }
            int ebias = ue8m0_exponent(amax);
            e[br * nbc + bc] = (uint8_t)ebias;
            float sc = (float)ldexp(1.0, ebias - 127);
            for (int64_t i = 0; i < block_rows; i++)
                for (int64_t j = 0; j < 128; j++) {
                    int64_t r = br * block_rows + i, c = bc * 128 + j;
                    q[r * cols + c] = or_e4m3_encode(or_bf16_to_f32(src[r * ld_src + c]) / sc);
                }
        }
    }
}

/* ------------------------------------------------------------------ */
/* routing ("Router replay": the decision that is captured)             */
/* ------------------------------------------------------------------ */
/* NVFP4: FP4 E2M1 values, 16-element blocks with E4M3 scales, and one  */
/* fp32 scale per tensor (the FP4 variant the pages list as future work, */
/* "RL at 1T Scale", closing section; the format is NVIDIA's published   */
/* NVFP4, taken as the plainest reading)                                 */
/* ------------------------------------------------------------------ */

/* E2M1 (low 4 bits of code): sign bit 3, exponent bits 2..1 (bias 1),
 * mantissa bit 0; exponent 0 is subnormal (m * 0.5).  Magnitudes of codes
 * 0..7: 0, 0.5, 1, 1.5, 2, 3, 4, 6.  No inf, no NaN. */
double or_e2m1_decode(uint8_t code)
{
    int sign = (code >> 3) & 1;
    int e = (code >> 1) & 3;
    int m = code & 1;
    double v = (e == 0) ? 0.5 * m : ldexp(1.0 + 0.5 * m, e - 1);
    return sign ? -v : v;
}

/* Round a binary32 to E2M1, nearest with ties to even, saturating to +-6
 * (a value whose rounding leaves the range becomes 6).  The sign is kept
 * (-0 -> 0x8).  The grid spacing is 0.5 below 2, 1 in [2, 4) and 2 in
 * [4, 8): dividing by it is exact in double and rint() rounds to the
 * nearest integer with ties to even, which is the even-mantissa code.  NaN
 * is outside the contract (the quantiser's inputs are finite). */
uint8_t or_e2m1_encode(float v)
{
    uint8_t sign = signbit(v) ? 0x8 : 0x0;
    double a = fabs((double)v);
    double step = a < 2.0 ? 0.5 : (a < 4.0 ? 1.0 : 2.0);
    double r = rint(a / step) * step;
    if (r > 6.0)
        r = 6.0;
    uint8_t code;
    if (r == 0.0)
        code = 0;
    else if (r < 1.0)
        code = 1;                                    /* 0.5, subnormal */
    else {
        int ex;
        frexp(r, &ex);                               /* r in [2^(ex-1), 2^ex) */
        int e = ex - 1;                              /* 0, 1 or 2 */
        int m = ldexp(r, -e) > 1.0 ? 1 : 0;          /* 1.5 * 2^e -> m = 1 */
        code = (uint8_t)(((e + 1) << 1) | m);
    }
    return (uint8_t)(sign | code);
}

/* NVFP4 quantisation of a [rows, cols] bf16 tensor (row stride ld_src),
 * blocks of 16 consecutive elements along each row (the contraction
 * dimension of the GEMM that consumes it):
 *   s_enc = (6 * 448) / amax over the whole tensor   (binary32 division;
 *           an all-zero tensor takes s_enc = 1),
 *   block scale byte sb = e4m3((amax_block / 6) * s_enc)  (binary32 division
 *           and product, then round-to-nearest-even saturating E4M3),
 *   per element: s_elem = s_enc / e4m3value(sb) (binary32; 0 when the scale
 *           byte decodes to 0), code = e2m1(x * s_elem).
 * Decoded value: e2m1value(code) * e4m3value(sb) / s_enc.
 * q [rows, cols/2]: element 2i in the low nibble of byte i, 2i+1 in the high
 * nibble; s [rows, cols/16] E4M3 bytes; *s_enc_out the tensor's s_enc. */
void or_quant_nvfp4(const uint16_t *src, int64_t rows, int64_t cols, int64_t ld_src, uint8_t *q, uint8_t *s,
                    float *s_enc_out)
{
    float amax_t = 0.0f;
    for (int64_t r = 0; r < rows; r++)
        for (int64_t c = 0; c < cols; c++)
            amax_t = fmaxf(amax_t, fabsf(or_bf16_to_f32(src[r * ld_src + c])));
    const float s_enc = amax_t == 0.0f ? 1.0f : (6.0f * 448.0f) / amax_t;
    *s_enc_out = s_enc;
    const int64_t nb = cols / 16;
#pragma omp parallel for schedule(static)
    for (int64_t r = 0; r < rows; r++)
        for (int64_t b = 0; b < nb; b++) {
            const uint16_t *x = src + r * ld_src + b * 16;
            float amax = 0.0f;
            for (int i = 0; i < 16; i++)
                amax = fmaxf(amax, fabsf(or_bf16_to_f32(x[i])));
            const float bd = amax / 6.0f;
            const uint8_t sb = or_e4m3_encode(bd * s_enc);
            s[r * nb + b] = sb;
            const float sbv = (float)or_e4m3_decode(sb);
            const float s_elem = sbv == 0.0f ? 0.0f : s_enc / sbv;
            for (int i = 0; i < 16; i += 2) {
                const uint8_t lo = or_e2m1_encode(or_bf16_to_f32(x[i]) * s_elem);
                const uint8_t hi = or_e2m1_encode(or_bf16_to_f32(x[i + 1]) * s_elem);
                q[r * (cols / 2) + b * 8 + i / 2] = (uint8_t)(lo | (hi << 4));
            }
        }
}

/* Sum over k (ascending) of e2m1(a_k) * e4m3(sa) * e2m1(b_k) * e4m3(sb) for
 * one row of each NVFP4 operand (packed codes, 16-element block scales).
 * Each product has at most 12 significant bits and lies in [2^-20, 2^23],
 * so the sum is exact for K <= 1024 (and rounded in ascending k beyond). */
static double nvfp4_dot(const uint8_t *aq, const uint8_t *as, const uint8_t *bq, const uint8_t *bs, int64_t K)
{
    double acc = 0.0;
    for (int64_t k = 0; k < K; k++) {
        const uint8_t ab = aq[k / 2], bb = bq[k / 2];
        const double av = or_e2m1_decode((k & 1) ? (ab >> 4) : (ab & 15)) * or_e4m3_decode(as[k / 16]);
        const double bv = or_e2m1_decode((k & 1) ? (bb >> 4) : (bb & 15)) * or_e4m3_decode(bs[k / 16]);
        acc += av * bv;
    }
    return acc;
}

/* out[m, n] = sum over k of dec(a[m, k]) * dec(b[n, k]) for NVFP4 operands
 * a [M, K] and b [N, K] as or_quant_nvfp4 writes them (K a multiple of 16):
 * nvfp4_dot / (a_enc * b_enc) in double (a_enc * b_enc is exact; one
 * division rounds).  The tensor-core result (fp32, order unspecified) is
 * compared with this. */
void or_gemm_nvfp4(const uint8_t *aq, const uint8_t *as, float a_enc, const uint8_t *bq, const uint8_t *bs,
                   float b_enc, int64_t M, int64_t N, int64_t K, double *out)
{
    const double enc = (double)a_enc * (double)b_enc;
#pragma omp parallel for schedule(static)
    for (int64_t m = 0; m < M; m++)
        for (int64_t n = 0; n < N; n++)
            out[m * N + n] = nvfp4_dot(aq + m * (K / 2), as + m * (K / 16), bq + n * (K / 2), bs + n * (K / 16), K) /
                             enc;
}

/* SwiGLU expert FFN in NVFP4 on n sorted rows (row r belongs to expert
 * row_expert[r]):
 *   x rows: NVFP4 with one tensor scale x_enc (the token tensor's);
 *   w13[e] [2F, d] and w2[e] [d, F]: NVFP4 with one tensor scale per expert
 *     matrix (w13_enc[e], w2_enc[e]);
 *   h = the exact GEMM1 value rounded once to binary32 (gate columns 0..F-1,
 *     up F..2F-1);
 *   act = silu(g) * u in double rounded to binary32 (the recipe FFN's
 *     formula), then to bf16 -- the act tensor is materialised, because its
 *     NVFP4 tensor scale needs the amax over all n rows first;
 *   act [n, F] -> NVFP4 (or_quant_nvfp4: one tensor scale act_enc);
 *   out = bf16(binary32(exact GEMM2 value)).
 * h [n, 2F] f32 and act_bf16 [n, F] are outputs; act_q [n, F/2], act_s
 * [n, F/16], *act_enc; out [n, d] bf16.  d, F multiples of 16. */
void or_expert_ffn_nvfp4(const uint8_t *xq, const uint8_t *xs, float x_enc, int64_t n, const int32_t *row_expert,
                         int d, int F, const uint8_t *w13_q, const uint8_t *w13_s, const float *w13_enc,
                         const uint8_t *w2_q, const uint8_t *w2_s, const float *w2_enc, float *h, uint16_t *act_bf16,
                         uint8_t *act_q, uint8_t *act_s, float *act_enc, uint16_t *out)
{
#pragma omp parallel for schedule(dynamic, 1)
    for (int64_t r = 0; r < n; r++) {
        const int64_t e = row_expert[r];
        const double enc = (double)x_enc * (double)w13_enc[e];
        for (int64_t j = 0; j < 2 * F; j++) {
            const int64_t wrow = e * 2 * F + j;
            h[r * 2 * F + j] = (float)(nvfp4_dot(xq + r * (d / 2), xs + r * (d / 16), w13_q + wrow * (d / 2),
                                                 w13_s + wrow * (d / 16), d) /
                                       enc);
        }
        for (int64_t c = 0; c < F; c++) {
            const double g = h[r * 2 * F + c], u = h[r * 2 * F + F + c];
            act_bf16[r * F + c] = or_f32_to_bf16((float)((g / (1.0 + exp(-g))) * u));
        }
    }
    or_quant_nvfp4(act_bf16, n, F, F, act_q, act_s, act_enc);
#pragma omp parallel for schedule(dynamic, 1)
    for (int64_t r = 0; r < n; r++) {
        const int64_t e = row_expert[r];
        const double enc = (double)(*act_enc) * (double)w2_enc[e];
        for (int64_t c = 0; c < d; c++) {
            const int64_t wrow = e * d + c;
            const double v = nvfp4_dot(act_q + r * (F / 2), act_s + r * (F / 16), w2_q + wrow * (F / 2),
                                       w2_s + wrow * (F / 16), F) /
                             enc;
            out[r * d + c] = or_f32_to_bf16((float)v);
        }
    }
}

/* ------------------------------------------------------------------ */

/* l[t,e] = sum_i x[t,i] * Wr[e,i] as one binary32 fused-multiply-add chain in
 * ascending i, starting from +0. */
void or_router_logits(const uint16_t *x, const uint16_t *wr, int64_t T, int d, int E,
                      float *logits)
{
#pragma omp parallel for schedule(static)
    for (int64_t t = 0; t < T; t++)
        for (int e = 0; e < E; e++) {
            float acc = 0.0f;
            for (int i = 0; i < d; i++)
                acc = fmaf(or_bf16_to_f32(x[t * d + i]), or_bf16_to_f32(wr[(int64_t)e * d + i]), acc);
            logits[t * E + e] = acc;
        }
}

/* Selection order: larger logit first; equal logits (including -0 == +0)
 * go to the lower expert index; NaN ranks below every number. */
static int ranks_before(float a, int ia, float b, int ib)
{
    int na = isnan(a), nb = isnan(b);
    if (na != nb)
        return nb;              /* a number beats NaN */
    if (!na && a != b)
        return a > b;
    return ia < ib;
}

/* Top-k by repeated selection of the best unselected expert; slot j holds the
 * j-th pick. */
void or_topk(const float *logits, int64_t T, int E, int k, int32_t *ids)
{
#pragma omp parallel for schedule(static)
    for (int64_t t = 0; t < T; t++) {
        const float *l = logits + t * E;
        unsigned char *taken = calloc((size_t)E, 1);
        for (int j = 0; j < k; j++) {
            int best = -1;
            for (int e = 0; e < E; e++) {
                if (taken[e])
                    continue;
                if (best < 0 || ranks_before(l[e], e, l[best], best))
                    best = e;
            }
            taken[best] = 1;
            ids[t * k + j] = best;
        }
        free(taken);
    }
}

/* Gate weights over the chosen experts, in double, rounded once to binary32.
 *   softmax: p_e = exp(l_e) / sum over all experts; renorm divides by the sum
 *            over the chosen ones (the full denominator cancels).
 *   sigmoid: p_e = 1 / (1 + exp(-l_e)); renorm divides by the chosen sum.
 * The result is multiplied by route_scale.  Tokens flagged invalid (valid !=
 * NULL and valid[t] == 0) get zero gates. */
void or_gates(const float *logits, const int32_t *ids, const uint8_t *valid, int64_t T, int E, int k,
              int score_fn, int renorm, float route_scale, float *gates)
{
#pragma omp parallel for schedule(static)
    for (int64_t t = 0; t < T; t++) {
        const float *l = logits + t * E;
        if (valid && !valid[t]) {
            for (int j = 0; j < k; j++)
                gates[t * k + j] = 0.0f;
            continue;
        }
        double p[64];
        double denom = 0.0;
        if (score_fn == 0) {
            double m = -INFINITY;
            if (renorm) {
                for (int j = 0; j < k; j++)
                    if (l[ids[t * k + j]] > m)
                        m = l[ids[t * k + j]];
                for (int j = 0; j < k; j++)
                    denom += exp((double)l[ids[t * k + j]] - m);
            } else {
                for (int e = 0; e < E; e++)
                    if (l[e] > m)
                        m = l[e];
                for (int e = 0; e < E; e++)
                    denom += exp((double)l[e] - m);
            }
            for (int j = 0; j < k; j++)
                p[j] = exp((double)l[ids[t * k + j]] - m) / denom;
        } else {
            for (int j = 0; j < k; j++) {
                p[j] = 1.0 / (1.0 + exp(-(double)l[ids[t * k + j]]));
                denom += p[j];
            }
            for (int j = 0; j < k; j++)
                if (renorm)
                    p[j] = p[j] / denom;
        }
        for (int j = 0; j < k; j++)
            gates[t * k + j] = (float)(p[j] * (double)route_scale);
    }
}

/* Backward of the router for a fixed choice of experts ("RL at 1T Scale",
 * "Router replay": the trainer replays the captured ids and still trains the
 * router through the gates it recomputes from their logits).  Given
 * d_gates[t,j] = dL/dg[t,j]:
 *   l_j = x[t] . Wr[ids[t,j]], the binary32 fma chain of or_router_logits;
 *   the gate function's derivative, in double (rs = route_scale):
 *     softmax, renorm:    p_j = exp(l_j) / sum_{i<k} exp(l_i),
 *                         dl_m = rs * p_m * (dg_m - sum_j dg_j p_j)
 *     sigmoid, renorm:    s_j = 1 / (1 + exp(-l_j)), S = sum_{i<k} s_i,
 *                         dl_m = rs * s_m (1 - s_m) * (dg_m - sum_j dg_j s_j / S) / S
 *     sigmoid, no renorm: dl_m = rs * dg_m * s_m (1 - s_m)
 *   (softmax without renorm depends on every expert's logit: not handled),
 *   rounded once to binary32 as d_logits[t,j]; a token with valid[t] == 0
 *   (valid nullable) gets zeros;
 *   dx[t, c] = sum_j d_logits[t,j] * Wr[ids[t,j], c] and
 *   dw[e, c] = sum over the (t, j) with ids[t,j] == e of d_logits[t,j] * x[t, c],
 *   both summed in double and rounded once to binary32 (dx, dw nullable). */
void or_router_backward(const uint16_t *x, const uint16_t *wr, const int32_t *ids, const uint8_t *valid,
                        const float *d_gates, int64_t T, int d, int E, int k, int score_fn, int renorm,
                        float route_scale, float *d_logits, float *dx, float *dw)
{
#pragma omp parallel for schedule(static)
    for (int64_t t = 0; t < T; t++) {
        const int32_t *id = ids + t * k;
        const float *dg = d_gates + t * k;
        if (valid && !valid[t]) {
            for (int j = 0; j < k; j++)
                d_logits[t * k + j] = 0.0f;
            continue;
        }
        double l[64], p[64], dl[64];
        for (int j = 0; j < k; j++) {
            float acc = 0.0f;
            for (int i = 0; i < d; i++)
                acc = fmaf(or_bf16_to_f32(x[t * d + i]), or_bf16_to_f32(wr[(int64_t)id[j] * d + i]), acc);
            l[j] = acc;
        }
        const double rs = route_scale;
        if (score_fn == 0) {
            double m = -INFINITY, den = 0.0, dot = 0.0;
            for (int j = 0; j < k; j++)
                if (l[j] > m)
                    m = l[j];
            for (int j = 0; j < k; j++) {
                p[j] = exp(l[j] - m);
                den += p[j];
            }
            for (int j = 0; j < k; j++) {
                p[j] /= den;
                dot += (double)dg[j] * p[j];
            }
            for (int j = 0; j < k; j++)
                dl[j] = rs * p[j] * ((double)dg[j] - dot);
        } else {
            double S = 0.0, dot = 0.0;
            for (int j = 0; j < k; j++) {
                p[j] = 1.0 / (1.0 + exp(-l[j]));
                S += p[j];
                dot += (double)dg[j] * p[j];
            }
            for (int j = 0; j < k; j++) {
                const double ds = p[j] * (1.0 - p[j]);
                dl[j] = renorm ? rs * ds * ((double)dg[j] - dot / S) / S : rs * (double)dg[j] * ds;
            }
        }
        for (int j = 0; j < k; j++)
            d_logits[t * k + j] = (float)dl[j];
    }
    if (dx) {
#pragma omp parallel for schedule(static)
        for (int64_t t = 0; t < T; t++)
            for (int c = 0; c < d; c++) {
                double acc = 0.0;
                for (int j = 0; j < k; j++)
                    if (!valid || valid[t])
                        acc += (double)d_logits[t * k + j] * or_bf16_to_f32(wr[(int64_t)ids[t * k + j] * d + c]);
                dx[t * d + c] = (float)acc;
            }
    }
    if (dw) {
#pragma omp parallel for schedule(dynamic)
        for (int e = 0; e < E; e++) {
            double *acc = calloc((size_t)d, sizeof(double));
            for (int64_t t = 0; t < T; t++) {
                if (valid && !valid[t])
                    continue;
                for (int j = 0; j < k; j++)
                    if (ids[t * k + j] == e) {
                        const double g = d_logits[t * k + j];
                        for (int c = 0; c < d; c++)
                            acc[c] += g * or_bf16_to_f32(x[t * d + c]);
                    }
            }
            for (int c = 0; c < d; c++)
                dw[(int64_t)e * d + c] = (float)acc[c];
            free(acc);
        }
    }
}

/* Replay one layer slice of the routed-experts payload: payload_kT is
 * [top_k, seq_len] row-major (the layer's slab of [num_layers, top_k,
 * seq_len]); ids[t, j] = payload_kT[j, t], an exact copy in slot order.
 * A token is valid when its k ids are in [0, E) and pairwise distinct.
 * valid[t] (nullable) receives 1/0; returns the number of invalid tokens. */
int64_t or_replay(const int32_t *payload_kT, int64_t T, int E, int k, int32_t *ids, uint8_t *valid)
{
    int64_t bad = 0;
    for (int64_t t = 0; t < T; t++) {
        int ok = 1;
        for (int j = 0; j < k; j++) {
            int32_t v = payload_kT[(int64_t)j * T + t];
            ids[t * k + j] = v;
            if (v < 0 || v >= E)
                ok = 0;
            for (int i = 0; i < j; i++)
                if (ids[t * k + i] == v)
                    ok = 0;
        }
        if (valid)
            valid[t] = (uint8_t)ok;
        if (!ok)
            bad++;
    }
    return bad;
}

/* Compact the routed-experts payload to one byte per id ("Router replay":
 * the captured [num_layers, top_k, seq_len] payload is large and is moved as
 * an opaque tensor).  With E <= 256 every valid id fits a byte:
 * out[i] = ids[i] for 0 <= ids[i] < E.  An id outside [0, E) is stored as
 * 0xFF and counted; returns the number of such ids. */
int64_t or_payload_pack_u8(const int32_t *ids, int64_t n, int E, uint8_t *out)
{
    int64_t bad = 0;
    for (int64_t i = 0; i < n; i++) {
        if (ids[i] >= 0 && ids[i] < E && ids[i] <= 255) {
            out[i] = (uint8_t)ids[i];
        } else {
            out[i] = 0xFF;
            bad++;
        }
    }
    return bad;
}

/* Widen a one-byte payload back to int32 ids: out[i] = in[i]. */
void or_payload_unpack_u8(const uint8_t *in, int64_t n, int32_t *out)
{
    for (int64_t i = 0; i < n; i++)
        out[i] = (int32_t)in[i];
}

/* ------------------------------------------------------------------ */
/* dispatch ("Expert parallelism": tokens to experts and back)          */
/* ------------------------------------------------------------------ */

/* Counting sort of the slots s = t*k + j by expert id, visiting slots in
 * ascending order (stable).  counts[e] = slots routed to e; offsets is the
 * exclusive prefix sum (offsets[E] = routed slots); sorted_to_slot[r] is the
 * slot at sorted position r; slot_to_sorted is its inverse.  Slots whose id is
 * out of [0, E) are not routed: slot_to_sorted = -1, and sorted_to_slot has
 * only offsets[E] entries (the rest are set to -1).  Returns the number of
 * such slots. */
int64_t or_dispatch(const int32_t *ids, int64_t T, int k, int E, int32_t *counts, int32_t *offsets,
                    int32_t *sorted_to_slot, int32_t *slot_to_sorted)
{
    int64_t A = T * (int64_t)k, dropped = 0;
    for (int e = 0; e < E; e++)
        counts[e] = 0;
    for (int64_t s = 0; s < A; s++) {
        if (ids[s] >= 0 && ids[s] < E)
            counts[ids[s]]++;
        else
            dropped++;
    }
    offsets[0] = 0;
    for (int e = 0; e < E; e++)
        offsets[e + 1] = offsets[e] + counts[e];
    int32_t *next = malloc(sizeof(int32_t) * (size_t)(E > 0 ? E : 1));
    for (int e = 0; e < E; e++)
        next[e] = offsets[e];
    for (int64_t r = 0; r < A; r++)
        sorted_to_slot[r] = -1;
    for (int64_t s = 0; s < A; s++) {
        int32_t e = ids[s];
        if (e < 0 || e >= E) {
            slot_to_sorted[s] = -1;
            continue;
        }
        int32_t r = next[e]++;
        sorted_to_slot[r] = (int32_t)s;
        slot_to_sorted[s] = r;
    }
    free(next);
    return dropped;
}

/* rows_sorted[r] = rows[sorted_to_slot[r] / k] for the first n_sorted rows
 * (byte rows of row_bytes each). */
void or_gather_rows(const uint8_t *rows, int64_t row_bytes, const int32_t *sorted_to_slot,
                    int64_t n_sorted, int k, uint8_t *rows_sorted)
{
    for (int64_t r = 0; r < n_sorted; r++) {
        int64_t t = sorted_to_slot[r] / k;
        memcpy(rows_sorted + r * row_bytes, rows + t * row_bytes, (size_t)row_bytes);
    }
}

/* ------------------------------------------------------------------ */
/* expert FFN: SwiGLU with block-scaled FP8 GEMMs ("FP8 training")      */
/* ------------------------------------------------------------------ */

/* One 128-long block of a dot product of E4M3 codes.  Each product of two
 * E4M3 values has at most 8 significant bits and lies in [2^-18, 2^17.6], so
 * every partial sum of 128 of them is an exact double; the order of the
 * additions therefore cannot matter and the result is the exact block sum. */
static double e4m3_block_dot(const uint8_t *a, const uint8_t *b, const double *dec)
{
    double s = 0.0;
    for (int i = 0; i < 128; i++)
        s += dec[a[i]] * dec[b[i]];
    return s;
}

/* out[n] = sum over K blocks kb of (sa[kb] * sb[n/128, kb]) * P_kb(n), where
 * P_kb is the exact block dot product rounded to binary32 (what an ideal FP8
 * MMA with an fp32 accumulator yields for one 128-deep block) and the sum
 * over kb is a binary32 fma chain in ascending kb -- the per-128 "promotion"
 * of the DeepSeek-V3 recipe.  a: one row [K] of codes, sa: its [K/128]
 * scales; w: [N, K] codes, sw: [N/128, K/128]. */
static void fp8_row_gemm(const uint8_t *a, const float *sa, const uint8_t *w, const float *sw,
                         int64_t N, int64_t K, const double *dec, float *out)
{
    int64_t nkb = K / 128;
    for (int64_t n = 0; n < N; n++) {
        float acc = 0.0f;
        for (int64_t kb = 0; kb < nkb; kb++) {
            float p = (float)e4m3_block_dot(a + kb * 128, w + n * K + kb * 128, dec);
            float sc = sa[kb] * sw[(n / 128) * nkb + kb];
            acc = fmaf(sc, p, acc);
        }
        out[n] = acc;
    }
}

/* The block-scaled GEMM alone: out [M, N] fp32 = A [M, K] (scales [M, K/128])
 * times W [N, K] (scales [N/128, K/128]) transposed, by fp8_row_gemm. */
void or_fp8_gemm(const uint8_t *a, const float *sa, int64_t M, const uint8_t *w, const float *sw,
                 int64_t N, int64_t K, float *out)
{
    double dec[256];
    for (int c = 0; c < 256; c++)
        dec[c] = or_e4m3_decode((uint8_t)c);
#pragma omp parallel for schedule(static)
    for (int64_t m = 0; m < M; m++)
        fp8_row_gemm(a + m * K, sa + m * (K / 128), w, sw, N, K, dec, out + m * N);
}

/* SwiGLU expert FFN on n sorted rows.  Row r belongs to expert
 * row_expert[r], an index into the weight arrays:
 *   w13_q [*, 2F, d] (rows 0..F-1 gate, F..2F-1 up), w13_s [*, 2F/128, d/128]
 *   w2_q  [*, d, F],                                 w2_s  [*, d/128, F/128]
 * h = X W13^T (block-scaled), act = silu(h_gate) * h_up in double rounded to
 * binary32, act re-quantised 1x128 along F, out = bf16(act_q W2^T).
 * act_f (nullable) [n, F], act_q [n, F], act_s [n, F/128], out [n, d].
 * ue8m0 = 0: act scales amax/448 (fp32); 1: power-of-two scales as
 * or_quant_ue8m0 (act_s holds their values). */
void or_expert_ffn_rule(const uint8_t *xq, const float *xs, int64_t n, const int32_t *row_expert, int d,
                        int F, const uint8_t *w13_q, const float *w13_s, const uint8_t *w2_q, const float *w2_s,
                        int ue8m0, float *act_f, uint8_t *act_q, float *act_s, uint16_t *out)
{
    double dec[256];
    for (int c = 0; c < 256; c++)
        dec[c] = or_e4m3_decode((uint8_t)c);
    int64_t nkd = d / 128, nkf = F / 128;
#pragma omp parallel for schedule(dynamic, 1)
    for (int64_t r = 0; r < n; r++) {
        int64_t e = row_expert[r];
        float *h = malloc(sizeof(float) * 2 * (size_t)F);
        float *o = malloc(sizeof(float) * (size_t)d);
        float *act = malloc(sizeof(float) * (size_t)F);
        fp8_row_gemm(xq + r * d, xs + r * nkd, w13_q + e * 2 * F * (int64_t)d,
                     w13_s + e * (2 * F / 128) * nkd, 2 * F, d, dec, h);
        for (int64_t c = 0; c < F; c++) {
            double g = h[c], u = h[F + c];
            act[c] = (float)((g / (1.0 + exp(-g))) * u);
        }
        for (int64_t b = 0; b < nkf; b++) {
            float amax = 0.0f;
            for (int i = 0; i < 128; i++)
                if (fabsf(act[b * 128 + i]) > amax)
                    amax = fabsf(act[b * 128 + i]);
            float sc = ue8m0 ? (float)ldexp(1.0, ue8m0_exponent(amax) - 127) : block_scale(amax);
            act_s[r * nkf + b] = sc;
            for (int i = 0; i < 128; i++)
                act_q[r * F + b * 128 + i] = or_e4m3_encode(act[b * 128 + i] / sc);
        }
        if (act_f)
            memcpy(act_f + r * F, act, sizeof(float) * (size_t)F);
        fp8_row_gemm(act_q + r * F, act_s + r * nkf, w2_q + e * (int64_t)d * F,
                     w2_s + e * (d / 128) * nkf, d, F, dec, o);
        for (int64_t c = 0; c < d; c++)
            out[r * d + c] = or_f32_to_bf16(o[c]);
        free(h);
        free(o);
        free(act);
    }
}

/* The recipe's FFN: fp32 amax/448 scales for the act re-quantisation. */
void or_expert_ffn(const uint8_t *xq, const float *xs, int64_t n, const int32_t *row_expert, int d, int F,
                   const uint8_t *w13_q, const float *w13_s, const uint8_t *w2_q, const float *w2_s,
                   float *act_f, uint8_t *act_q, float *act_s, uint16_t *out)
{
    or_expert_ffn_rule(xq, xs, n, row_expert, d, F, w13_q, w13_s, w2_q, w2_s, 0, act_f, act_q, act_s, out);
}

/* ------------------------------------------------------------------ */
/* combine                                                              */
/* ------------------------------------------------------------------ */

/* y[t] = bf16( sum_j g[t,j] * out_sorted[slot_to_sorted[t*k+j]] ), a binary32
 * fma chain over j in slot order starting at +0; unrouted slots (-1) are
 * skipped.  out_sorted rows are bf16 [*, d]. */
void or_combine(const uint16_t *out_sorted, const int32_t *slot_to_sorted, const float *gates,
                int64_t T, int k, int d, uint16_t *y)
{
#pragma omp parallel for schedule(static)
    for (int64_t t = 0; t < T; t++)
        for (int c = 0; c < d; c++) {
            float acc = 0.0f;
            for (int j = 0; j < k; j++) {
                int32_t r = slot_to_sorted[t * k + j];
                if (r < 0)
                    continue;
                acc = fmaf(gates[t * k + j], or_bf16_to_f32(out_sorted[(int64_t)r * d + c]), acc);
            }
            y[t * d + c] = or_f32_to_bf16(acc);
        }
}

/* Number of OpenMP threads the parallel loops above use (1 without OpenMP). */
/* ------------------------------------------------------------------ */
/* backward of the expert path under replay (the trainer replays routing */
/* to train; "Router replay", "FP8 training")                           */
/* ------------------------------------------------------------------ */

/* Combine backward.  y[t] = sum_j g[t,j] * out[r(t,j)], so for a routed slot
 * the expert output's gradient is d_out[r] = g[t,j] * dy[t] (one binary32
 * product per element) and the gate's gradient is d_g[t,j] = <dy[t], out[r]>
 * (computed in double, rounded once); an unrouted slot gets d_g = 0.  d_out
 * is then quantised 1 x 128 along d by the recipe's rule (fp32 scale
 * amax/448, IEEE division) for the dgrad GEMM.  d_out_f (nullable) [A, d]
 * receives the fp32 values before quantisation. */
void or_combine_backward(const uint16_t *dy, const float *gates, const uint16_t *out_sorted,
                         const int32_t *slot_to_sorted, int64_t T, int k, int d, int64_t A,
                         float *d_out_f, uint8_t *d_out_q, float *d_out_s, float *d_gates)
{
    int64_t nb = d / 128;
#pragma omp parallel for schedule(static)
    for (int64_t t = 0; t < T; t++) {
        for (int j = 0; j < k; j++) {
            int32_t r = slot_to_sorted[t * k + j];
            if (r < 0 || r >= A) {
                d_gates[t * k + j] = 0.0f;
                continue;
            }
            float g = gates[t * k + j];
            double dot = 0.0;
            for (int c = 0; c < d; c++)
                dot += (double)or_bf16_to_f32(dy[t * d + c]) * (double)or_bf16_to_f32(out_sorted[(int64_t)r * d + c]);
            d_gates[t * k + j] = (float)dot;
            for (int64_t b = 0; b < nb; b++) {
                float v[128], amax = 0.0f;
                for (int i = 0; i < 128; i++) {
                    v[i] = g * or_bf16_to_f32(dy[t * d + b * 128 + i]);
                    if (fabsf(v[i]) > amax)
                        amax = fabsf(v[i]);
                }
                float sc = block_scale(amax);
                d_out_s[(int64_t)r * nb + b] = sc;
                for (int i = 0; i < 128; i++) {
                    d_out_q[(int64_t)r * d + b * 128 + i] = or_e4m3_encode(v[i] / sc);
                    if (d_out_f)
                        d_out_f[(int64_t)r * d + b * 128 + i] = v[i];
                }
            }
        }
    }
}

/* Transposed copy of block-quantised weights: q [E, R, C] codes with scales
 * [E, R/128, C/128] -> qt [E, C, R], st [E, C/128, R/128].  Block
 * quantisation commutes with transposition, so this is the quantisation of
 * the transposed weights (the operand layout of the dgrad GEMMs). */
void or_weight_transpose(const uint8_t *q, const float *s, int64_t E, int64_t R, int64_t C, uint8_t *qt, float *st)
{
    for (int64_t e = 0; e < E; e++) {
        for (int64_t r = 0; r < R; r++)
            for (int64_t c = 0; c < C; c++)
                qt[e * R * C + c * R + r] = q[e * R * C + r * C + c];
        int64_t br = R / 128, bc = C / 128;
        for (int64_t i = 0; i < br; i++)
            for (int64_t j = 0; j < bc; j++)
                st[e * br * bc + j * br + i] = s[e * br * bc + i * bc + j];
    }
}

/* The forward's GEMM1 pre-activations h = [gate | up] [n, 2F] (fp32, the
 * promotion of fp8_row_gemm), saved by the forward for the backward. */
void or_expert_ffn_preact(const uint8_t *xq, const float *xs, int64_t n, const int32_t *row_expert, int d, int F,
                          const uint8_t *w13_q, const float *w13_s, float *h)
{
    double dec[256];
    for (int c = 0; c < 256; c++)
        dec[c] = or_e4m3_decode((uint8_t)c);
    int64_t nkd = d / 128;
#pragma omp parallel for schedule(static)
    for (int64_t r = 0; r < n; r++) {
        int64_t e = row_expert[r];
        fp8_row_gemm(xq + r * d, xs + r * nkd, w13_q + e * 2 * F * (int64_t)d, w13_s + e * (2 * F / 128) * nkd,
                     2 * F, d, dec, h + r * 2 * F);
    }
}

/* Grouped block-scaled GEMM with bf16 output: out[r, :] = bf16(fp8_row_gemm(
 * a[r], sa[r], b[row_expert[r]])) with b [E, N, K] codes, sb [E, N/128, K/128].
 * The forward's GEMM2 is (K, N) = (F, d) with W2; the dgrad GEMMs are
 * (d, F) with W2 transposed and (2F, d) with W13 transposed. */
void or_grouped_gemm(const uint8_t *a, const float *sa, int64_t n, const int32_t *row_expert, int64_t K, int64_t N,
                     const uint8_t *b, const float *sb, uint16_t *out)
{
    double dec[256];
    for (int c = 0; c < 256; c++)
        dec[c] = or_e4m3_decode((uint8_t)c);
#pragma omp parallel for schedule(static)
    for (int64_t r = 0; r < n; r++) {
        int64_t e = row_expert[r];
        float *o = malloc(sizeof(float) * (size_t)N);
        fp8_row_gemm(a + r * K, sa + r * (K / 128), b + e * N * K, sb + e * (N / 128) * (K / 128), N, K, dec, o);
        for (int64_t c = 0; c < N; c++)
            out[r * N + c] = or_f32_to_bf16(o[c]);
        free(o);
    }
}

/* SwiGLU backward: act = silu(g) * u with silu(g) = g * sigma(g), so
 *   d_g = d_act * u * sigma(g) * (1 + g * (1 - sigma(g))),   d_u = d_act * silu(g)
 * in double from the bf16 d_act and the saved fp32 h = [g | u], rounded to
 * fp32 (dh_f, nullable), then quantised 1 x 128 along 2F by the recipe's
 * rule: dh_q [n, 2F], dh_s [n, 2F/128]. */
void or_swiglu_backward(const uint16_t *d_act, const float *h, int64_t n, int F, float *dh_f, uint8_t *dh_q,
                        float *dh_s)
{
    int64_t nb = 2 * (int64_t)F / 128;
#pragma omp parallel for schedule(static)
    for (int64_t r = 0; r < n; r++) {
        float *dh = malloc(sizeof(float) * 2 * (size_t)F);
        for (int64_t c = 0; c < F; c++) {
            double da = or_bf16_to_f32(d_act[r * F + c]);
            double g = h[r * 2 * F + c], u = h[r * 2 * F + F + c];
            double sg = 1.0 / (1.0 + exp(-g));
            dh[c] = (float)(da * u * sg * (1.0 + g * (1.0 - sg)));
            dh[F + c] = (float)(da * g * sg);
        }
        for (int64_t b = 0; b < nb; b++) {
            float amax = 0.0f;
            for (int i = 0; i < 128; i++)
                if (fabsf(dh[b * 128 + i]) > amax)
                    amax = fabsf(dh[b * 128 + i]);
            float sc = block_scale(amax);
            dh_s[r * nb + b] = sc;
            for (int i = 0; i < 128; i++)
                dh_q[r * 2 * F + b * 128 + i] = or_e4m3_encode(dh[b * 128 + i] / sc);
        }
        if (dh_f)
            memcpy(dh_f + r * 2 * F, dh, sizeof(float) * 2 * (size_t)F);
        free(dh);
    }
}

/* Padded segment offsets of the weight-gradient layouts: expert e's rows
 * [offsets[e], offsets[e+1]) start at pad[e] = sum_{e'<e} roundup128(rows_e')
 * so that every 128-row block holds rows of one expert; pad[E] is the total. */
void or_pad_offsets(const int32_t *offsets, int E, int32_t *pad)
{
    int64_t acc = 0;
    for (int e = 0; e < E; e++) {
        pad[e] = (int32_t)acc;
        int64_t rows = offsets[e + 1] - offsets[e];
        acc += (rows + 127) / 128 * 128;
    }
    pad[E] = (int32_t)acc;
}

/* 128 x 1 quantisation for the weight-gradient GEMMs (the contraction runs
 * over tokens): src [A, C] fp32 rows in expert order; for every expert's
 * 128-row block and every channel c, amax over the block's real rows, scale
 * amax / 448 (1 if 0), codes e4m3(v / s); written transposed, channel-major:
 * q [C, pad[E]] (zero codes in the padding rows), s [C, pad[E] / 128]. */
void or_quant_128x1(const float *src, const int32_t *offsets, const int32_t *pad, int E, int64_t C,
                    uint8_t *q, float *s)
{
    int64_t P = pad[E], nbk = P / 128;
    memset(q, 0, (size_t)(C * P));
#pragma omp parallel for schedule(static)
    for (int64_t c = 0; c < C; c++) {
        for (int e = 0; e < E; e++) {
            int64_t r0 = offsets[e], rows = offsets[e + 1] - offsets[e];
            for (int64_t b = 0; b * 128 < rows; b++) {
                int64_t n = rows - b * 128 < 128 ? rows - b * 128 : 128;
                float amax = 0.0f;
                for (int64_t i = 0; i < n; i++) {
                    float v = fabsf(src[(r0 + b * 128 + i) * C + c]);
                    if (v > amax)
                        amax = v;
                }
                float sc = block_scale(amax);
                int64_t kb = pad[e] / 128 + b;
                s[c * nbk + kb] = sc;
                for (int64_t i = 0; i < n; i++)
                    q[c * P + pad[e] + b * 128 + i] = or_e4m3_encode(src[(r0 + b * 128 + i) * C + c] / sc);
            }
        }
    }
}

/* Weight gradient of one grouped GEMM: out[e] [M, N] fp32 =
 * sum over expert e's 128-row blocks kb of (sa[m, kb] * sb[n, kb]) * P_kb(m, n),
 * P_kb the exact 128-term dot of the two channel rows (rounded to binary32),
 * a binary32 fma chain in ascending kb (the forward's promotion, with the
 * contraction over tokens).  a [M, P] codes with sa [M, P/128], b [N, P] with
 * sb [N, P/128] (the 128 x 1 layouts above). */
void or_wgrad(const uint8_t *a, const float *sa, const uint8_t *b, const float *sb, const int32_t *pad, int E,
              int64_t M, int64_t N, float *out)
{
    double dec[256];
    for (int c = 0; c < 256; c++)
        dec[c] = or_e4m3_decode((uint8_t)c);
    int64_t P = pad[E], nbk = P / 128;
#pragma omp parallel for schedule(dynamic, 1)
    for (int64_t em = 0; em < (int64_t)E * M; em++) {
        int64_t e = em / M, m = em % M;
        for (int64_t n = 0; n < N; n++) {
            float acc = 0.0f;
            for (int64_t kb = pad[e] / 128; kb < pad[e + 1] / 128; kb++) {
                float pk = (float)e4m3_block_dot(a + m * P + kb * 128, b + n * P + kb * 128, dec);
                acc = fmaf(sa[m * nbk + kb] * sb[n * nbk + kb], pk, acc);
            }
            out[(e * M + m) * N + n] = acc;
        }
    }
}

/* Dispatch backward: the input rows' gradient is the sum of their sorted
 * copies' gradients, dx[t] = bf16( sum_j dx_sorted[r(t,j)] ), a binary32
 * chain over j in slot order from +0 (unrouted slots skipped). */
void or_dispatch_backward(const uint16_t *dx_sorted, const int32_t *slot_to_sorted, int64_t T, int k, int d,
                          uint16_t *dx)
{
#pragma omp parallel for schedule(static)
    for (int64_t t = 0; t < T; t++)
        for (int c = 0; c < d; c++) {
            float acc = 0.0f;
            for (int j = 0; j < k; j++) {
                int32_t r = slot_to_sorted[t * k + j];
                if (r < 0)
                    continue;
                acc = acc + or_bf16_to_f32(dx_sorted[(int64_t)r * d + c]);
            }
            dx[t * d + c] = or_f32_to_bf16(acc);
        }
}

#ifdef _OPENMP
#include <omp.h>
int or_num_threads(void) { return omp_get_max_threads(); }
void or_set_num_threads(int n) { omp_set_num_threads(n); }
#else
int or_num_threads(void) { return 1; }
void or_set_num_threads(int n) { (void)n; }
#endif
