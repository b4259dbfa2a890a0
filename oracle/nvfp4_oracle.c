/*
 * nvfp4_oracle.c -- TEST INFRASTRUCTURE ONLY.
 *
 * A plain, slow, single-threaded CPU restatement of what the NVFP4 W4A4 + RAC
 * hot path computes.  It exists to check the CUDA library; only the test
 * suite, the smoke check and the benchmark's CPU-baseline leg load it.  It
 * shares no code, header, table or constant generator with the CUDA library,
 * and the library never loads it.
 *
 * Source.  "QUADS" below is the paper "QUADS: Stabilizing NVFP4 Reinforcement
 * Learning for MoE via QUantization-error Alignment across Dual Sides"
 * (arXiv 2607.15810, HTML mirror).  Every function names the section or
 * equation it follows.  Where the paper is silent the function states the
 * reading it takes (the readings are listed together in the design notes).
 *
 * Arithmetic.  The paper fixes the formats (E2M1 elements, E4M3 block scales,
 * an FP32 per-tensor scale), so every decision that produces a code or a scale
 * is taken in IEEE binary32, one rounding per operation (the file is compiled
 * with -ffp-contract=off and without fast-math).  Sums that only produce a
 * real-valued result (GEMMs, norms, softmax) are taken in binary64.
 *
 * Parity status of each function (what pins it, see tests/test_oracle_*.py):
 *   orc_e2m1_value / orc_e2m1_encode   pinned: page value set, brute force
 *   orc_e4m3_value / orc_e4m3_encode   pinned: torch float8_e4m3fn, brute force
 *   orc_bf16_round                      pinned: torch bfloat16 cast
 *   orc_quantize / orc_dequantize       pinned: grid, amax->6, idempotence,
 *                                       symmetry, zero tensor, scale brute force
 *   orc_scale_layout                    pinned on the GPU only (GEMM parity);
 *                                       on the CPU: bijection + zero padding
 *   orc_rac_gemm / orc_bf16_gemm        pinned: numpy matmul, exact-integer case,
 *                                       k=0 and k=K special cases
 *   orc_channel_scores / orc_select     pinned: brute force over subsets
 *   orc_route_topk                      pinned: numpy stable argsort + scipy softmax
 *   orc_swiglu                          pinned: closed-form values of silu
 *   orc_combine                         pinned: numpy einsum
 */
#include <math.h>
#include <stdint.h>
#include <stdlib.h>
#include <string.h>

/* ------------------------------------------------------------------------ */
/* Formats.  QUADS §2.2 Eq. 4 and "FP4." / "FP8.".                           */
/* ------------------------------------------------------------------------ */

/* E2M1 code s|e1 e0|m -> value.  QUADS §2.2 "FP4.": the NVFP4 core yields
 * {0, 0.5, 1, 1.5, 2, 3, 4, 6} per sign.  Eq. 4 with b=4, e=2, one mantissa
 * bit; exponent bias 1, exponent field 0 is subnormal (m * 0.5). */
double orc_e2m1_value(int code)
{
    int s = (code >> 3) & 1, e = (code >> 1) & 3, m = code & 1;
    double mag = (e == 0) ? 0.5 * m : ldexp(1.0 + 0.5 * m, e - 1);
    return s ? -mag : mag;
}

/* E4M3 code s|eeee|mmm -> value.  QUADS §2.2 "FP8.": b=8, e=4, three mantissa
 * bits, largest magnitude 448.  Bias 7; exponent field 0 is subnormal
 * (m * 2^-9); exponent 15 with mantissa 7 is NaN (the only non-finite code). */
double orc_e4m3_value(int code)
{
    int s = (code >> 7) & 1, e = (code >> 3) & 15, m = code & 7;
    double mag;
    if (e == 15 && m == 7) return NAN;
    mag = (e == 0) ? ldexp((double)m, -9) : ldexp(1.0 + m / 8.0, e - 7);
    return s ? -mag : mag;
}

/* Round a non-negative finite value to an integer multiple of `quantum`,
 * nearest, ties to the even multiple.  rint() in the default rounding mode is
 * round-half-even; v/quantum is exact because quantum is a power of two. */
static double round_to_quantum(double v, double quantum)
{
    return rint(v / quantum) * quantum;
}

/* value -> E2M1 code, round to nearest, ties to even, saturating at 6, the
 * sign bit copied from v (so -0 and small negatives give code 0x8).
 * Reading (the paper does not state the rounding): round-to-nearest-even with
 * saturation, the IEEE default applied to the E2M1 grid. */
int orc_e2m1_encode(float v)
{
    double a = fabs((double)v), q, g;
    int sign = signbit(v) ? 8 : 0, code;
    /* spacing of the E2M1 grid: 0.5 below 2, 1 in [2,4), 2 from 4 on */
    q = (a < 2.0) ? 0.5 : (a < 4.0) ? 1.0 : 2.0;
    g = round_to_quantum(a, q);
    if (g > 6.0) g = 6.0;
    /* grid value -> code: index into {0,0.5,1,1.5,2,3,4,6} */
    if (g < 2.0) code = (int)(g * 2.0);          /* 0,0.5,1,1.5 -> 0..3 */
    else if (g < 4.0) code = 4 + (int)(g - 2.0); /* 2,3 -> 4,5 */
    else code = (g == 4.0) ? 6 : 7;              /* 4,6 -> 6,7 */
    return sign | code;
}

/* non-negative value -> E4M3 code, round to nearest, ties to even, values
 * above 448 saturate to 448 (0x7E).  Used for block scales, which are never
 * negative.  Reading: the paper names E4M3 but not its rounding; RNE with
 * saturation keeps every scale finite. */
int orc_e4m3_encode(float v)
{
    double a = (double)v, q, g;
    int ex;
    if (!(a > 0.0)) return 0; /* zero (and, outside the contract, NaN) */
    if (a < ldexp(1.0, -6)) {
        q = ldexp(1.0, -9); /* subnormal spacing */
    } else {
        (void)frexp(a, &ex); /* a = f * 2^ex, f in [0.5,1) */
        q = ldexp(1.0, ex - 1 - 3);
    }
    g = round_to_quantum(a, q);
    if (g > 448.0) g = 448.0;
    if (g < ldexp(1.0, -6)) return (int)(g / ldexp(1.0, -9)); /* 0..8 (8 = 2^-6) */
    (void)frexp(g, &ex);
    {
        int e = ex - 1 + 7;                                   /* biased exponent */
        int m = (int)((g / ldexp(1.0, ex - 1) - 1.0) * 8.0); /* exact */
        return (e << 3) | m;
    }
}

/* binary32 -> bfloat16 bits, round to nearest even (textbook bit form). */
uint16_t orc_bf16_round(float f)
{
    uint32_t u;
    memcpy(&u, &f, 4);
    if ((u & 0x7fffffffu) > 0x7f800000u) return (uint16_t)((u >> 16) | 0x40); /* NaN */
    u += 0x7fffu + ((u >> 16) & 1u);
    return (uint16_t)(u >> 16);
}

float orc_bf16_value(uint16_t b)
{
    uint32_t u = (uint32_t)b << 16;
    float f;
    memcpy(&f, &u, 4);
    return f;
}

/* ------------------------------------------------------------------------ */
/* NVFP4 quantizer Q_A / Q_W.  QUADS §2.2 "FP4.", §3.1 Eq. 7 and Eq. 9.     */
/* ------------------------------------------------------------------------ */

/* Per-tensor amax = max |x|; exact. */
float orc_amax(const uint16_t *x, int64_t M, int64_t K, int64_t ldx)
{
    float m = 0.0f;
    for (int64_t i = 0; i < M; i++)
        for (int64_t j = 0; j < K; j++) {
            float a = fabsf(orc_bf16_value(x[i * ldx + j]));
            if (a > m) m = a;
        }
    return m;
}

/* The optional FP32 per-tensor scale of §2.2.  Reading: the smallest power of
 * two not below fl(amax / (6*448)), so every block scale target
 * amax16 / (6*gs) is at most 448 (the E4M3 maximum) and the largest block's
 * lies in (224, 448]; an all-zero tensor gets gs = 1.  A power of two keeps
 * (code*sb)*gs exact and lets the RAC residual be carried exactly in units
 * of gs (see orc_quantize). */
float orc_tensor_scale(float amax)
{
    float q;
    int e;
    double f;
    if (amax == 0.0f) return 1.0f;
    q = amax / 2688.0f;
    f = frexp((double)q, &e); /* q = f * 2^e, f in [0.5, 1) */
    if (f == 0.5) return q;   /* already a power of two */
    return (float)ldexp(1.0, e);
}

/* The E4M3 block scale of one 16-element block.  Reading: the block scale is
 * the block amax divided by (6 * gs), rounded to E4M3 (RNE, saturating). */
static int block_scale_code(float amax_b, float gs)
{
    float p = gs * 6.0f;
    float s = amax_b / p;
    return orc_e4m3_encode(s);
}

/* One element of a block: the value put on the E2M1 grid.  Reading: the
 * element is scaled by the correctly rounded reciprocal of the block's
 * effective scale den = sb * gs (one binary32 multiply), then rounded to E2M1.
 * A zero block scale encodes every element as a zero with the element's sign. */
static int element_code(float x, float den)
{
    float inv, q;
    if (den == 0.0f) return signbit(x) ? 8 : 0;
    inv = 1.0f / den;
    q = x * inv;
    return orc_e2m1_encode(q);
}

/* Dequantized value of one element: (code value * sb) * gs.  The first
 * product is exact (at most 6 significant bits), the second rounds once. */
static float element_dequant(int code, float sbf, float gs)
{
    float cs = (float)orc_e2m1_value(code) * sbf;
    return cs * gs;
}

/*
 * NVFP4 quantize of a BF16 matrix x [M, K] (row stride ldx, K % 16 == 0).
 * Blocks are 16 consecutive elements along K (QUADS §2.2: "sixteen
 * consecutive elements share an E4M3 block scale").
 *   codes  [M, K/2]  two E2M1 codes per byte, element 2i in the low nibble
 *   scales [M, K/16] E4M3 block-scale codes, row-major (canonical layout)
 *   resid  [M, k]    for the channels S[0..k) (strictly increasing): the
 *                    residual r = bf16(x - dequant(q(x))) -- the negative of
 *                    the activation quantization error Delta X_q of Eq. 9 /
 *                    Eq. 20, which Residual Activation Compensation (Eq. 21)
 *                    adds back -- stored in units of gs: bf16(r * (1/gs)).
 *                    With gs a power of two this is r / gs exactly (unless it
 *                    falls below the BF16 normal range).
 * gs is the per-tensor scale (orc_tensor_scale of the tensor's amax).
 */
void orc_quantize(const uint16_t *x, int64_t M, int64_t K, int64_t ldx, float gs,
                  uint8_t *codes, uint8_t *scales, const int32_t *S, int32_t k,
                  uint16_t *resid)
{
    int64_t nb = K / 16;
    float *xq_row = (float *)malloc(sizeof(float) * (size_t)(K > 0 ? K : 1));
    for (int64_t i = 0; i < M; i++) {
        for (int64_t b = 0; b < nb; b++) {
            const uint16_t *xb = x + i * ldx + b * 16;
            float amax_b = 0.0f, sbf, den;
            int sb;
            for (int t = 0; t < 16; t++) {
                float a = fabsf(orc_bf16_value(xb[t]));
                if (a > amax_b) amax_b = a;
            }
            sb = block_scale_code(amax_b, gs);
            scales[i * nb + b] = (uint8_t)sb;
            sbf = (float)orc_e4m3_value(sb);
            den = sbf * gs;
            for (int t = 0; t < 16; t++) {
                float xv = orc_bf16_value(xb[t]);
                int c = element_code(xv, den);
                int64_t j = b * 16 + t;
                uint8_t *byte = codes + i * (K / 2) + j / 2;
                if ((j & 1) == 0) *byte = (uint8_t)((*byte & 0xF0) | c);
                else *byte = (uint8_t)((*byte & 0x0F) | (c << 4));
                xq_row[j] = element_dequant(c, sbf, gs);
            }
        }
        for (int32_t s = 0; s < k; s++) {
            int64_t j = S[s];
            float xv = orc_bf16_value(x[i * ldx + j]);
            float d = xv - xq_row[j];
            float r = orc_bf16_value(orc_bf16_round(d));
            resid[i * (int64_t)k + s] = orc_bf16_round(r * (1.0f / gs));
        }
    }
    free(xq_row);
}

/* Dequantize to the exact real values code * sb * gs (binary64 holds them
 * exactly: at most 6 + 24 significant bits).  This is what the block-scaled
 * tensor-core product multiplies. */
void orc_dequantize_exact(const uint8_t *codes, const uint8_t *scales, int64_t M, int64_t K,
                          float gs, double *out)
{
    int64_t nb = K / 16;
    for (int64_t i = 0; i < M; i++)
        for (int64_t j = 0; j < K; j++) {
            uint8_t byte = codes[i * (K / 2) + j / 2];
            int c = (j & 1) ? (byte >> 4) : (byte & 15);
            double sbf = orc_e4m3_value(scales[i * nb + j / 16]);
            out[i * K + j] = orc_e2m1_value(c) * sbf * (double)gs;
        }
}

/* Dequantize rounded to binary32, the value the residual is taken against. */
void orc_dequantize_f32(const uint8_t *codes, const uint8_t *scales, int64_t M, int64_t K,
                        float gs, float *out)
{
    int64_t nb = K / 16;
    for (int64_t i = 0; i < M; i++)
        for (int64_t j = 0; j < K; j++) {
            uint8_t byte = codes[i * (K / 2) + j / 2];
            int c = (j & 1) ? (byte >> 4) : (byte & 15);
            float sbf = (float)orc_e4m3_value(scales[i * nb + j / 16]);
            out[i * K + j] = element_dequant(c, sbf, gs);
        }
}

/* Scale layout shared by the quantizer and the block-scaled GEMM, for
 * activations and weights alike (a layout choice of this library: the paper
 * only asks that the rollout quantizer's layout match its GEMM's, §3.2).  The
 * canonical [M, K/16] block scales are grouped by tiles of 128 rows x 16
 * blocks (one 256-element GEMM K-slice), tile (m/128, kb/16) the
 * ((m/128) * ceil(K/256) + kb/16)-th, 2048 bytes each: four 512-byte groups,
 * one per 4 consecutive blocks (one MMA's 64 elements of K); in group j/4
 * (j = kb%16) row r = m%128 sits on line r%32 (16 bytes), block j at byte
 * 4*(r/32) + j%4.  Rows beyond M and blocks beyond K/16 are zero. */
void orc_scale_layout(const uint8_t *scales, int64_t M, int64_t K, uint8_t *out)
{
    int64_t nb = K / 16, mt = (M + 127) / 128, kt = (nb + 15) / 16;
    memset(out, 0, (size_t)(mt * kt * 2048));
    for (int64_t m = 0; m < M; m++)
        for (int64_t kb = 0; kb < nb; kb++) {
            int64_t r = m % 128, j = kb % 16;
            int64_t off = ((m / 128) * kt + kb / 16) * 2048 + (j / 4) * 512 + (r % 32) * 16 + (r / 32) * 4 + j % 4;
            out[off] = scales[m * nb + kb];
        }
}

/* Trainer-side weight fake-quantization QDQ_W of QUADS §3.2 Eq. 12:
 * W_hat = bf16(dequant(quantize(W))) with W's own per-tensor scale, the same
 * block layout and rounding as the rollout quantizer (the paper requires the
 * scale layout and rounding to match the rollout kernel). */
void orc_fake_quant(const uint16_t *w, int64_t M, int64_t K, uint16_t *w_hat, float *gs_out)
{
    float gs = orc_tensor_scale(orc_amax(w, M, K, K));
    uint8_t *codes = (uint8_t *)calloc((size_t)(M * K / 2 + 1), 1);
    uint8_t *scales = (uint8_t *)calloc((size_t)(M * K / 16 + 1), 1);
    float *deq = (float *)malloc(sizeof(float) * (size_t)(M * K + 1));
    orc_quantize(w, M, K, K, gs, codes, scales, NULL, 0, NULL);
    orc_dequantize_f32(codes, scales, M, K, gs, deq);
    for (int64_t i = 0; i < M * K; i++) w_hat[i] = orc_bf16_round(deq[i]);
    *gs_out = gs;
    free(codes);
    free(scales);
    free(deq);
}

/* ------------------------------------------------------------------------ */
/* GEMMs.  QUADS §3.3 Eq. 21 (RAC) and §3.2 Eq. 12 (asymmetric QAT).          */
/* ------------------------------------------------------------------------ */

/*
 * W4A4 + RAC product for one expert, accumulated in binary64:
 *   y[i,n] = sum_K xq[i,K] * wq[n,K]  +  sum_{s<k} (gs_a * r[i,s]) * wq[n, S[s]]
 * xq, wq: exact dequantized operands [M,K], [N,K] (orc_dequantize_exact);
 * r: the BF16 residual [M,k] on channels S in units of the activation's
 * per-tensor scale gs_a (orc_quantize's resid).  The first sum is the native
 * W4A4 GEMM; the second is the rank-k correction on the selected channels
 * (Eq. 21, with the residual kept in BF16 and the weight dequantized NVFP4).
 */
void orc_rac_gemm(const double *xq, const uint16_t *r, const int32_t *S, int32_t k, double gs_a,
                  const double *wq, int64_t M, int64_t N, int64_t K, double *y)
{
    for (int64_t i = 0; i < M; i++)
        for (int64_t n = 0; n < N; n++) {
            double acc = 0.0;
            for (int64_t j = 0; j < K; j++) acc += xq[i * K + j] * wq[n * K + j];
            for (int32_t s = 0; s < k; s++)
                acc += gs_a * (double)orc_bf16_value(r[i * (int64_t)k + s]) * wq[n * K + S[s]];
            y[i * N + n] = acc;
        }
}

/* The trainer's forward of Eq. 12: y = X_bf16 * W_hat^T, binary64 sums. */
void orc_bf16_gemm(const uint16_t *x, const uint16_t *w, int64_t M, int64_t N, int64_t K, double *y)
{
    for (int64_t i = 0; i < M; i++)
        for (int64_t n = 0; n < N; n++) {
            double acc = 0.0;
            for (int64_t j = 0; j < K; j++)
                acc += (double)orc_bf16_value(x[i * K + j]) * (double)orc_bf16_value(w[n * K + j]);
            y[i * N + n] = acc;
        }
}

/* ------------------------------------------------------------------------ */
/* Channel selection.  QUADS §3.3 Eq. 23-24.                                   */
/* ------------------------------------------------------------------------ */

/* Squared residual score per channel, Eq. 23 before the square root:
 * ssq[j] = sum_i (Q_A(X)[i,j] - X[i,j])^2 over the batch, binary64, rows in
 * order, using the exact dequantized values. */
void orc_channel_scores(const uint16_t *x, int64_t M, int64_t K, float gs, double *ssq)
{
    int64_t nb = K / 16;
    uint8_t *codes = (uint8_t *)calloc((size_t)(M * K / 2 + 1), 1);
    uint8_t *scales = (uint8_t *)calloc((size_t)(M * nb + 1), 1);
    orc_quantize(x, M, K, K, gs, codes, scales, NULL, 0, NULL);
    for (int64_t j = 0; j < K; j++) ssq[j] = 0.0;
    for (int64_t i = 0; i < M; i++)
        for (int64_t j = 0; j < K; j++) {
            uint8_t byte = codes[i * (K / 2) + j / 2];
            int c = (j & 1) ? (byte >> 4) : (byte & 15);
            double xq = orc_e2m1_value(c) * orc_e4m3_value(scales[i * nb + j / 16]) * (double)gs;
            double d = xq - (double)orc_bf16_value(x[i * K + j]);
            ssq[j] += d * d;
        }
    free(codes);
    free(scales);
}

/* Eq. 24 with a channel count k: the k channels of largest score, ties to
 * the lower channel index, written in increasing channel order.  Selection
 * by plain repeated arg-max. */
void orc_select_channels(const double *ssq, int64_t K, int32_t k, int32_t *S)
{
    char *taken = (char *)calloc((size_t)K + 1, 1);
    int32_t got = 0;
    for (int32_t r = 0; r < k; r++) {
        int64_t best = -1;
        for (int64_t j = 0; j < K; j++)
            if (!taken[j] && (best < 0 || ssq[j] > ssq[best])) best = j;
        if (best < 0) break; /* k > K: outside the contract */
        taken[best] = 1;
    }
    for (int64_t j = 0; j < K; j++)
        if (taken[j]) S[got++] = (int32_t)j;
    free(taken);
}

/* ------------------------------------------------------------------------ */
/* MoE glue (not on the paper's pages; the plainest reading of a top-k        */
/* softmax router, SwiGLU experts and a weighted combine).                    */
/* ------------------------------------------------------------------------ */

/* Router: softmax over E in binary64; top-k by logit (ties to the lower
 * expert index), weights = the softmax probabilities of the chosen experts
 * (no renormalization). */
void orc_route_topk(const float *logits, int32_t T, int32_t E, int32_t topk, int32_t *ids,
                    double *weights)
{
    char *taken = (char *)malloc((size_t)E + 1);
    for (int32_t t = 0; t < T; t++) {
        const float *l = logits + (int64_t)t * E;
        double mx = -INFINITY, den = 0.0;
        for (int32_t e = 0; e < E; e++)
            if (l[e] > mx) mx = l[e];
        for (int32_t e = 0; e < E; e++) den += exp((double)l[e] - mx);
        memset(taken, 0, (size_t)E);
        for (int32_t s = 0; s < topk; s++) {
            int32_t best = -1;
            for (int32_t e = 0; e < E; e++)
                if (!taken[e] && (best < 0 || l[e] > l[best])) best = e;
            taken[best] = 1;
            ids[(int64_t)t * topk + s] = best;
            weights[(int64_t)t * topk + s] = exp((double)l[best] - mx) / den;
        }
    }
    free(taken);
}

/* SwiGLU on the gate_up projection output y [M, 2I]: gate = columns [0, I),
 * up = [I, 2I); h = silu(gate) * up, silu(g) = g / (1 + exp(-g)); binary64. */
void orc_swiglu(const double *y, int64_t M, int64_t I, double *h)
{
    for (int64_t i = 0; i < M; i++)
        for (int64_t j = 0; j < I; j++) {
            double g = y[i * 2 * I + j], u = y[i * 2 * I + I + j];
            h[i * I + j] = g / (1.0 + exp(-g)) * u;
        }
}

/* Combine: out[t] = sum over slots of weight[t,s] * y[row[t,s]], slot order. */
void orc_combine(const double *y, int64_t ldy, const int32_t *row, const double *weights,
                 int32_t T, int32_t topk, int64_t H, double *out)
{
    for (int32_t t = 0; t < T; t++)
        for (int64_t c = 0; c < H; c++) {
            double acc = 0.0;
            for (int32_t s = 0; s < topk; s++) {
                int64_t rr = row[(int64_t)t * topk + s];
                acc += weights[(int64_t)t * topk + s] * y[rr * ldy + c];
            }
            out[(int64_t)t * H + c] = acc;
        }
}

/* ------------------------------------------------------------------------ */
/* Array helpers for the tests (element-wise loops over the functions above). */
/* ------------------------------------------------------------------------ */

void orc_e2m1_encode_array(const float *v, int64_t n, uint8_t *out)
{
    for (int64_t i = 0; i < n; i++) out[i] = (uint8_t)orc_e2m1_encode(v[i]);
}

void orc_e4m3_encode_array(const float *v, int64_t n, uint8_t *out)
{
    for (int64_t i = 0; i < n; i++) out[i] = (uint8_t)orc_e4m3_encode(v[i]);
}

void orc_bf16_round_array(const float *v, int64_t n, uint16_t *out)
{
    for (int64_t i = 0; i < n; i++) out[i] = orc_bf16_round(v[i]);
}
