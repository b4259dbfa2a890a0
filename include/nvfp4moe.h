/*
 * nvfp4moe.h -- C ABI of the NVFP4 W4A4 + RAC MoE hot path for sm_103a (GB300).
 *
 * "QUADS" is the paper "QUADS: Stabilizing NVFP4 Reinforcement Learning for
 * MoE via QUantization-error Alignment across Dual Sides".  Each entry point
 * cites the passage that defines what it computes.
 *
 * Conventions (all entry points):
 *  - Every function returns an nvfp4_status.  Argument errors are detected on
 *    the host before anything is launched; nothing is launched when a call
 *    returns an error.  Errors found on the device (a non-finite amax, a
 *    bounded wait that ran out) are written to the optional `dev_status`
 *    word (device int32, first error wins, 0 = OK) which the caller reads
 *    whenever it likes.  No exception crosses the ABI.
 *  - The caller owns all memory.  Pointers marked "device" are CUDA device
 *    pointers; the library allocates nothing and frees nothing.
 *  - Every call is asynchronous and stream-ordered on `stream` (a
 *    cudaStream_t passed as void*; NULL = legacy default stream) and never
 *    synchronizes.  Outputs are valid once the stream reaches them.
 *  - BF16 is passed as `void*` holding IEEE bfloat16 bit patterns.
 *  - Device pointers must be 16-byte aligned (NVFP4_ERR_ALIGNMENT otherwise).
 *  - A batch of no tokens is valid: the token-sized buffers of nvfp4_amax,
 *    nvfp4_quantize, nvfp4_route_topk, nvfp4_moe_scatter_rows,
 *    nvfp4_moe_combine, nvfp4_moe_combine_backward and
 *    nvfp4_rac_select_channels_online may be NULL when they hold no element.
 *  - There is no CPU path: without an sm_103 device every call returns
 *    NVFP4_ERR_ARCH.
 *
 * NVFP4 tensor format (QUADS §2.2 "FP4."):
 *  - codes  [rows, K/2] uint8: E2M1 codes, two per byte, element 2i in the
 *           low nibble, element 2i+1 in the high nibble.
 *  - scales E4M3 block scales, one per 16 consecutive elements along K, in
 *           tiles of 128 rows x 16 blocks (one GEMM K-slice of 256 elements):
 *           tile (m/128, kb/16) starts at byte ((m/128)*KS + kb/16)*2048, KS =
 *           ceil(K/256).  A tile is four 512-byte groups, one per 4 consecutive
 *           blocks (one MMA's 64 elements of K): block j = kb%16 of row
 *           r = m%128 sits in group j/4, on line r%32 (16 bytes), at byte
 *           4*(r/32) + j%4.  This is the 128-row x 4-block interleave the
 *           block-scaled MMA reads from tensor memory: the GEMM copies a group
 *           as is (one 32x128b.warpx4 tcgen05.cp).  The same layout serves
 *           activations (nvfp4_quantize) and weights (nvfp4_prepare_weights).
 *           Size ceil(rows/128) * KS * 2048 bytes (= rows * K/16 for
 *           rows % 128 == 0 and K % 256 == 0); the bytes of rows past the
 *           tensor's last row and of blocks past K/16 are not written.
 *  - gs     FP32 per-tensor scale: the smallest power of two not below
 *           fl(amax/2688) (amax = max|x| over the tensor; 2688 = 6*448), so
 *           every block-scale target amax16/(6*gs) is at most 448; gs = 1 for
 *           an all-zero tensor.
 *  - value  of element (m, j) = e2m1(code) * e4m3(scale) * gs.
 *
 * Scratch: no entry point allocates.  Where a kernel needs scratch in device
 * memory (an amax, channel scores) the caller passes it with the call
 * (`amax_ws`, `score_ws`, `amax_out` ...), sized as each call states;
 * nvfp4_fake_quant_noalloc is the one variant that needs none from the caller.
 */
#ifndef NVFP4MOE_H
#define NVFP4MOE_H

#include <stdint.h>

#ifdef __cplusplus
extern "C" {
#endif

typedef enum {
    NVFP4_OK = 0,
    NVFP4_ERR_INVALID_ARG = 1, /* a null pointer, a negative size, a bad enum  */
    NVFP4_ERR_UNSUPPORTED = 2, /* a shape outside the kernels' rules           */
    NVFP4_ERR_ALIGNMENT = 3,   /* a pointer or stride not 16-byte aligned      */
    NVFP4_ERR_CUDA = 4,        /* a CUDA runtime call or launch failed         */
    NVFP4_ERR_TIMEOUT = 5,     /* a bounded device wait ran out (dev_status)   */
    NVFP4_ERR_NONFINITE = 6,   /* a tensor amax was Inf/NaN (dev_status)       */
    NVFP4_ERR_ARCH = 7         /* no sm_103 device current                     */
} nvfp4_status;

/* Output element type of the GEMMs. */
enum { NVFP4_OUT_F32 = 0, NVFP4_OUT_BF16 = 1 };
/* Epilogue of the grouped GEMMs: none, SwiGLU of the gate/up product (forward),
 * or the SwiGLU backward of the input-gradient GEMM (nvfp4_bf16_grouped_gemm_dgrad). */
enum { NVFP4_EPI_NONE = 0, NVFP4_EPI_SWIGLU = 1, NVFP4_EPI_SWIGLU_BWD = 2, NVFP4_EPI_SWIGLU_SAVE = 3 };
enum { NVFP4_PIPELINE_AUTO = 0, NVFP4_PIPELINE_SINGLE = 1, NVFP4_PIPELINE_PAIR = 2 };

/* Name of a status code ("NVFP4_OK", ...); never NULL. */
const char *nvfp4_status_str(int status);

/* Library set-up (no counterpart in QUADS).
 * Checks that the current CUDA device is an sm_103 part and loads the driver
 * entry point used to build TMA descriptors.  Called implicitly by every
 * entry point; returns NVFP4_ERR_ARCH on any other device. */
int nvfp4_init(void);

/* Text of the last CUDA error seen by the library in this thread ("" if none). */
const char *nvfp4_last_error(void);

/* ------------------------------------------------------------------------ */
/* Quantization (QUADS §2.2 "FP4."; §3.1 Eq. 9; §3.3 Eq. 20-21)              */
/* ------------------------------------------------------------------------ */

/* The amax behind the per-tensor FP32 scale of QUADS §2.2 "FP4.".
 * Per-tensor amax = max |x| for `ntensors` BF16 matrices of M x K (row
 * stride ldx elements) laid out `tensor_stride` elements apart.
 *   x          device, BF16
 *   amax_out   device float[ntensors]; overwritten (it is cleared first).
 * NaN/Inf inputs propagate to amax_out as a non-finite value.
 * Errors: INVALID_ARG (null, negative sizes, ldx < K), ALIGNMENT (x not 16-byte
 * aligned or ldx % 8 != 0), UNSUPPORTED (K % 8 != 0). */
int nvfp4_amax(const void *x, int64_t M, int64_t K, int64_t ldx, int32_t ntensors,
               int64_t tensor_stride, float *amax_out, void *stream);

/* NVFP4 quantize of a BF16 activation matrix x [M, K] (row stride ldx) with
 * the RAC residual of QUADS §3.3 Eq. 20-21 on a fixed channel set S.
 *   amax        device float: the tensor's amax (from nvfp4_amax, or any
 *               caller value); gs = its power-of-two tensor scale (see top).
 *   gs_out      device float or NULL: receives gs.
 *   S, k        device int32[k], strictly increasing channel indices < K,
 *               0 <= k <= K, k % 8 == 0 (k = 0: no residual; S may be NULL).
 *   dst_row     device int32[M*fanout] or NULL.  NULL: row m is written to
 *               output row m (fanout must be 1).  Otherwise row m is written
 *               to every output row dst_row[m*fanout + f], f < fanout (the MoE
 *               dispatch: each token's codes go to its routed rows).
 *   rows_out    number of output rows (>= M when dst_row is NULL).
 *   codes       device uint8 [rows_out, K/2]
 *   scales      device uint8, the scale layout for rows_out rows (see top)
 *   resid       device BF16 [rows_out, k]: the residual r = bf16(x -
 *               dequant(q(x))) on S -- minus the quantization error Delta X_q
 *               of Eq. 20 -- in units of gs: bf16(r * (1/gs)), which is r/gs
 *               exactly (gs is a power of two) unless it falls below the BF16
 *               normal range.  The GEMM multiplies it by gs again.
 *   row_limit   device int32 or NULL: only source rows m < *row_limit (read
 *               when the kernel runs; clamped to [0, M]) are quantized, later
 *               rows are neither read nor written.  The MoE layer passes
 *               offsets + E for its routed h: rows past the last expert segment
 *               are never read by the grouped GEMM.
 * Per element: block scale sb = e4m3_rn_sat(amax16 / (6*gs)); den = sb*gs;
 * code = e2m1_rn_sat(x * (1/den)) with 1/den correctly rounded (a zero den
 * gives a signed zero code); dequant = (code*sb)*gs in binary32.
 * Output rows not named by dst_row are left untouched (see
 * nvfp4_moe_clear_padding).  dev_status gets NONFINITE if amax is not finite.
 * Errors: INVALID_ARG (null pointers, negative sizes, fanout < 1),
 * ALIGNMENT (pointers; ldx % 8), UNSUPPORTED (K % 32, K > 16384, k % 8,
 * fanout > 32, M or rows_out above 2^31 - 1). */
int nvfp4_quantize(const void *x, int64_t M, int64_t K, int64_t ldx, const float *amax,
                   float *gs_out, const int32_t *S, int32_t k, const int32_t *dst_row,
                   int32_t fanout, int64_t rows_out, uint8_t *codes, uint8_t *scales,
                   void *resid, const int32_t *row_limit, int32_t *dev_status, void *stream);

/* Trainer-side weight fake-quantization QDQ_W of QUADS §3.2 Eq. 12:
 * w_hat = bf16((code*sb)*gs) for `ntensors` BF16 weights of rows x cols,
 * each with its own gs (one per tensor), the same block layout and rounding
 * as nvfp4_quantize, so that the learner sees exactly the weights rollout
 * dequantizes (Eq. 15-16).
 *   w, w_hat    device BF16 [ntensors, rows, cols] (may not alias)
 *   gs_out      device float[ntensors] or NULL
 *   amax_ws     device scratch of 2*ntensors + 1 32-bit words, cleared by the
 *               call on `stream`: the amax of each tensor (as float), then
 *               the work-scheduling counters.  One persistent launch reads
 *               each tensor from HBM once: a tensor's amax items are taken
 *               shortly before its quantize-dequantize items, which re-read
 *               its rows from L2 (and wait, with a 2 s bound, for the amax;
 *               dev_status gets TIMEOUT if it ran out).
 * Errors: INVALID_ARG, ALIGNMENT, UNSUPPORTED (cols % 32, cols > 16384,
 * ntensors > 65535). */
int nvfp4_fake_quant(const void *w, int32_t ntensors, int64_t rows, int64_t cols, void *w_hat,
                     float *gs_out, float *amax_ws, int32_t *dev_status, void *stream);

/* nvfp4_fake_quant that also writes the transpose, for the learner's backward
 * (QUADS §3.2 Eq. 13: dX = W_hat^T dY wants W_hat^T with the reduction axis
 * contiguous): w_hat as nvfp4_fake_quant writes it, bit for bit, and
 * w_hat_t[t] = w_hat[t]^T (device BF16 [ntensors, cols, rows]), from one read
 * of w.  Errors: INVALID_ARG, ALIGNMENT, UNSUPPORTED (rows % 64, cols % 64). */
int nvfp4_fake_quant_transposed(const void *w, int32_t ntensors, int64_t rows, int64_t cols, void *w_hat,
                                void *w_hat_t, float *gs_out, float *amax_ws, int32_t *dev_status, void *stream);

/* nvfp4_fake_quant for callers that cannot allocate device memory.  The paper
 * has no counterpart; this is a convenience of the library.  A framework that
 * owns all device memory through its own pool, or a latency-critical loop
 * that must not call cudaMalloc/cudaFree (which can stall the whole device),
 * cannot provide the amax scratch that nvfp4_fake_quant asks for.  This
 * variant takes the same arguments minus `amax_ws` and computes the same
 * w_hat and gs_out (bit for bit), using a fixed array of 8193 32-bit words
 * that the library declares in device memory (32 KB held on every GPU that
 * loads the library, until the process exits) as nvfp4_fake_quant's scratch
 * for up to 4096 tensors.  Nothing is allocated by the call.
 *   - ntensors must be <= 4096: larger calls return NVFP4_ERR_UNSUPPORTED
 *     (nvfp4_last_error() says why) and launch nothing.
 *   - The first call on a device, with that device current, looks up the
 *     array's device address (cudaGetSymbolAddress); make that first call
 *     before any stream capture begins.  The address is kept per device and
 *     CUDA context: after a cudaDeviceReset the next call looks it up again
 *     (so, again, make that call outside any capture).
 *   - Device ordinals above 63 return NVFP4_ERR_ARCH, as every entry point.
 *   - Every call shares the one array: the slots a call uses are cleared on
 *     `stream` before use, and keep that call's amax values afterwards.  Calls
 *     whose work can overlap on the GPU (different streams without ordering
 *     between them, or several host threads) race on the array and must be
 *     serialized by the caller. */
int nvfp4_fake_quant_noalloc(const void *w, int32_t ntensors, int64_t rows, int64_t cols,
                             void *w_hat, float *gs_out, int32_t *dev_status, void *stream);

/* Rollout weight preparation, once per weight update (QUADS §3.2 Eq. 15: the
 * rollout loads the trainer's weights): per expert e of w [E, N, K] BF16,
 * NVFP4-quantize with the expert's own gs and gather the dequantized,
 * unscaled weight on the RAC channels:
 *   w_codes     device uint8 [E, N, K/2]
 *   w_scales    device uint8, E tensors of N x K in the scale layout (see
 *               top), E * ceil(N/128) * ceil(K/256) * 2048 bytes
 *   gs_w        device float[E]
 *   w_sel       device BF16 [E, N, k]: w_sel[e,n,s] = code*sb of W[e,n,S[s]]
 *               (exact in BF16; the GEMM multiplies by gs_w[e])
 *   amax_ws     device float[E] scratch.
 *   interleave  1: store rows in gate/up tile order for the fused SwiGLU
 *               epilogue: packed row 256t+i is source row 128t+i (i < 128, a
 *               gate row) or N/2 + 128t + i-128 (i >= 128, an up row).  Needs
 *               N % 256 == 0.  0: rows in source order.
 * Errors: INVALID_ARG, ALIGNMENT, UNSUPPORTED (K % 64, N % 128 (N % 256 when
 * interleaving), k % 8). */
int nvfp4_prepare_weights(const void *w, int32_t E, int64_t N, int64_t K, const int32_t *S,
                          int32_t k, int32_t interleave, uint8_t *w_codes, uint8_t *w_scales,
                          float *gs_w, void *w_sel, float *amax_ws, int32_t *dev_status,
                          void *stream);

/* Channel calibration, QUADS §3.3 Eq. 23-24 on a calibration batch x [M, K]
 * (BF16): score_j = ||Q_A(X)[:,j] - X[:,j]||_2 (summed in binary64, rows in
 * order), S = the k channels of largest score (ties to the lower index),
 * written in increasing order.  The build fixes S per projection site from
 * a calibration batch rather than online per forward pass.
 *   amax        device float: the batch's amax (nvfp4_amax)
 *   S_out       device int32[k]
 *   score_ws    device double[K] scratch; holds the squared scores after.
 * Errors: INVALID_ARG, ALIGNMENT, UNSUPPORTED (K % 16, K > 16384, k > K). */
int nvfp4_rac_select_channels(const void *x, int64_t M, int64_t K, const float *amax, int32_t k,
                              int32_t *S_out, double *score_ws, void *stream);

/* The literal second-pass form of RAC, QUADS §3.3 Eq. 21: the residual on S
 * is itself NVFP4-quantized, X~ = Q_A(X) + M_S * Q_A(r) with r = -Delta X_q.
 * Reading: Q_A acts on the gathered [rows, k] residual -- 16-element blocks
 * along the gathered channel axis -- with a tensor scale of its own, from
 * amax |r| over the routed rows.  Replaces, in place, the BF16 residual that
 * nvfp4_quantize stored (in units of gs_a) by Q_A(r) in the same units; every
 * such value is exact in BF16, so nvfp4_w4a4_rac_grouped_gemm applies the
 * second-pass correction unchanged.
 *   resid     device BF16 [rows_cap, k] (row pitch k), nvfp4_quantize's resid
 *   offsets   device int32[E+1] from nvfp4_route_topk: rows [0, offsets[E])
 *             are processed (their padding rows hold zeros); NULL: all rows
 *   amax_ws   device float scratch: receives max |resid| of those rows
 *   gs_out    device float or NULL: the residual's tensor scale (units of gs_a)
 * Rows past offsets[E] are neither read nor written.  dev_status gets
 * NONFINITE (and resid is left as it was) if the amax is not finite.
 * Errors: INVALID_ARG, ALIGNMENT, UNSUPPORTED (k % 16). */
int nvfp4_rac_requant_residual(void *resid, int64_t rows_cap, int32_t k, const int32_t *offsets, int32_t E,
                               float *amax_ws, float *gs_out, int32_t *dev_status, void *stream);

/* Online channel selection, QUADS §3.3 Eq. 23-24 applied to the batch at hand
 * on every forward pass (the paper's own mode; nvfp4_rac_select_channels is
 * the calibration form).  Same score and rule -- score_j^2 = sum over rows of
 * (Q_A(X)[i,j] - X[i,j])^2, S = the k largest, ties to the lower index, in
 * increasing order -- over the rows [0, offsets[E]) of a routed activation
 * (all rows_cap rows when offsets is NULL).  The sums are taken in a fixed
 * order built for speed (four-row binary32 partials into compensated binary32
 * sums per lane, binary64 across lanes and row chunks): deterministic, within
 * a few binary32 ulp of the exact sums, so channels whose scores tie that
 * closely may be chosen either way.
 *   x          device BF16 [rows_cap, K]
 *   amax       device float: the activation's amax (nvfp4_amax, or a GEMM's amax_out)
 *   S_out      device int32[k]
 *   score_ws   device double[257 * K]: squared scores in [0, K), then scratch.
 * Errors: INVALID_ARG, ALIGNMENT, UNSUPPORTED (K % 16, K > 16384, k > K). */
int nvfp4_rac_select_channels_online(const void *x, int64_t rows_cap, int64_t K, const int32_t *offsets, int32_t E,
                                     const float *amax, int32_t k, int32_t *S_out, double *score_ws, void *stream);

/* W_hat on S for the correction of QUADS §3.3 Eq. 21 when S changes (online
 * selection, Eq. 23-24).
 * The selected weight columns of a rollout weight pack, for a new channel set:
 * w_sel[e, n, s] = bf16(code * sb) of element (n, S[s]) of expert e -- what
 * nvfp4_prepare_weights writes for S -- read from its packed codes and block
 * scales (rows in the pack's own order, interleaved or not).
 *   w_codes, w_scales   from nvfp4_prepare_weights (E experts, N x K)
 *   S                   device int32[k], entries in [0, K) (others are clamped)
 *   w_sel               device BF16 [E, N, k]
 *   dev_status          device int32 or NULL: TIMEOUT if a copy wait ran out
 * Errors: INVALID_ARG, ALIGNMENT, UNSUPPORTED (K % 64, N % 128, k % 8,
 * E > 65535, K > 16384, or K and k too large for one block's shared memory). */
int nvfp4_gather_selected_weights(const uint8_t *w_codes, const uint8_t *w_scales, int32_t E, int64_t N, int64_t K,
                                  const int32_t *S, int32_t k, void *w_sel, int32_t *dev_status, void *stream);

/* A channel-major copy of a weight pack for the online selection of QUADS
 * §3.3 Eq. 23-24, made once per weight update, so that re-gathering W_hat on a
 * new S reads only the selected channels (nvfp4_gather_selected_weights_t):
 *   codes_t   device uint8 [E, K, N/2]: channel j of rows n, n+1 in one byte
 *             (row n in the low nibble)
 *   scales_t  device uint8 [E, K/16, N]: the block scale of row n, block kb
 * from w_codes [E, N, K/2] and w_scales (the pack of nvfp4_prepare_weights).
 * Errors: INVALID_ARG, ALIGNMENT (w_codes, codes_t), UNSUPPORTED (K % 64,
 * N % 128, E > 65535). */
int nvfp4_transpose_weight_pack(const uint8_t *w_codes, const uint8_t *w_scales, int32_t E, int64_t N, int64_t K,
                                uint8_t *codes_t, uint8_t *scales_t, void *stream);

/* nvfp4_gather_selected_weights from the channel-major copy
 * (nvfp4_transpose_weight_pack): the same w_sel [E, N, k], bit for bit,
 * reading k/K of the codes (QUADS §3.3 Eq. 21's W_hat on the S of Eq. 23-24).
 * Errors: INVALID_ARG, ALIGNMENT (codes_t, scales_t, w_sel), UNSUPPORTED
 * (K % 64, N % 128, k % 8, E > 65535). */
int nvfp4_gather_selected_weights_t(const uint8_t *codes_t, const uint8_t *scales_t, int32_t E, int64_t N, int64_t K,
                                    const int32_t *S, int32_t k, void *w_sel, void *stream);

/* ------------------------------------------------------------------------ */
/* Grouped GEMMs (QUADS §3.3 Eq. 21; §3.2 Eq. 12)                            */
/* ------------------------------------------------------------------------ */

/* W4A4 + RAC grouped GEMM on the FP4 tensor cores (tcgen05 block-scaled MMA
 * with E4M3 block scales, FP32 accumulation in tensor memory) plus the rank-k
 * BF16 correction of Residual Activation Compensation, QUADS §3.3 Eq. 21:
 *   y[r, n] = gs_a*gs_w[e] * ( sum_K (ca*sa)(cw*sw) + sum_{s<k} rg[r,s]*w_sel[e,n,s] )
 * for every routed row r in expert e's segment [offsets[e], offsets[e+1]),
 * where rg = r/gs_a is the residual as nvfp4_quantize stores it: both sums
 * accumulate in one FP32 tensor-memory accumulator, the correction as BF16
 * MMAs over the k selected channels.
 *   a_codes/a_scales  device, the routed activations from nvfp4_quantize,
 *                     rows_cap rows; a_resid device BF16 [rows_cap, k]
 *   gs_a              device float (nvfp4_quantize's gs_out)
 *   w_codes/w_scales/gs_w/w_sel  from nvfp4_prepare_weights (E experts, N x K)
 *   offsets           device int32[E+1], non-decreasing multiples of 128,
 *                     offsets[0] = 0, offsets[E] <= rows_cap
 *   epilogue          NVFP4_EPI_NONE: y [rows_cap, N] (ldy >= N).
 *                     NVFP4_EPI_SWIGLU: the weights were prepared with
 *                     interleave = 1; y = bf16(silu(gate) * up) [rows_cap, N/2]
 *                     (ldy >= N/2, out_dtype must be BF16).
 * Tiles: 128 x 256 outputs per CTA (single-CTA pipeline, the default for this
 * kind) or 256 x 256 per CTA pair (pair pipeline); see nvfp4_gemm_pipeline.
 *   out_dtype         NVFP4_OUT_F32 or NVFP4_OUT_BF16 (= bf16_rn of the F32 value)
 *   amax_out          device float or NULL: receives max|y| of the stored
 *                     values (the next quantize's amax); the call clears it
 *                     on `stream` before the kernel runs.
 * Rows of a segment beyond the expert's real token count must hold zero
 * codes/scales/residual (nvfp4_moe_clear_padding); their outputs are zero.
 * The correction runs ceil(k/64) BF16 slices after the K loop, so any k up to
 * K works (the pages' k = 50% of the channels, QUADS §4.4.1, included; its
 * cost grows with k).
 * Errors: INVALID_ARG, ALIGNMENT, UNSUPPORTED (K % 256, N % 256, k % 16,
 * k > K, E > 1024); dev_status gets TIMEOUT if a pipeline wait runs out. */
int nvfp4_w4a4_rac_grouped_gemm(const uint8_t *a_codes, const uint8_t *a_scales,
                                const void *a_resid, const float *gs_a, const uint8_t *w_codes,
                                const uint8_t *w_scales, const float *gs_w, const void *w_sel,
                                int32_t k, const int32_t *offsets, int32_t E, int64_t rows_cap,
                                int64_t N, int64_t K, int32_t epilogue, int32_t out_dtype,
                                void *y, int64_t ldy, float *amax_out, int32_t *dev_status,
                                void *stream);

/* BF16 grouped GEMM of the asymmetric-QAT forward, QUADS §3.2 Eq. 12:
 * y[r, n] = sum_K x[r, K] * w_hat[e, n, K] (tcgen05 BF16 MMA, FP32 accumulate)
 * for routed rows r of expert e.
 *   x        device BF16 [rows_cap, K] (routed rows, see nvfp4_moe_scatter_rows)
 *   w_hat    device BF16 [E, N, K] (nvfp4_fake_quant output, rows in source
 *            order: for SwiGLU, gate rows [0, N/2) then up rows [N/2, N))
 *   offsets  as for nvfp4_w4a4_rac_grouped_gemm
 *   epilogue NVFP4_EPI_NONE: y [rows_cap, N]; NVFP4_EPI_SWIGLU: y =
 *            bf16(silu(gate) * up) [rows_cap, N/2] (out_dtype must be BF16);
 *            NVFP4_EPI_SWIGLU_SAVE: y as for NVFP4_EPI_SWIGLU, and the
 *            pre-activations bf16(gate | up) -- the NVFP4_EPI_NONE output
 *            with BF16 out_dtype, bit for bit -- to gu (the learner's
 *            forward keeps them for the SwiGLU backward of Eq. 13).
 *   gu       device BF16 [rows_cap, N] for NVFP4_EPI_SWIGLU_SAVE, else NULL
 * Errors: INVALID_ARG, ALIGNMENT, UNSUPPORTED (K % 64, N % 256, E > 1024). */
int nvfp4_bf16_grouped_gemm(const void *x, const void *w_hat, const int32_t *offsets, int32_t E,
                            int64_t rows_cap, int64_t N, int64_t K, int32_t out_dtype,
                            int32_t epilogue, void *y, int64_t ldy, void *gu, int32_t *dev_status,
                            void *stream);

/* Pipeline of the two grouped GEMMs above (no counterpart in the paper: an
 * implementation choice).  Both pipelines compute the same results:
 *   NVFP4_PIPELINE_SINGLE  one CTA per 128 x 256 output tile (tcgen05 cta_group::1)
 *   NVFP4_PIPELINE_PAIR    a cluster of two CTAs per 256 x 256 tile
 *                          (tcgen05 cta_group::2: each SM holds half of B)
 *   NVFP4_PIPELINE_AUTO    (initial) the one measured faster per kind on GB300:
 *                          single for W4A4 + RAC, pair for BF16.
 * Process-wide; takes effect for calls made after it returns.
 *   previous  host int32 or NULL: receives the setting it replaces.
 * Errors: INVALID_ARG (unknown value). */
int nvfp4_gemm_pipeline(int32_t which, int32_t *previous);

/* ------------------------------------------------------------------------ */
/* MoE routing, dispatch and combine (not described by QUADS; the plainest    */
/* top-k softmax MoE)                                                         */
/* ------------------------------------------------------------------------ */

/* MoE glue (not described by QUADS).
 * Top-k softmax router.  For each token t: p = softmax(logits[t]) in FP32;
 * ids[t] = the topk experts of largest logit (ties to the lower expert
 * index, in decreasing order), weights[t] = their p (no renormalization).
 * Routed rows are ordered by (expert, token); each expert segment starts at
 * a multiple of 128:
 *   counts   device int32[E]      tokens routed to each expert
 *   offsets  device int32[E+1]    padded segment starts (offsets[E] = total)
 *   dst_row  device int32[T*topk] routed row of (t, slot)
 * All outputs are overwritten.  Needs topk <= 32 and topk <= E <= 1024. */
int nvfp4_route_topk(const float *logits, int32_t T, int32_t E, int32_t topk, int32_t *ids,
                     float *weights, int32_t *counts, int32_t *offsets, int32_t *dst_row,
                     void *stream);

/* MoE glue (not described by QUADS).
 * Zero the padding rows [offsets[e]+counts[e], offsets[e+1]) of a routed
 * NVFP4 activation (codes [rows_cap, K/2], block scales, resid [rows_cap,
 * k] BF16 or NULL when k = 0), so that padded rows contribute zeros. */
int nvfp4_moe_clear_padding(const int32_t *counts, const int32_t *offsets, int32_t E,
                            int64_t rows_cap, int64_t K, int32_t k, uint8_t *codes,
                            uint8_t *scales, void *resid, void *stream);

/* MoE glue (not described by QUADS).
 * Copy BF16 token rows x [T, K] to their routed rows y [rows_cap, K]
 * (y[dst_row[t*topk+s]] = x[t]) and zero the padding rows (the QAT path's
 * dispatch).  counts/offsets/dst_row from nvfp4_route_topk. */
int nvfp4_moe_scatter_rows(const void *x, int32_t T, int64_t K, int32_t topk,
                           const int32_t *dst_row, const int32_t *counts, const int32_t *offsets,
                           int32_t E, int64_t rows_cap, void *y, void *stream);

/* MoE glue (not described by QUADS).
 * Weighted combine: out[t, :] = sum_{s<topk} weights[t,s] * y[dst_row[t,s], :]
 * in FP32, slots in order.  y is F32 or BF16 (y_dtype) with row stride ldy.
 *   out  device float [T, H] (overwritten). */
int nvfp4_moe_combine(const void *y, int32_t y_dtype, int64_t ldy, const int32_t *dst_row,
                      const float *weights, int32_t T, int32_t topk, int64_t H, float *out,
                      void *stream);

/* ------------------------------------------------------------------------ */
/* Trainer backward (QUADS §3.2 Eq. 13: straight-through estimator)           */
/* ------------------------------------------------------------------------ */
/* The asymmetric-QAT learner treats the weight fake-quantizer as the identity
 * in the backward pass: dW = dW_hat and dX = W_hat^T dY (Eq. 13).  For one MoE
 * layer out = combine(swiglu(scatter(x) W13_hat^T) Wd_hat^T) the backward is
 * combine backward -> dY routed; dh = dY Wd_hat; dWd = dY^T h; SwiGLU backward
 * -> d(gate|up); dx_routed = d(gate|up) W13_hat; dW13 = d(gate|up)^T x_routed;
 * dx = the sum of each token's routed rows (nvfp4_moe_combine with unit
 * weights).  The input-gradient products run on nvfp4_bf16_grouped_gemm_dgrad,
 * which reads W_hat as stored (no transposed copy), the weight gradients on
 * nvfp4_bf16_grouped_gemm_wgrad_rows, which reads the routed rows as stored
 * (no transposes); nvfp4_bf16_grouped_gemm_wgrad takes transposed operands. */

/* Data movement of the trainer backward (QUADS §3.2 Eq. 13).
 * y[b] = x[b]^T for `batch` row-major BF16 matrices of rows x cols (y[b] is
 * cols x rows).  x and y may not overlap.  Errors: INVALID_ARG, UNSUPPORTED
 * (batch > 65535). */
int nvfp4_transpose_bf16(const void *x, int32_t batch, int64_t rows, int64_t cols, void *y, void *stream);

/* The SwiGLU of the MoE experts (glue, not described by QUADS), on saved
 * pre-activations for the trainer backward of QUADS §3.2 Eq. 13.
 * h = bf16(silu(g) * u) from saved BF16 pre-activations gu = [g | u]
 * (rows x 2I, the gate columns first), silu(g) = g / (1 + exp(-g)) in
 * binary32.  h: device BF16 [rows, I].  Errors: INVALID_ARG. */
int nvfp4_swiglu(const void *gu, int64_t rows, int64_t I, void *h, void *stream);

/* Part of the trainer backward of QUADS §3.2 Eq. 13.
 * SwiGLU backward: from gu = [g | u] and dh (rows x I, BF16),
 * d(gate) = bf16(dh * u * s (1 + g (1 - s))) and d(up) = bf16(dh * g * s),
 * s = 1 / (1 + exp(-g)), in binary32, written as dgu = [dg | du] (rows x 2I).
 * Errors: INVALID_ARG. */
int nvfp4_swiglu_backward(const void *gu, const void *dh, int64_t rows, int64_t I, void *dgu, void *stream);

/* Part of the trainer backward of QUADS §3.2 Eq. 13.
 * Backward of nvfp4_moe_combine: dy[dst_row[t,s]] = bf16(weights[t,s] *
 * dout[t]) for every token t and slot s (rows outside [0, rows_cap) are
 * skipped), the padding rows [offsets[e] + counts[e], offsets[e+1]) of dy set
 * to zero, and, when dweights is not NULL, the combine weights' gradient
 * dweights[t,s] = sum_h y[dst_row[t,s], h] * dout[t, h] (binary32).
 *   dout      device float [T, H];  y  device BF16 [rows_cap, H] (the forward's rows)
 *   dy        device BF16 [rows_cap, H];  dweights  device float [T, topk] or NULL
 * Errors: INVALID_ARG, ALIGNMENT (16-byte pointers), UNSUPPORTED (E > 65535,
 * H % 8, H > 8192, topk > 32). */
int nvfp4_moe_combine_backward(const float *dout, const void *y, const int32_t *dst_row, const float *weights,
                               int32_t T, int32_t topk, int64_t H, const int32_t *counts, const int32_t *offsets,
                               int32_t E, int64_t rows_cap, void *dy, float *dweights, void *stream);

/* dW = dW_hat of the straight-through estimator, QUADS §3.2 Eq. 13.
 * Grouped weight gradient: dw[e] = a_t[:, seg e] . b_t[:, seg e]^T for every
 * expert e, seg e = the routed rows [offsets[e], offsets[e+1]) (tcgen05 BF16
 * MMA, FP32 accumulation over the expert's rows; an expert without rows gets
 * zeros).  The operands are the transposed routed tensors, so the reduction
 * axis is contiguous:
 *   a_t      device BF16 [M, R] (e.g. dY^T of a projection's output)
 *   b_t      device BF16 [N, R] (e.g. its input, transposed)
 *   offsets  device int32[E+1] as for nvfp4_bf16_grouped_gemm, offsets[E] <= R
 *   dw       device [E, M, N], F32 or BF16 (out_dtype)
 * Runs on the single-CTA pipeline whatever nvfp4_gemm_pipeline selects.
 * Errors: INVALID_ARG, ALIGNMENT, UNSUPPORTED (M % 128, N % 256, R % 128,
 * E > 1024); dev_status gets TIMEOUT if a pipeline wait runs out. */
int nvfp4_bf16_grouped_gemm_wgrad(const void *a_t, const void *b_t, const int32_t *offsets, int32_t E, int64_t R,
                                  int64_t M, int64_t N, int32_t out_dtype, void *dw, int32_t *dev_status,
                                  void *stream);

/* dX = W_hat^T dY of the straight-through estimator, QUADS §3.2 Eq. 13.
 * Grouped input gradient with the weights as stored:
 * y[r, n] = sum_k dy[r, k] * w_hat[e, k, n] for the routed rows r of expert e
 * (tcgen05 BF16 MMA, FP32 accumulate; the weights are read MN-major, so no
 * transposed copy of W_hat is needed).
 *   dy       device BF16 [rows_cap, K] (routed output gradient)
 *   w_hat    device BF16 [E, K, N] (the forward weight: K outputs x N inputs,
 *            e.g. nvfp4_fake_quant output)
 *   offsets  as for nvfp4_bf16_grouped_gemm
 *   epilogue NVFP4_EPI_NONE: y [rows_cap, N] (ldy >= N), F32 or BF16 (out_dtype).
 *            NVFP4_EPI_SWIGLU_BWD: the product is dh, the gradient of a SwiGLU
 *            output h = silu(g) * u; with gu = the saved pre-activations
 *            [g | u] (device BF16 [rows_cap, 2N]) the epilogue writes
 *            y = [d(gate) | d(up)] (BF16 [rows_cap, 2N], ldy >= 2N), exactly
 *            what nvfp4_swiglu_backward computes from dh rounded to BF16 -- so
 *            dh itself never goes to memory.  out_dtype must be BF16.
 *   gu       device BF16 [rows_cap, 2N] for NVFP4_EPI_SWIGLU_BWD, else NULL
 * Runs on the pipeline nvfp4_gemm_pipeline selects for BF16.
 * Errors: INVALID_ARG, ALIGNMENT, UNSUPPORTED (K % 64, N % 256, E > 1024,
 * E*K > 2^31); dev_status gets TIMEOUT if a pipeline wait runs out. */
int nvfp4_bf16_grouped_gemm_dgrad(const void *dy, const void *w_hat, const int32_t *offsets, int32_t E,
                                  int64_t rows_cap, int64_t N, int64_t K, int32_t out_dtype,
                                  int32_t epilogue, const void *gu, void *y, int64_t ldy,
                                  int32_t *dev_status, void *stream);

/* dW = dW_hat of the straight-through estimator, QUADS §3.2 Eq. 13, from the
 * routed rows as stored: dw[e] = a[seg e, :]^T . b[seg e, :] for every expert
 * e, seg e = the routed rows [offsets[e], offsets[e+1]) -- the same product
 * as nvfp4_bf16_grouped_gemm_wgrad, with both operands read MN-major, so no
 * transposes are needed.
 *   a   device BF16 [R, M] (e.g. dY of a projection's output)
 *   b   device BF16 [R, N] (e.g. its input)
 *   offsets, dw, out_dtype, errors: as for nvfp4_bf16_grouped_gemm_wgrad. */
int nvfp4_bf16_grouped_gemm_wgrad_rows(const void *a, const void *b, const int32_t *offsets, int32_t E,
                                       int64_t R, int64_t M, int64_t N, int32_t out_dtype, void *dw,
                                       int32_t *dev_status, void *stream);

/* ------------------------------------------------------------------------ */
/* Diagnostics                                                                */
/* ------------------------------------------------------------------------ */

/* Failure handling (no counterpart in QUADS).
 * Runs one CTA that waits, with the library's bounded-wait routine and a
 * limit of `limit_us` microseconds (1 .. 10^7), on a pipeline barrier that
 * nothing ever signals; when the limit runs out it writes NVFP4_ERR_TIMEOUT
 * to dev_status and returns normally.  Exercises the timeout path without a
 * real fault.  The GEMM pipelines use the same routine with a 2 s limit. */
int nvfp4_selftest_wait_timeout(int32_t limit_us, int32_t *dev_status, void *stream);

/* dX = W_hat^T dY of the straight-through estimator, QUADS §3.2 Eq. 13.
 * Grouped input gradient with the weights as stored:
 * y[r, n] = sum_k dy[r, k] * w_hat[e, k, n] for the routed rows r of expert e
 * (tcgen05 BF16 MMA, FP32 accumulate; the weights are read MN-major, so no
 * transposed copy of W_hat is needed).
 *   dy       device BF16 [rows_cap, K] (routed output gradient)
 *   w_hat    device BF16 [E, K, N] (the forward weight: K outputs x N inputs,
 *            e.g. nvfp4_fake_quant output)
 *   offsets  as for nvfp4_bf16_grouped_gemm
 *   epilogue NVFP4_EPI_NONE: y [rows_cap, N] (ldy >= N), F32 or BF16 (out_dtype).
 *            NVFP4_EPI_SWIGLU_BWD: the product is dh, the gradient of a SwiGLU
 *            output h = silu(g) * u; with gu = the saved pre-activations
 *            [g | u] (device BF16 [rows_cap, 2N]) the epilogue writes
 *            y = [d(gate) | d(up)] (BF16 [rows_cap, 2N], ldy >= 2N), exactly
 *            what nvfp4_swiglu_backward computes from dh rounded to BF16 -- so
 *            dh itself never goes to memory.  out_dtype must be BF16.
 *   gu       device BF16 [rows_cap, 2N] for NVFP4_EPI_SWIGLU_BWD, else NULL
 * Runs on the pipeline nvfp4_gemm_pipeline selects for BF16.
 * Errors: INVALID_ARG, ALIGNMENT, UNSUPPORTED (K % 64, N % 256, E > 1024,
 * E*K > 2^31); dev_status gets TIMEOUT if a pipeline wait runs out. */
int nvfp4_bf16_grouped_gemm_dgrad(const void *dy, const void *w_hat, const int32_t *offsets, int32_t E,
                                  int64_t rows_cap, int64_t N, int64_t K, int32_t out_dtype,
                                  int32_t epilogue, const void *gu, void *y, int64_t ldy,
                                  int32_t *dev_status, void *stream);

/* dW = dW_hat of the straight-through estimator, QUADS §3.2 Eq. 13, from the
 * routed rows as stored: dw[e] = a[seg e, :]^T . b[seg e, :] for every expert
 * e, seg e = the routed rows [offsets[e], offsets[e+1]) -- the same product
 * as nvfp4_bf16_grouped_gemm_wgrad, with both operands read MN-major, so no
 * transposes are needed.
 *   a   device BF16 [R, M] (e.g. dY of a projection's output)
 *   b   device BF16 [R, N] (e.g. its input)
 *   offsets, dw, out_dtype, errors: as for nvfp4_bf16_grouped_gemm_wgrad. */
int nvfp4_bf16_grouped_gemm_wgrad_rows(const void *a, const void *b, const int32_t *offsets, int32_t E,
                                       int64_t R, int64_t M, int64_t N, int32_t out_dtype, void *dw,
                                       int32_t *dev_status, void *stream);

/* ------------------------------------------------------------------------ */
/* Diagnostics                                                                */
/* ------------------------------------------------------------------------ */

/* Layer-wise forward mismatch of QUADS §3.1 Eq. 11, dY = ||Y_infer - Y_train||_2
 * (Frobenius norm over the layer output), with the reference's own norm for
 * scale: acc[0] = sum (y_infer - y_train)^2 and acc[1] = sum y_train^2 over
 * the n elements, in binary64 (per-block partial sums added atomically, so the
 * last bits depend on the order the blocks finish).  The call clears acc on
 * `stream` first; dY = sqrt(acc[0]).
 *   y_infer, y_train  device float[n]
 *   acc               device double[2]
 * Errors: INVALID_ARG, ALIGNMENT (16-byte pointers). */
int nvfp4_mismatch_norm(const float *y_infer, const float *y_train, int64_t n, double *acc, void *stream);

#ifdef __cplusplus
}
#endif

#endif /* NVFP4MOE_H */
