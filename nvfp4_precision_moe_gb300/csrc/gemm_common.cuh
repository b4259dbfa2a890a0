// gemm_common.cuh -- what the two grouped-GEMM pipelines (gemm_single.cu,
// gemm_pair.cu) share: tile and tensor-memory constants, the warp layout and
// its register split, the launch parameters, and the epilogue helpers that
// scale, apply SwiGLU and store an accumulator row segment.
#pragma once
#include "common.cuh"

namespace nvfp4 {

constexpr int kBM = 128;             // output rows per CTA
constexpr int kBN = 256;             // output columns per tile
constexpr int kATileBytes = 16384;   // 128 rows x 128 bytes of K
constexpr int kSFABytes = 2048;      // the A tile's scales: one 2048-byte tile of the scale layout
constexpr int kSFBBytes = 4096;      // the scales of all 256 B rows of a tile: two tiles
constexpr uint32_t kTmemCols = 512;
// Tensor memory: the accumulator, then one scale slot per stage.  A scales in
// its first 16 columns: MMA chunk c reads columns 4c..4c+3, in lane quarter q
// column 4c + q at lane r%32 for row r = 32q + r%32 (every quarter gets the
// same copy of group c).  B scales in the next 32: chunk c reads columns
// 16 + 8c .. 16 + 8c + 7, column 16 + 8c + n/32 at lane n%32 of every quarter
// for B row n.  (Scale addresses of the block-scaled MMA are 4-column aligned.)
constexpr uint32_t kAcc = 0, kSFCol0 = 256, kSFSlotCols = 48, kSFBCol = 16;
// Instruction-descriptor bits of kind::f16 MMAs: operand A / B is MN-major
// (its M / N index contiguous in shared memory) rather than K-major.
constexpr uint32_t kIdescTransA = 1u << 15, kIdescTransB = 1u << 16;
constexpr uint64_t kWaitLimitNs = 2000000000ull;  // 2 s per wait
constexpr int kMaxExperts = 1024;
// Warp roles per CTA (512 threads, four warpgroups):
//   warp 0      TMA producer (one lane)
//   warp 1      TMEM owner + MMA issuer (one lane)
//   warps 2-3   idle
//   warps 4-7   scale warps (FP4, single-CTA pipeline): once a stage's block
//               scales have landed, each writes them into its 32-lane quarter
//               of tensor memory with tcgen05.st, as the block-scaled MMA reads
//               them.  (The pair pipeline copies them with tcgen05.cp in the
//               MMA stream instead; there these warps idle.)
//   warps 8-15  epilogue: warp w reads TMEM lane quarter w%4 and column half
//               (w-8)/4 of the tile -- all 128 of a thread's columns at once --
//               releases the accumulator, then scales, applies SwiGLU and
//               stores while the next tile's MMAs run
constexpr int kEpiWarps = 8;
constexpr int kSFWarps = 4;
constexpr int kSFWarp0 = 4;   // warpgroup 1
constexpr int kEpiWarp0 = 8;  // warpgroups 2 and 3
constexpr int kThreads = 32 * (kEpiWarp0 + kEpiWarps);
// Register split (per thread) after launch at 65536 / 512 = 128: the producer
// and MMA warpgroup and the scale warpgroup give registers to the epilogue,
// which holds a thread's 128 accumulator columns at once.
constexpr uint32_t kRegsCtl = 88, kRegsSF = 72, kRegsEpi = 176;
static_assert(128 * kRegsCtl + 128 * kRegsSF + 256 * kRegsEpi <= 65536, "register split above the launch budget");

struct GemmParams {
    const uint8_t *a_codes_base;  // the A operand's base (at least 16 KB readable): the pair pipeline's abort drain
    const uint8_t *a_scales;
    const uint8_t *w_scales;
    const float *gs_a;
    const float *gs_w;
    const int32_t *offsets;
    int32_t rows_cap;
    int32_t E, k;
    int64_t N, K;
    int32_t epilogue, out_dtype;
    void *y;
    int64_t ldy;
    int32_t vec32;  // y and its row pitch are 32-byte aligned: whole-sector stores
    float *amax_out;
    int32_t *dev_status;
    // weight-gradient mode (BF16, single-CTA pipeline): y[e] (M x N) = A[:, seg e] . B[:, seg e]^T,
    // A [M, rows_cap] and B [N, rows_cap] K-major (or [rows_cap, M] and [rows_cap, N] MN-major),
    // seg e = [offsets[e], offsets[e+1])
    int32_t wgrad;
    int64_t M;
    int32_t wgrad_f32;  // FP32 weight gradients: rows staged through shared memory, stored 128 bytes at a time
    // BF16 operands stored MN-major (the M or N index contiguous): A (weight-gradient mode) and B
    // (both modes) arrive as TMA boxes of 64 MN-elements x 64 K-rows, 8 KB apart (desc_sw128_mn)
    int32_t a_mn, b_mn;
    // NVFP4_EPI_SWIGLU_BWD (BF16): the saved pre-activations [g | u], [rows_cap, 2N]
    const uint16_t *gu;
    // NVFP4_EPI_SWIGLU_SAVE (BF16): where the pre-activations go, [rows_cap, N]; gu_vec32: 32-byte aligned
    uint16_t *gu_out;
    int32_t gu_vec32;
};

__device__ __forceinline__ uint32_t pack_bf16x2(float a, float b) {
    return (uint32_t)__bfloat16_as_ushort(__float2bfloat16_rn(a)) |
           ((uint32_t)__bfloat16_as_ushort(__float2bfloat16_rn(b)) << 16);
}

// silu(g) * u with the fast exponential and division (a few ulp; the BF16
// rounding of the result dominates).
__device__ __forceinline__ float swiglu1(float g, float u) {
    const float e = __expf(-g);
    return __fmul_rn(__fdividef(g, 1.0f + e), u);
}

// 16 accumulator columns rounded to BF16 (bf16_rn, as the NVFP4_EPI_NONE BF16
// output) and stored as 32 bytes.
__device__ __forceinline__ void store_bf16x16(uint16_t *dst, bool vec32, const uint32_t *d);

// 8 words to a 32-byte output segment: one whole-sector store when the
// output allows it (stores are a large share of the kernel's L2 requests),
// else two 16-byte stores.
__device__ __forceinline__ void store32B(void *dst, bool vec32, uint32_t a0, uint32_t a1, uint32_t a2, uint32_t a3,
                                         uint32_t a4, uint32_t a5, uint32_t a6, uint32_t a7) {
    if (vec32) {
        st_global_v8(dst, a0, a1, a2, a3, a4, a5, a6, a7);
    } else {
        uint4 *d = reinterpret_cast<uint4 *>(dst);
        d[0] = make_uint4(a0, a1, a2, a3);
        d[1] = make_uint4(a4, a5, a6, a7);
    }
}

__device__ __forceinline__ void store_bf16x16(uint16_t *dst, bool vec32, const uint32_t *d) {
    uint32_t o[8];
#pragma unroll
    for (int i = 0; i < 8; ++i) o[i] = pack_bf16x2(__uint_as_float(d[2 * i]), __uint_as_float(d[2 * i + 1]));
    store32B(dst, vec32, o[0], o[1], o[2], o[3], o[4], o[5], o[6], o[7]);
}

// 16 columns of this warp's TMEM rows -> 16 BF16 stores (32 bytes), or 16
// FP32 stores (64 bytes); tracks max|stored value|.
__device__ __forceinline__ void store16(const GemmParams &p, int64_t row, int64_t col, float gmul,
                                        const uint32_t *d, float &amax_local) {
    float v[16];
#pragma unroll
    for (int i = 0; i < 16; ++i) v[i] = __fmul_rn(gmul, __uint_as_float(d[i]));
    if (p.out_dtype == NVFP4_OUT_F32) {
        float *dst = reinterpret_cast<float *>(p.y) + row * p.ldy + col;
#pragma unroll
        for (int i = 0; i < 2; ++i)
            store32B(dst + 8 * i, p.vec32, __float_as_uint(v[8 * i]), __float_as_uint(v[8 * i + 1]),
                     __float_as_uint(v[8 * i + 2]), __float_as_uint(v[8 * i + 3]), __float_as_uint(v[8 * i + 4]),
                     __float_as_uint(v[8 * i + 5]), __float_as_uint(v[8 * i + 6]), __float_as_uint(v[8 * i + 7]));
#pragma unroll
        for (int i = 0; i < 16; ++i) amax_local = fmaxf(amax_local, fabsf(v[i]));
    } else {
        uint32_t o[8];
#pragma unroll
        for (int i = 0; i < 8; ++i) {
            o[i] = pack_bf16x2(v[2 * i], v[2 * i + 1]);
            amax_local = fmaxf(amax_local, fabsf(__uint_as_float(o[i] << 16)));
            amax_local = fmaxf(amax_local, fabsf(__uint_as_float(o[i] & 0xffff0000u)));
        }
        store32B(reinterpret_cast<uint16_t *>(p.y) + row * p.ldy + col, p.vec32, o[0], o[1], o[2], o[3], o[4], o[5],
                 o[6], o[7]);
    }
}

// 16 SwiGLU outputs from 16 gate and 16 up columns -> 32 bytes of BF16.
__device__ __forceinline__ void swiglu16(uint16_t *dst16, bool vec32, float gmul, const uint32_t *g,
                                         const uint32_t *u, float &amax_local) {
    uint32_t o[8];
#pragma unroll
    for (int i = 0; i < 16; i += 2) {
        const float h0 = swiglu1(__fmul_rn(gmul, __uint_as_float(g[i])), __fmul_rn(gmul, __uint_as_float(u[i])));
        const float h1 =
            swiglu1(__fmul_rn(gmul, __uint_as_float(g[i + 1])), __fmul_rn(gmul, __uint_as_float(u[i + 1])));
        o[i / 2] = pack_bf16x2(h0, h1);
        amax_local = fmaxf(amax_local, fabsf(__uint_as_float(o[i / 2] << 16)));
        amax_local = fmaxf(amax_local, fabsf(__uint_as_float(o[i / 2] & 0xffff0000u)));
    }
    store32B(dst16, vec32, o[0], o[1], o[2], o[3], o[4], o[5], o[6], o[7]);
}

// The SwiGLU backward of 16 columns col..col+15 of row `row` (BF16 pipelines,
// NVFP4_EPI_SWIGLU_BWD): the accumulator holds dh = dY W_hat; rounded to BF16
// (as a stored dh would be) and with the saved pre-activations g, u of those
// columns it gives d(gate) = bf16(dh u s (1 + g (1 - s))) and d(up) =
// bf16(dh g s), s = 1 / (1 + exp(-g)) in binary32, stored at columns col and
// N + col of y -- the arithmetic of nvfp4_swiglu_backward.
__device__ __forceinline__ void swiglu_bwd16(const GemmParams &p, int64_t row, int64_t col, const uint32_t *d) {
    const uint16_t *gr = p.gu + row * 2 * p.N + col;
    const uint4 g0 = __ldg(reinterpret_cast<const uint4 *>(gr)), g1 = __ldg(reinterpret_cast<const uint4 *>(gr) + 1);
    const uint4 u0 = __ldg(reinterpret_cast<const uint4 *>(gr + p.N)),
                u1 = __ldg(reinterpret_cast<const uint4 *>(gr + p.N) + 1);
    const uint32_t G[8] = {g0.x, g0.y, g0.z, g0.w, g1.x, g1.y, g1.z, g1.w};
    const uint32_t U[8] = {u0.x, u0.y, u0.z, u0.w, u1.x, u1.y, u1.z, u1.w};
    uint32_t og[8], ou[8];
#pragma unroll
    for (int i = 0; i < 8; ++i) {
        float rg[2], ru[2];
#pragma unroll
        for (int hh = 0; hh < 2; ++hh) {
            const float g = __uint_as_float(hh ? (G[i] & 0xffff0000u) : (G[i] << 16));
            const float u = __uint_as_float(hh ? (U[i] & 0xffff0000u) : (U[i] << 16));
            const float dh = __bfloat162float(__float2bfloat16_rn(__uint_as_float(d[2 * i + hh])));
            const float s = __frcp_rn(__fadd_rn(1.0f, expf(-g)));
            const float ds = __fmul_rn(s, __fadd_rn(1.0f, __fmul_rn(g, __fsub_rn(1.0f, s))));
            rg[hh] = __fmul_rn(__fmul_rn(dh, u), ds);
            ru[hh] = __fmul_rn(dh, __fmul_rn(g, s));
        }
        og[i] = pack_bf16x2(rg[0], rg[1]);
        ou[i] = pack_bf16x2(ru[0], ru[1]);
    }
    uint16_t *yr = reinterpret_cast<uint16_t *>(p.y) + row * p.ldy + col;
    store32B(yr, p.vec32, og[0], og[1], og[2], og[3], og[4], og[5], og[6], og[7]);
    store32B(yr + p.N, p.vec32, ou[0], ou[1], ou[2], ou[3], ou[4], ou[5], ou[6], ou[7]);
}

// One stage's block scales, from shared memory to this warp's 32-lane quarter
// of the stage's tensor-memory slot -- the image the pair pipeline's
// tcgen05.cp copies produce.  Shared memory holds the A tile's scale tile and
// then those of B rows 0-127 and 128-255 (2048 bytes each: a 512-byte group
// per MMA chunk c, row r on line r%32, 4 bytes per row at 4*(r/32)).  Line
// `lane` of group c goes to columns 4c..4c+3 (A) or 16 + 8c + 4t .. +3 (B,
// tile t).  The caller waits for the stores.
__device__ __forceinline__ void sf_stage_to_tmem(const uint8_t *sfs, uint32_t base, int lane) {
    uint32_t ra[16];
#pragma unroll
    for (int c = 0; c < 4; ++c) {
        const uint4 w = *reinterpret_cast<const uint4 *>(sfs + c * 512 + 16 * lane);
        ra[4 * c] = w.x;
        ra[4 * c + 1] = w.y;
        ra[4 * c + 2] = w.z;
        ra[4 * c + 3] = w.w;
    }
    tmem_st16(base, ra);
    uint32_t rb[32];
#pragma unroll
    for (int c = 0; c < 4; ++c)
#pragma unroll
        for (int t = 0; t < 2; ++t) {
            const uint4 w = *reinterpret_cast<const uint4 *>(sfs + kSFABytes + t * 2048 + c * 512 + 16 * lane);
            rb[8 * c + 4 * t] = w.x;
            rb[8 * c + 4 * t + 1] = w.y;
            rb[8 * c + 4 * t + 2] = w.z;
            rb[8 * c + 4 * t + 3] = w.w;
        }
    tmem_st32(base + kSFBCol, rb);
}

// Launchers of the two pipelines (FP4: W4A4 + RAC; !FP4: BF16).  Tensor maps:
// A rows (box 128 rows), B rows (single: 256-row box for FP4, two 128-row
// boxes for BF16; pair: one 128-row box, this CTA's half), the RAC residual and
// the selected weight columns (single: 256-row box; pair: 128-row box).
template <bool FP4>
int launch_single_gemm(const CUtensorMap &tA, const CUtensorMap &tB, const CUtensorMap &tR, const CUtensorMap &tW,
                       const GemmParams &p, int64_t rows_cap, int64_t N, cudaStream_t stream);
// The pair pipeline also takes the two scale tensors as maps (FP4; unused for
// BF16): the activation's and the weights' scales, each as rows of 256 bytes.
template <bool FP4>
int launch_pair_gemm(const CUtensorMap &tA, const CUtensorMap &tB, const CUtensorMap &tR, const CUtensorMap &tW,
                     const CUtensorMap &tSA, const CUtensorMap &tSB, const GemmParams &p, int64_t rows_cap, int64_t N,
                     cudaStream_t stream);

}  // namespace nvfp4
