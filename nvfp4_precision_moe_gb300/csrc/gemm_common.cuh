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
constexpr int kSFABytes = 2048;      // 4 MMA-K chunks x 512 bytes (128 rows x 4 scales)
constexpr int kSFBBytes = 4096;      // the scales of all 256 B rows of a tile
constexpr uint32_t kTmemCols = 512;
constexpr uint32_t kAcc = 0, kSFCol0 = 256, kSFSlotCols = 48;  // accumulator; per-stage scale slots
constexpr uint64_t kWaitLimitNs = 2000000000ull;  // 2 s per wait
constexpr int kMaxExperts = 1024;
// Warp roles per CTA (512 threads, four warpgroups):
//   warp 0      TMA producer (one lane)
//   warp 1      TMEM owner + MMA issuer (one lane)
//   warps 2-3   idle
//   warps 4-7   scale warps (FP4): once a stage's block scales have landed,
//               each writes them into its 32-lane quarter of tensor memory with
//               tcgen05.st, replicated as the block-scaled MMA reads them
//               (tcgen05.cp would occupy the tensor pipe between MMAs)
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
    // A [M, rows_cap] and B [N, rows_cap] K-major, seg e = [offsets[e], offsets[e+1])
    int32_t wgrad;
    int64_t M;
    int32_t wgrad_tma;  // FP32 weight gradients stored through shared memory by TMA (the map in tmR)
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

// One stage's block scales, from shared memory to this warp's 32-lane quarter
// of the stage's tensor-memory slot (every quarter holds the same copy, as the
// block-scaled MMA reads it).  Shared memory holds the A tile [128 rows][16 B]
// and then the B tile's rows 0-127 and 128-255, each [128][16 B]; MMA-K chunk
// c of a row is its bytes 4c..4c+3.  Slot columns: A chunk c -> 4c..4c+3
// (column 4c+j holds row 32j+lane); B chunk c -> 16+8c+j, rows 32j+lane for
// j < 4 and 128+32(j-4)+lane for j >= 4.  The caller waits for the stores.
__device__ __forceinline__ void sf_stage_to_tmem(const uint8_t *sfs, uint32_t base, int lane) {
    {
        uint32_t r[16];  // A: column 4c + j
#pragma unroll
        for (int j = 0; j < 4; ++j) {
            const uint4 a = *reinterpret_cast<const uint4 *>(sfs + 16 * (lane + 32 * j));
            r[j] = a.x;
            r[4 + j] = a.y;
            r[8 + j] = a.z;
            r[12 + j] = a.w;
        }
        tmem_st16(base, r);
    }
    uint32_t rb[32];  // B: column 16 + 8c + j -> index 8c + j
#pragma unroll
    for (int j = 0; j < 8; ++j) {
        const uint4 w = *reinterpret_cast<const uint4 *>(sfs + kSFABytes + (j < 4 ? 0 : kSFBBytes / 2) +
                                                         16 * (lane + 32 * (j & 3)));
        rb[j] = w.x;
        rb[8 + j] = w.y;
        rb[16 + j] = w.z;
        rb[24 + j] = w.w;
    }
    tmem_st32(base + 16, rb);
}

// Launchers of the two pipelines (FP4: W4A4 + RAC; !FP4: BF16).  Tensor maps:
// A rows (box 128 rows), B rows (single: 256-row box for FP4, two 128-row
// boxes for BF16; pair: one 128-row box, this CTA's half), the RAC residual and
// the selected weight columns (single: 256-row box; pair: 128-row box).
template <bool FP4>
int launch_single_gemm(const CUtensorMap &tA, const CUtensorMap &tB, const CUtensorMap &tR, const CUtensorMap &tW,
                       const GemmParams &p, int64_t rows_cap, int64_t N, cudaStream_t stream);
template <bool FP4>
int launch_pair_gemm(const CUtensorMap &tA, const CUtensorMap &tB, const CUtensorMap &tR, const CUtensorMap &tW,
                     const GemmParams &p, int64_t rows_cap, int64_t N, cudaStream_t stream);

}  // namespace nvfp4
