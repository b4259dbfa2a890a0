// quantize.cu -- NVFP4 quantization kernels (HBM-bound).
//
// QUADS §2.2 "FP4.": E2M1 elements, one E4M3 scale per 16 consecutive
// elements, an FP32 per-tensor scale; §3.1 Eq. 9 / §3.3 Eq. 20-21: the
// activation quantizer Q_A and the RAC residual on a channel set S; §3.2
// Eq. 12: the weight fake-quantizer QDQ_W, which must round exactly like the
// rollout quantizer (both use quant_block below).
//
// Work split: one warp per (row, segment of 32 blocks); each lane owns one
// 16-element block (32 bytes of BF16 in, 8 bytes of codes out), so a warp
// reads 1 KB contiguous and writes 256 B of codes contiguous.  Four lanes
// pack their block scales into one 32-bit store of the swizzled layout.
#include <mutex>

#include "common.cuh"

namespace nvfp4 {

constexpr int kMaxBlocksPerRow = 1024;  // K <= 16384

enum QuantMode { kModeAct = 0, kModeWeight = 1 };

struct QuantArgs {
    const uint16_t *x;
    int64_t M, K, ldx, x_tstride;  // elements
    const float *amax;             // [ntensors]
    float *gs_out;                 // [ntensors] or null
    const int32_t *S;
    int32_t k;
    const int32_t *dst_row;
    int32_t fanout;
    int64_t rows_out;
    uint8_t *codes;
    int64_t codes_tstride;  // bytes
    uint8_t *scales;
    int64_t scales_tstride;  // bytes
    uint16_t *resid;         // act mode: [rows_out, k]
    uint16_t *wsel;          // weight mode: [rows, k] per tensor
    int64_t wsel_tstride;
    int32_t interleave;
    const int32_t *row_limit;  // act mode, or null: source rows at or past *row_limit are skipped
    int32_t *dev_status;
};

// Scale layout (activations and weights alike): tiles of 128 rows x 16 blocks
// (one 256-element GEMM K-slice), tile (m/128, kb/16) number
// (m/128)*kslices + kb/16, 2048 bytes each: four 512-byte groups, one per 4
// consecutive blocks (one MMA's 64 elements of K); in a group row r of the
// tile sits on line r%32 (16 bytes), its blocks at bytes 4*(r/32) + kb%4.  A
// group is what the GEMM copies into tensor memory with one 32x128b.warpx4
// tcgen05.cp (line l -> lane l of every lane quarter).  Four consecutive
// blocks kb..kb+3 (kb % 4 == 0) are four consecutive bytes, stored as one word.
__device__ __forceinline__ int64_t scale_row_offset(int64_t m, int64_t kslices) {
    return (m >> 7) * kslices * 2048 + (m & 31) * 16 + ((m & 127) >> 5) * 4;
}
__device__ __forceinline__ int64_t scale_block_offset(int64_t b) {  // b % 4 == 0
    return (b >> 4) * 2048 + ((b & 15) >> 2) * 512;
}

// E2M1 code -> value, from a packed table of 2*|value| (0,1,2,3,4,6,8,12).
__device__ __forceinline__ float e2m1_val(uint32_t c) {
    const float mag = 0.5f * (float)((0xC8643210u >> (4u * (c & 7u))) & 15u);
    return (c & 8u) ? -mag : mag;
}

// One 16-element block: the E4M3 scale code, its value, and the 16 E2M1 codes
// packed two per byte (element 2i in the low nibble) into two words.
struct BlockQ {
    uint32_t sb;
    float sbf;
    uint32_t w0, w1;
    __device__ __forceinline__ uint32_t code(int t) const { return ((t < 8 ? w0 : w1) >> (4 * (t & 7))) & 15u; }
};

// four pairs of binary32 values -> four E2M1 byte pairs in one word
__device__ __forceinline__ uint32_t e2m1x8(const float *q) {
    uint32_t w;
    asm("{ .reg .b8 b0, b1, b2, b3;\n"
        "cvt.rn.satfinite.e2m1x2.f32 b0, %2, %1;\n"
        "cvt.rn.satfinite.e2m1x2.f32 b1, %4, %3;\n"
        "cvt.rn.satfinite.e2m1x2.f32 b2, %6, %5;\n"
        "cvt.rn.satfinite.e2m1x2.f32 b3, %8, %7;\n"
        "mov.b32 %0, {b0, b1, b2, b3}; }"
        : "=r"(w)
        : "f"(q[0]), "f"(q[1]), "f"(q[2]), "f"(q[3]), "f"(q[4]), "f"(q[5]), "f"(q[6]), "f"(q[7]));
    return w;
}

// Four code pairs (a word of packed E2M1 codes, element 2i in the low nibble)
// -> their exact values as four f16x2 (element 2i in the low half).
__device__ __forceinline__ void e2m1x8_to_f16x2(uint32_t w, uint32_t &h0, uint32_t &h1, uint32_t &h2, uint32_t &h3) {
    asm("{ .reg .b8 b0, b1, b2, b3;\n"
        "mov.b32 {b0, b1, b2, b3}, %4;\n"
        "cvt.rn.f16x2.e2m1x2 %0, b0;\n"
        "cvt.rn.f16x2.e2m1x2 %1, b1;\n"
        "cvt.rn.f16x2.e2m1x2 %2, b2;\n"
        "cvt.rn.f16x2.e2m1x2 %3, b3; }"
        : "=r"(h0), "=r"(h1), "=r"(h2), "=r"(h3)
        : "r"(w));
}

// One E2M1 code (the low nibble of c) -> its exact value in binary32.
__device__ __forceinline__ float e2m1_to_f32_hw(uint32_t c) {
    float lo;
    asm("{ .reg .b8 b0, b1, b2, b3; .reg .b32 h; .reg .f16 l, u;\n"
        "mov.b32 {b0, b1, b2, b3}, %1;\n"
        "cvt.rn.f16x2.e2m1x2 h, b0;\n"
        "mov.b32 {l, u}, h; cvt.f32.f16 %0, l; }"
        : "=f"(lo)
        : "r"(c & 15u));
    return lo;
}

// f16x2 -> its two values in binary32 (exact), low half first.
__device__ __forceinline__ void f16x2_to_f32(uint32_t h, float &lo, float &hi) {
    asm("{ .reg .f16 l, u; mov.b32 {l, u}, %2; cvt.f32.f16 %0, l; cvt.f32.f16 %1, u; }" : "=f"(lo), "=f"(hi) : "r"(h));
}

// Two binary32 values -> BF16 (round to nearest even), lo in the low half.
__device__ __forceinline__ uint32_t bf16x2_rn(float lo, float hi) {
    uint32_t r;
    asm("cvt.rn.bf16x2.f32 %0, %2, %1;" : "=r"(r) : "f"(lo), "f"(hi));
    return r;
}

// (a0, a1) * (b0, b1) as two IEEE binary32 products (round to nearest) in one
// packed instruction.
__device__ __forceinline__ void fmul2_rn(float a0, float a1, float b0, float b1, float &r0, float &r1) {
    asm("{ .reg .b64 x, y, z; mov.b64 x, {%2, %3}; mov.b64 y, {%4, %5}; mul.rn.f32x2 z, x, y; mov.b64 {%0, %1}, z; }"
        : "=f"(r0), "=f"(r1)
        : "f"(a0), "f"(a1), "f"(b0), "f"(b1));
}

// (a0, a1) + (b0, b1), (a0, a1) - (b0, b1) and (a0, a1) * (b0, b1) + (c0, c1):
// two IEEE binary32 operations each (round to nearest), one packed instruction.
__device__ __forceinline__ void fadd2_rn(float a0, float a1, float b0, float b1, float &r0, float &r1) {
    asm("{ .reg .b64 x, y, z; mov.b64 x, {%2, %3}; mov.b64 y, {%4, %5}; add.rn.f32x2 z, x, y; mov.b64 {%0, %1}, z; }"
        : "=f"(r0), "=f"(r1)
        : "f"(a0), "f"(a1), "f"(b0), "f"(b1));
}
__device__ __forceinline__ void fsub2_rn(float a0, float a1, float b0, float b1, float &r0, float &r1) {
    asm("{ .reg .b64 x, y, z; mov.b64 x, {%2, %3}; mov.b64 y, {%4, %5}; sub.rn.f32x2 z, x, y; mov.b64 {%0, %1}, z; }"
        : "=f"(r0), "=f"(r1)
        : "f"(a0), "f"(a1), "f"(b0), "f"(b1));
}
__device__ __forceinline__ void ffma2_rn(float a0, float a1, float b0, float b1, float c0, float c1, float &r0,
                                         float &r1) {
    asm("{ .reg .b64 x, y, w, z; mov.b64 x, {%2, %3}; mov.b64 y, {%4, %5}; mov.b64 w, {%6, %7};\n"
        "fma.rn.f32x2 z, x, y, w; mov.b64 {%0, %1}, z; }"
        : "=f"(r0), "=f"(r1)
        : "f"(a0), "f"(a1), "f"(b0), "f"(b1), "f"(c0), "f"(c1));
}

// Per-block tables, filled once per CTA (gs is a power of two, so scaling by
// it commutes with rounding in the normal range):
//   div6[m] = fl((1 + m/128) / 6): fl(a / (6 gs)) = div6[mant7(a)] * 2^exp(a) / gs
//            for a BF16 block amax a (7 mantissa bits);
//   rcp[c]  = fl(1 / e4m3(c)):      fl(1 / (sb * gs)) = rcp[sb] / gs.
struct QTables {
    float div6[128];
    float rcp[128];
};

__device__ __forceinline__ void fill_tables(QTables &t) {
    for (int i = threadIdx.x; i < 128; i += blockDim.x) {
        t.div6[i] = __fdiv_rn(1.0f + (float)i * (1.0f / 128.0f), 6.0f);
        t.rcp[i] = __frcp_rn(e4m3_to_f32((uint32_t)i));
    }
}

// 2^n for |n| within the normal exponent range
__device__ __forceinline__ float pow2f(int n) { return __uint_as_float((uint32_t)(n + 127) << 23); }

__device__ __forceinline__ void quant_block(const float (&v)[16], float gs, float p6, float inv_gs,
                                            const QTables &tb, BlockQ &q) {
    float m8[8];  // the block amax as a tree of maxima (a short dependency chain)
#pragma unroll
    for (int t = 0; t < 8; ++t) m8[t] = fmaxf(fabsf(v[2 * t]), fabsf(v[2 * t + 1]));
#pragma unroll
    for (int t = 0; t < 4; ++t) m8[t] = fmaxf(m8[t], m8[t + 4]);
    const float amax_b = fmaxf(fmaxf(m8[0], m8[2]), fmaxf(m8[1], m8[3]));
    // block scale: E4M3 of fl(amax_b / (6*gs)), RNE with saturation
    const uint32_t ab = __float_as_uint(amax_b);
    const int ex = (int)(ab >> 23);  // biased exponent of the block amax
    float s;
    if (ex >= 8) s = __fmul_rn(__fmul_rn(tb.div6[(ab >> 16) & 127u], pow2f(ex - 127)), inv_gs);
    else s = __fdiv_rn(amax_b, p6);  // tiny or zero block amax: the plain division
    q.sb = e4m3_from_f32(s);
    q.sbf = e4m3_to_f32(q.sb);
    const float den = __fmul_rn(q.sbf, gs);
    if (den != 0.0f) {
        const float inv = __fmul_rn(tb.rcp[q.sb], inv_gs);  // = the correctly rounded 1/den
        float qv[16];
#pragma unroll
        for (int t = 0; t < 16; t += 2) fmul2_rn(v[t], v[t + 1], inv, inv, qv[t], qv[t + 1]);
        q.w0 = e2m1x8(qv);
        q.w1 = e2m1x8(qv + 8);
    } else {  // a zero block scale: signed zeros
        uint32_t w0 = 0, w1 = 0;
#pragma unroll
        for (int t = 0; t < 8; ++t) {
            w0 |= ((__float_as_uint(v[t]) >> 31) << 3) << (4 * t);
            w1 |= ((__float_as_uint(v[t + 8]) >> 31) << 3) << (4 * t);
        }
        q.w0 = w0;
        q.w1 = w1;
    }
}

__device__ __forceinline__ void unpack_block(const uint4 &a, const uint4 &b, float (&v)[16]) {
    const uint32_t w[8] = {a.x, a.y, a.z, a.w, b.x, b.y, b.z, b.w};
#pragma unroll
    for (int i = 0; i < 8; ++i) {
        v[2 * i] = __uint_as_float(w[i] << 16);
        v[2 * i + 1] = __uint_as_float(w[i] & 0xffff0000u);
    }
}

// The block's dequantized values (code * sb) * gs, both products in binary32,
// the code's exact value from the hardware conversion.
__device__ __forceinline__ void dequant_block_f32(const BlockQ &q, float gs, float (&d)[16]) {
    uint32_t h[8];
    e2m1x8_to_f16x2(q.w0, h[0], h[1], h[2], h[3]);
    e2m1x8_to_f16x2(q.w1, h[4], h[5], h[6], h[7]);
#pragma unroll
    for (int u = 0; u < 8; ++u) {
        float c0, c1;
        f16x2_to_f32(h[u], c0, c1);
        fmul2_rn(c0, c1, q.sbf, q.sbf, c0, c1);
        fmul2_rn(c0, c1, gs, gs, d[2 * u], d[2 * u + 1]);
    }
}

// The block's QDQ as BF16, two elements per word (element 2i in the low half).
__device__ __forceinline__ void dequant_block_bf16(const BlockQ &q, float gs, uint32_t (&o)[8]) {
    float d[16];
    dequant_block_f32(q, gs, d);
#pragma unroll
    for (int u = 0; u < 8; ++u) o[u] = bf16x2_rn(d[2 * u], d[2 * u + 1]);
}

constexpr int kQThreads = 256;
constexpr int kQWarps = kQThreads / 32;
constexpr int kMaxStagedK = 1024;  // residual row staged in shared memory up to this k
constexpr int kQSlots = 4;         // 1 KB segments in flight per warp
// Resident blocks per SM: 3 (24 warps, 96 KB of segments in flight per SM);
// 4 blocks of activations measured no faster.
template <int MODE>
constexpr int q_blocks_per_sm() {
    return 3;
}
// per warp: the staged RAC row (k <= kMaxStagedK) or, beyond it, the row's block scales
constexpr int kQRowBuf = 2 * kMaxStagedK > kMaxBlocksPerRow ? 2 * kMaxStagedK : kMaxBlocksPerRow;
constexpr size_t kQRingBytes = (size_t)kQWarps * kQSlots * 1024;
constexpr uint64_t kQWaitNs = 2000000000ull;  // 2 s per wait for a segment

// The RAC value of one selected element x (BF16 bits) of a block with scale
// code sb: its E2M1 code is recomputed exactly as the block's quantization
// computed it; activations give the residual bf16(x - (code*sb)*gs) in units
// of gs, weights the unscaled dequantized value bf16(code*sb).
template <int MODE>
__device__ __forceinline__ uint16_t resid_value(uint16_t xb, uint32_t sb, float gs, float inv_gs, const QTables &tb) {
    const float v = __uint_as_float((uint32_t)xb << 16);
    const float sbf = e4m3_to_f32(sb);
    uint32_t c;
    if (__fmul_rn(sbf, gs) != 0.0f) c = e2m1x2_from_f32(__fmul_rn(v, __fmul_rn(tb.rcp[sb], inv_gs)), 0.0f) & 15u;
    else c = (__float_as_uint(v) >> 31) << 3;
    const float cs = __fmul_rn(e2m1_val(c), sbf);  // exact
    if (MODE == kModeWeight) return __bfloat16_as_ushort(__float2bfloat16_rn(cs));
    const float r = __bfloat162float(__float2bfloat16_rn(__fsub_rn(v, __fmul_rn(cs, gs))));
    return __bfloat16_as_ushort(__float2bfloat16_rn(__fmul_rn(r, inv_gs)));
}

// The RAC value of element x (BF16 bits) already quantized to code c in a
// block of scale value sbf -- the value resid_value computes, from the code the
// block stored rather than a recomputed one.
template <int MODE>
__device__ __forceinline__ uint16_t rac_from_code(uint16_t xb, uint32_t c, float sbf, float gs, float inv_gs) {
    const float cs = __fmul_rn(e2m1_to_f32_hw(c), sbf);  // exact
    if (MODE == kModeWeight) return __bfloat16_as_ushort(__float2bfloat16_rn(cs));
    const float v = __uint_as_float((uint32_t)xb << 16);
    const float r = __bfloat162float(__float2bfloat16_rn(__fsub_rn(v, __fmul_rn(cs, gs))));
    return __bfloat16_as_ushort(__float2bfloat16_rn(__fmul_rn(r, inv_gs)));
}

// One warp per output row (grid-stride), the row in segments of 32 blocks
// (512 elements, one block per lane).  A warp's segments -- all of its rows',
// in order -- stream through a ring of kQSlots 1 KB slots in shared memory:
// lane 0 keeps kQSlots segments in flight with bulk copies (one mbarrier per
// slot), so the bytes in flight do not cost registers.  Each row's destination
// rows are resolved once: their code-row offsets and the row part of their
// scale offsets sit in shared memory, so a block's stores to every destination
// cost an add each.  The RAC values of a segment's selected channels are
// computed right after its blocks, one selected channel per lane (the lane
// reads the element from the slot and the block scale from the block's lane by
// a shuffle, then recomputes the element's code exactly as the block did);
// they are staged in shared memory and written once per destination row as
// 16-byte chunks.
template <int MODE>
__global__ void __launch_bounds__(kQThreads, q_blocks_per_sm<MODE>()) quantize_kernel(QuantArgs a) {
    extern __shared__ __align__(128) uint8_t q_ring[];  // [kQWarps][kQSlots][1024]
    __shared__ uint64_t s_qbar[kQWarps][kQSlots];
    __shared__ __align__(16) uint8_t s_row[kQWarps][kQRowBuf];
    __shared__ int64_t s_cbase[kQWarps][32];  // destination f: byte offset of its code row (-1: skipped)
    __shared__ int64_t s_sbase[kQWarps][32];  // destination f: row part of its scale offsets
    __shared__ int32_t s_dm[kQWarps][32];     // destination f: its row
    __shared__ int32_t s_S[kMaxStagedK];
    // per 512-element segment: the position in S of its first selected channel
    __shared__ int32_t s_segfirst[kMaxBlocksPerRow / 32 + 1];
    __shared__ QTables s_tab;
    const int tensor = blockIdx.y;
    fill_tables(s_tab);
    const int nb = (int)(a.K >> 4);
    const int64_t kslices = (nb + 15) >> 4;
    const bool has_sel = a.k > 0;
    const bool staged = a.k <= kMaxStagedK;
    const int segs = (nb + 31) >> 5;
    if (has_sel && staged) {
        for (int i = threadIdx.x; i < a.k; i += blockDim.x) s_S[i] = min(max(a.S[i], 0), (int32_t)(a.K - 1));
        __syncthreads();
        // S is increasing: the first position of segment s is the first i with S[i] >= 512 s
        for (int sg = threadIdx.x; sg <= segs; sg += blockDim.x) {
            int lo = 0, hi = a.k;
            while (lo < hi) {
                const int mid = (lo + hi) >> 1;
                if (s_S[mid] < 512 * sg) lo = mid + 1;
                else hi = mid;
            }
            s_segfirst[sg] = lo;
        }
    }
    __syncthreads();  // tables (and S) are ready

    const float amax_t = a.amax[tensor];
    const float gs = tensor_scale(amax_t);
    const float p6 = __fmul_rn(gs, 6.0f);
    const float inv_gs = __frcp_rn(gs);  // exact: gs is a power of two
    if (blockIdx.x == 0 && threadIdx.x == 0) {
        if (a.gs_out) a.gs_out[tensor] = gs;
        if (!isfinite(amax_t)) report(a.dev_status, NVFP4_ERR_NONFINITE);
    }

    const int lane = threadIdx.x & 31, wid = threadIdx.x >> 5;
    const int64_t nwarps_total = (int64_t)gridDim.x * kQWarps;
    const uint16_t *xt = a.x + (int64_t)tensor * a.x_tstride;
    uint16_t *stage = reinterpret_cast<uint16_t *>(s_row[wid]);  // staged: the RAC row
    uint8_t *row_sb = s_row[wid];                                 // not staged: the block scales
    const int fanout = (MODE == kModeAct) ? a.fanout : 1;
    uint8_t *codes = a.codes + (int64_t)tensor * a.codes_tstride;
    uint8_t *scales = a.scales + (int64_t)tensor * a.scales_tstride;

    // source row of output row m (weights may be stored in gate/up tile order)
    auto source_row = [&](int64_t m) -> int64_t {
        if (MODE == kModeWeight && a.interleave) {  // 256-row tiles: 128 gate rows, then 128 up rows
            const int64_t t = m >> 8, i = m & 255;
            return (i < 128) ? (t * 128 + i) : (a.M / 2 + t * 128 + (i - 128));
        }
        return m;
    };
    // This warp's rows m = first + i * nwarps_total (i < nrows) and their
    // segments, in order, flat index j; slot j % kQSlots of the warp's ring
    // holds segment j.  Lane 0 issues them ahead of the warp (position pm, pseg,
    // count pj); the warp consumes them at (m, seg), j.
    static_assert((kQSlots & (kQSlots - 1)) == 0, "slot index by mask");
    uint8_t *ring = q_ring + (size_t)wid * kQSlots * 1024;
    uint64_t *bars = s_qbar[wid];
    const int64_t first = (int64_t)blockIdx.x * kQWarps + wid;
    // source rows [0, Mq): all M, or those below the caller's device-side bound
    const int64_t Mq = a.row_limit ? min(a.M, (int64_t)max(__ldg(a.row_limit), 0)) : a.M;
    const int64_t nrows = first < Mq ? (Mq - 1 - first) / nwarps_total + 1 : 0;
    const int64_t nseg = nrows * segs;
    int64_t pm = first, pj = 0;
    int pseg = 0;
    auto issue_next = [&]() {  // lane 0: segment pj into its slot
        const int slot = (int)(pj & (kQSlots - 1));
        const uint32_t bytes = (uint32_t)min(32, nb - 32 * pseg) * 32u;
        mbar_arrive_expect_tx(&bars[slot], bytes);
        bulk_load(ring + slot * 1024, xt + source_row(pm) * a.ldx + (int64_t)pseg * 512, bytes, &bars[slot]);
        ++pj;
        if (++pseg == segs) {
            pseg = 0;
            pm += nwarps_total;
        }
    };
    if (lane == 0) {
        for (int sl = 0; sl < kQSlots; ++sl) mbar_init(&bars[sl], 1);
        fence_barrier_init();
        while (pj < nseg && pj < kQSlots) issue_next();
    }
    __syncwarp();
    int64_t j = 0, m = first;
    int seg = 0;
    bool ok = true;
    for (; j < nseg; ++j) {
        if (seg == 0) {
            // destination rows of this source row: lane f resolves the f-th
            __syncwarp();  // the previous row's readers of s_cbase / s_sbase are done
            if (lane < fanout) {
                int64_t dm = m;
                if (MODE == kModeAct && a.dst_row) dm = (int64_t)a.dst_row[m * fanout + lane];
                const bool okd = dm >= 0 && dm < ((MODE == kModeAct) ? a.rows_out : a.M);  // others are skipped
                s_cbase[wid][lane] = okd ? dm * (a.K >> 1) : -1;
                s_sbase[wid][lane] = okd ? scale_row_offset(dm, kslices) : 0;
                s_dm[wid][lane] = okd ? (int32_t)dm : 0;
            }
            __syncwarp();
        }
        const int slot = (int)(j & (kQSlots - 1));
        const bool got = mbar_wait_bounded(&bars[slot], (uint32_t)(j / kQSlots) & 1u, kQWaitNs);
        if (!__all_sync(0xffffffffu, got)) {
            ok = false;
            break;
        }
        const uint16_t *xs = reinterpret_cast<const uint16_t *>(ring + slot * 1024);  // the segment
        const int b = seg * 32 + lane;
        const bool valid = b < nb;
        float v[16];
        BlockQ q;
        if (valid) {
            unpack_block(*reinterpret_cast<const uint4 *>(xs + lane * 16),
                         *reinterpret_cast<const uint4 *>(xs + lane * 16 + 8), v);
            quant_block(v, gs, p6, inv_gs, s_tab, q);
        } else {
            q.sb = 0u;
            q.sbf = 0.0f;
            q.w0 = q.w1 = 0u;
        }

        {
            if (has_sel) {
                if (staged) {
                    // this segment's selected channels, one or two per lane per pass: the
                    // element from the slot, its code and block scale from the block's lane;
                    // the RAC value goes to the stage
                    const int i0 = s_segfirst[seg], i1 = s_segfirst[seg + 1];
                    for (int base = i0; base < i1; base += 64) {  // the same trip count in every lane
                        const int ia = base + lane, ib = base + 32 + lane;
                        const int ja = ia < i1 ? s_S[ia] : 0;
                        const uint16_t xa = ia < i1 ? xs[ja - seg * 512] : 0;
                        const int oa = (ja >> 4) & 31;
                        const uint32_t a0 = __shfl_sync(0xffffffffu, q.w0, oa), a1 = __shfl_sync(0xffffffffu, q.w1, oa);
                        const float fa = __shfl_sync(0xffffffffu, q.sbf, oa);
                        if (base + 32 < i1) {  // uniform: a second channel for some lanes
                            const int jb = ib < i1 ? s_S[ib] : 0;
                            const uint16_t xb = ib < i1 ? xs[jb - seg * 512] : 0;
                            const int ob = (jb >> 4) & 31;
                            const uint32_t b0 = __shfl_sync(0xffffffffu, q.w0, ob), b1 = __shfl_sync(0xffffffffu, q.w1, ob);
                            const float fb = __shfl_sync(0xffffffffu, q.sbf, ob);
                            if (ib < i1) {
                                const int tb = jb & 15;
                                stage[ib] = rac_from_code<MODE>(xb, ((tb < 8 ? b0 : b1) >> (4 * (tb & 7))) & 15u, fb, gs,
                                                                inv_gs);
                            }
                        }
                        if (ia < i1) {
                            const int ta = ja & 15;
                            stage[ia] = rac_from_code<MODE>(xa, ((ta < 8 ? a0 : a1) >> (4 * (ta & 7))) & 15u, fa, gs,
                                                            inv_gs);
                        }
                    }
                } else if (valid) {
                    row_sb[b] = (uint8_t)q.sb;
                }
            }
            // four consecutive blocks' scales -> one 32-bit word (lane%4 == 0 stores)
            uint32_t sw = q.sb;
            const uint32_t s1 = __shfl_down_sync(0xffffffffu, sw, 1);
            const uint32_t s2 = __shfl_down_sync(0xffffffffu, sw, 2);
            const uint32_t s3 = __shfl_down_sync(0xffffffffu, sw, 3);
            sw = sw | (s1 << 8) | (s2 << 16) | (s3 << 24);
            const bool group_lead = ((lane & 3) == 0) && (b < ((nb + 3) & ~3));
            const int64_t boff = scale_block_offset(b);  // block part of the scale offsets
            if (fanout == 1) {
                const int64_t cbase = s_cbase[wid][0];
                if (cbase >= 0) {
                    if (valid) *reinterpret_cast<uint2 *>(codes + cbase + b * 8) = make_uint2(q.w0, q.w1);
                    if (group_lead) *reinterpret_cast<uint32_t *>(scales + s_sbase[wid][0] + boff) = sw;
                }
            } else if (fanout <= 8) {
                // up to 8 destinations: every base read first, so one shared-memory
                // latency covers them all
                int64_t cb[8], sbb[8];
#pragma unroll
                for (int f = 0; f < 8; ++f) {
                    cb[f] = f < fanout ? s_cbase[wid][f] : -1;
                    sbb[f] = f < fanout ? s_sbase[wid][f] : 0;
                }
#pragma unroll
                for (int f = 0; f < 8; ++f) {
                    if (cb[f] < 0) continue;
                    if (valid) *reinterpret_cast<uint2 *>(codes + cb[f] + b * 8) = make_uint2(q.w0, q.w1);
                    if (group_lead) *reinterpret_cast<uint32_t *>(scales + sbb[f] + boff) = sw;
                }
            } else {
                for (int f = 0; f < fanout; ++f) {
                    const int64_t cbase = s_cbase[wid][f];
                    if (cbase < 0) continue;
                    if (valid) *reinterpret_cast<uint2 *>(codes + cbase + b * 8) = make_uint2(q.w0, q.w1);
                    if (group_lead) *reinterpret_cast<uint32_t *>(scales + s_sbase[wid][f] + boff) = sw;
                }
            }
        }
        __syncwarp();  // every lane is done with the slot (and, at a row's end, the stage is complete)
        if (lane == 0 && pj < nseg) issue_next();

        if (has_sel && seg == segs - 1) {
            // the row's residual (activation) or unscaled dequantized weight on S
            const uint16_t *xrow = xt + source_row(m) * a.ldx;
            if (!staged) {  // k beyond the stage: one selected channel per lane, straight to every destination
                for (int si = lane; si < a.k; si += 32) {
                    const int jc = __ldg(a.S + si);
                    const uint16_t val = resid_value<MODE>(__ldg(xrow + jc), row_sb[jc >> 4], gs, inv_gs, s_tab);
                    for (int f = 0; f < fanout; ++f) {
                        if (s_cbase[wid][f] < 0) continue;
                        const int64_t dm = s_dm[wid][f];
                        if (MODE == kModeWeight) a.wsel[(int64_t)tensor * a.wsel_tstride + dm * a.k + si] = val;
                        else a.resid[dm * a.k + si] = val;
                    }
                }
            } else {  // the row's k values -> every destination row
                const int chunks = a.k >> 3;  // 16-byte chunks (k % 8 == 0)
                const uint4 *src = reinterpret_cast<const uint4 *>(stage);
                for (int f = 0; f < fanout; ++f) {
                    if (s_cbase[wid][f] < 0) continue;
                    const int64_t dm = s_dm[wid][f];
                    uint16_t *row = (MODE == kModeWeight) ? a.wsel + (int64_t)tensor * a.wsel_tstride + dm * a.k
                                                          : a.resid + dm * a.k;
                    for (int c = lane; c < chunks; c += 32) reinterpret_cast<uint4 *>(row)[c] = src[c];
                }
            }
            __syncwarp();  // the stage is read out before the next row writes it
        }
        if (++seg == segs) {
            seg = 0;
            m += nwarps_total;
        }
    }
    if (!ok && lane == 0) {
        // a segment never arrived: report it, and let every copy still in flight land before the CTA exits
        report(a.dev_status, NVFP4_ERR_TIMEOUT);
        for (int64_t jj = j; jj < pj; ++jj)
            (void)mbar_wait_bounded(&bars[jj & (kQSlots - 1)], (uint32_t)(jj / kQSlots) & 1u, kQWaitNs);
    }
}

// max |x| per tensor: bit patterns of |bf16| compare like the values (NaN
// sorts above Inf, so it propagates).
__global__ void __launch_bounds__(256) amax_kernel(const uint16_t *x, int64_t M, int64_t K, int64_t ldx,
                                                   int64_t tstride, float *out) {
    const uint16_t *xt = x + (int64_t)blockIdx.y * tstride;
    uint32_t mx = 0u;
    const int64_t vec_per_row = K >> 3;
    const int64_t total = M * vec_per_row;
    const int64_t stride = (int64_t)gridDim.x * blockDim.x;
    int64_t i = (int64_t)blockIdx.x * blockDim.x + threadIdx.x;
    if (ldx == K) {
        const uint4 *p = reinterpret_cast<const uint4 *>(xt);
        for (; i + 7 * stride < total; i += 8 * stride) {  // eight 16-byte loads in flight per thread
            uint4 v[8];
#pragma unroll
            for (int u = 0; u < 8; ++u) v[u] = __ldg(p + i + u * stride);
#pragma unroll
            for (int u = 0; u < 8; ++u) {
                mx = __vmaxu2(mx, v[u].x & 0x7fff7fffu);
                mx = __vmaxu2(mx, v[u].y & 0x7fff7fffu);
                mx = __vmaxu2(mx, v[u].z & 0x7fff7fffu);
                mx = __vmaxu2(mx, v[u].w & 0x7fff7fffu);
            }
        }
        for (; i < total; i += stride) {
            uint4 v = __ldg(p + i);
            mx = __vmaxu2(mx, v.x & 0x7fff7fffu);
            mx = __vmaxu2(mx, v.y & 0x7fff7fffu);
            mx = __vmaxu2(mx, v.z & 0x7fff7fffu);
            mx = __vmaxu2(mx, v.w & 0x7fff7fffu);
        }
    } else {
        for (; i < total; i += stride) {
            int64_t r = i / vec_per_row, c = i - r * vec_per_row;
            uint4 v = __ldg(reinterpret_cast<const uint4 *>(xt + r * ldx) + c);
            mx = __vmaxu2(mx, v.x & 0x7fff7fffu);
            mx = __vmaxu2(mx, v.y & 0x7fff7fffu);
            mx = __vmaxu2(mx, v.z & 0x7fff7fffu);
            mx = __vmaxu2(mx, v.w & 0x7fff7fffu);
        }
    }
    uint32_t m16 = max(mx & 0xffffu, mx >> 16);
#pragma unroll
    for (int o = 16; o > 0; o >>= 1) m16 = max(m16, __shfl_xor_sync(0xffffffffu, m16, o));
    __shared__ uint32_t red[8];
    if ((threadIdx.x & 31) == 0) red[threadIdx.x >> 5] = m16;
    __syncthreads();
    if (threadIdx.x == 0) {
        uint32_t r = 0;
        for (int w = 0; w < (int)(blockDim.x >> 5); ++w) r = max(r, red[w]);
        atomicMax(reinterpret_cast<unsigned int *>(out + blockIdx.y), r << 16);
    }
}

// zero the padding rows of each expert segment of a routed NVFP4 activation
__global__ void clear_padding_kernel(const int32_t *counts, const int32_t *offsets, int64_t rows_cap, int64_t K,
                                     int32_t k, uint8_t *codes, uint8_t *scales, uint16_t *resid) {
    const int e = blockIdx.y;
    const int64_t r0 = (int64_t)offsets[e] + counts[e], r1 = offsets[e + 1];
    const int64_t row = r0 + blockIdx.x;
    if (row >= r1 || row >= rows_cap || row < 0) return;
    const int64_t nb = K >> 4, kslices = (nb + 15) >> 4;
    uint32_t *c = reinterpret_cast<uint32_t *>(codes + row * (K >> 1));
    for (int64_t i = threadIdx.x; i < (K >> 3); i += blockDim.x) c[i] = 0u;
    const int64_t srow = scale_row_offset(row, kslices);
    for (int64_t g = threadIdx.x; g < kslices * 4; g += blockDim.x)  // the row's 4-byte words, 4 per K-slice
        *reinterpret_cast<uint32_t *>(scales + srow + scale_block_offset(g * 4)) = 0u;
    if (resid)
        for (int64_t i = threadIdx.x; i < k; i += blockDim.x) resid[row * k + i] = 0;
}

// BF16 rows to routed order (QAT dispatch); padding rows zeroed
__global__ void scatter_rows_kernel(const uint16_t *x, int32_t T, int64_t K, int32_t topk, const int32_t *dst_row,
                                    int64_t rows_cap, uint16_t *y) {
    const int64_t t = blockIdx.x;
    const uint4 *src = reinterpret_cast<const uint4 *>(x + t * K);
    for (int64_t i = threadIdx.x; i < (K >> 3); i += blockDim.x) {
        uint4 v = __ldg(src + i);
        for (int s = 0; s < topk; ++s) {
            const int64_t r = dst_row[t * topk + s];
            if (r >= 0 && r < rows_cap) reinterpret_cast<uint4 *>(y + r * K)[i] = v;
        }
    }
}

__global__ void zero_pad_rows_kernel(const int32_t *counts, const int32_t *offsets, int64_t rows_cap, int64_t K,
                                     uint16_t *y) {
    const int e = blockIdx.y;
    const int64_t row = (int64_t)offsets[e] + counts[e] + blockIdx.x;
    if (row >= offsets[e + 1] || row >= rows_cap || row < 0) return;
    uint4 *d = reinterpret_cast<uint4 *>(y + row * K);
    for (int64_t i = threadIdx.x; i < (K >> 3); i += blockDim.x) d[i] = make_uint4(0, 0, 0, 0);
}

// Eq. 23 squared scores in binary64, each channel's sum taken in row order.
// A block owns 32 channels (one per lane); its 32 warps compute the squared
// quantization errors of 32 rows at a time into shared memory, then warp 0
// adds them to the channels' sums row by row, so every sum is the sequential
// one while the element work runs on all warps.
constexpr int kScoreWarps = 32;
__global__ void __launch_bounds__(32 * kScoreWarps) channel_score_kernel(const uint16_t *x, int64_t M, int64_t K,
                                                                         const float *amax, double *ssq) {
    __shared__ double sq[kScoreWarps][33];
    const int lane = threadIdx.x & 31, w = threadIdx.x >> 5;
    const int64_t j = (int64_t)blockIdx.x * 32 + lane;  // K % 16 == 0: a 16-lane block is all valid or all not
    const bool valid = j < K;
    const float gs = tensor_scale(amax[0]);
    const float p6 = __fmul_rn(gs, 6.0f);
    const double gsd = (double)gs;
    double acc = 0.0;
    for (int64_t i0 = 0; i0 < M; i0 += kScoreWarps) {
        const int64_t i = i0 + w;
        float v = (valid && i < M) ? __uint_as_float((uint32_t)x[i * K + j] << 16) : 0.0f;
        float am = fabsf(v);
#pragma unroll
        for (int o = 8; o > 0; o >>= 1) am = fmaxf(am, __shfl_xor_sync(0xffffffffu, am, o));
        const float sbf = e4m3_to_f32(e4m3_from_f32(__fdiv_rn(am, p6)));
        const float den = __fmul_rn(sbf, gs);
        uint32_t c;
        if (den != 0.0f) {
            const float qv = __fmul_rn(v, __frcp_rn(den));
            c = e2m1x2_from_f32(qv, qv) & 15u;
        } else {
            c = (__float_as_uint(v) >> 31) << 3;
        }
        const double xq = __dmul_rn((double)__fmul_rn(e2m1_to_f32(c), sbf), gsd);  // exact
        const double d = __dsub_rn(xq, (double)v);
        sq[w][lane] = __dmul_rn(d, d);
        __syncthreads();
        if (w == 0) {
            const int n = (M - i0 < kScoreWarps) ? (int)(M - i0) : kScoreWarps;
            for (int r = 0; r < n; ++r) acc = __dadd_rn(acc, sq[r][lane]);
        }
        __syncthreads();
    }
    if (w == 0 && valid) ssq[j] = acc;
}

// Eq. 24: keep the k largest (ties to the lower index), write them in order.
// Non-negative doubles order like their bit patterns.  Radix selection: the
// k-th largest key T is found 8 bits at a time with shared-memory histograms
// of the keys that share the bits found so far; then every channel with a key
// above T, and the first (k - #above) channels with key T in channel order,
// are written in channel order.  When the bucket that holds the k-th key holds
// exactly the keys still needed, every key in it is kept whatever its lower
// bits, so the search stops there (usually after two or three of the eight
// passes) and the channels whose bits down to that digit are at least T's are
// written -- the same set.
constexpr int kTopkPerThread = 16;  // keys per thread: K <= 16 * 1024
__global__ void __launch_bounds__(1024) select_topk_kernel(const double *ssq, int64_t K, int32_t k, int32_t *S) {
    __shared__ uint32_t hist[256];
    __shared__ int32_t warp_a[32], warp_b[32];
    __shared__ unsigned long long s_prefix;
    __shared__ int32_t s_need, carry_eq, carry_out, s_stop;
    const unsigned long long *key = reinterpret_cast<const unsigned long long *>(ssq);
    // the keys stay in registers for all passes: key j = threadIdx.x + i * blockDim.x
    unsigned long long kv[kTopkPerThread];
#pragma unroll
    for (int i = 0; i < kTopkPerThread; ++i) {
        const int64_t j = threadIdx.x + (int64_t)i * blockDim.x;
        kv[i] = j < K ? key[j] : 0ull;
    }
    if (threadIdx.x == 0) {
        s_prefix = 0ull;
        s_need = k;  // rank of T among the keys that share the prefix, counted from the top
        carry_eq = 0;
        carry_out = 0;
        s_stop = -1;  // the digit's shift once the bucket of the k-th key is kept whole
    }
    const int lane = threadIdx.x & 31, wid = threadIdx.x >> 5, nw = (int)(blockDim.x >> 5);
    for (int shift = 56; shift >= 0; shift -= 8) {
        for (int b = threadIdx.x; b < 256; b += blockDim.x) hist[b] = 0u;
        __syncthreads();
        const unsigned long long hi = shift == 56 ? 0ull : (~0ull << (shift + 8));
        const unsigned long long prefix = s_prefix;
        // warp-aggregated counts: the keys of a warp that fall in one bucket add once
#pragma unroll
        for (int i = 0; i < kTopkPerThread; ++i) {
            const int64_t j0 = (int64_t)i * blockDim.x;
            if (j0 >= K) break;  // the same in every thread
            const int64_t j = j0 + threadIdx.x;
            const unsigned long long v = kv[i];
            const bool act = j < K && (v & hi) == prefix;
            const uint32_t bucket = act ? (uint32_t)((v >> shift) & 255u) : 256u + (uint32_t)lane;
            const unsigned peers = __match_any_sync(0xffffffffu, bucket);
            if (act && lane == __ffs(peers) - 1) atomicAdd(&hist[bucket], (uint32_t)__popc(peers));
        }
        __syncthreads();
        if (wid == 0) {
            // lane l holds buckets 255-8l down to 248-8l; find the bucket of rank s_need from the top
            uint32_t h[8], tot = 0;
#pragma unroll
            for (int i = 0; i < 8; ++i) {
                h[i] = hist[255 - 8 * lane - i];
                tot += h[i];
            }
            uint32_t incl = tot;
#pragma unroll
            for (int o = 1; o < 32; o <<= 1) {
                const uint32_t t = __shfl_up_sync(0xffffffffu, incl, o);
                if (lane >= o) incl += t;
            }
            const int32_t need = s_need;
            const unsigned hit = __ballot_sync(0xffffffffu, (int32_t)incl >= need);
            if (lane == __ffs(hit) - 1) {
                int32_t cum = (int32_t)(incl - tot);
                for (int i = 0; i < 8; ++i) {
                    if (cum + (int32_t)h[i] >= need) {
                        s_prefix = prefix | ((unsigned long long)(255 - 8 * lane - i) << shift);
                        s_need = need - cum;
                        if (cum + (int32_t)h[i] == need) s_stop = shift;
                        break;
                    }
                    cum += (int32_t)h[i];
                }
            }
        }
        __syncthreads();
        if (s_stop >= 0) break;  // the same in every thread
    }
    const unsigned long long T = s_prefix;
    const int32_t need_eq = s_need;  // keys equal to T to keep, lowest channels first
    const int stop = s_stop;
#pragma unroll
    for (int i = 0; i < kTopkPerThread; ++i) {
        const int64_t j0 = (int64_t)i * blockDim.x;
        if (j0 >= K) break;  // the same in every thread
        const int64_t j = j0 + threadIdx.x;
        const unsigned long long v = kv[i];
        const int eq = stop < 0 && j < K && v == T;
        // rank of this channel among the equal keys, in channel order
        const unsigned be = __ballot_sync(0xffffffffu, eq);
        if (lane == 0) warp_a[wid] = __popc(be);
        __syncthreads();
        int pre_eq = carry_eq + __popc(be & ((1u << lane) - 1u));
        for (int w = 0; w < wid; ++w) pre_eq += warp_a[w];
        const int flag = j < K && (stop >= 0 ? (v >> stop) >= (T >> stop) : (v > T || (eq && pre_eq < need_eq)));
        const unsigned bf = __ballot_sync(0xffffffffu, flag);
        if (lane == 0) warp_b[wid] = __popc(bf);
        __syncthreads();
        int pos = carry_out + __popc(bf & ((1u << lane) - 1u));
        for (int w = 0; w < wid; ++w) pos += warp_b[w];
        if (flag) S[pos] = (int32_t)j;
        __syncthreads();
        if (threadIdx.x == 0) {
            for (int w = 0; w < nw; ++w) {
                carry_eq += warp_a[w];
                carry_out += warp_b[w];
            }
        }
        __syncthreads();
    }
}

// ---- literal second-pass RAC residual (QUADS §3.3 Eq. 21): the BF16 residual
// that quantize_kernel stored for the routed rows [0, offsets[E]) is itself
// NVFP4-quantized -- 16-element blocks along the gathered channel axis, a
// tensor scale of its own -- and replaced in place by its dequantized value
// (exact in BF16: a grid value times an E4M3 scale has at most 6 significant
// bits, and the tensor scale is a power of two).  Rows past offsets[E] are
// left alone, so stale rows of an earlier, larger batch cannot reach the amax.
__device__ __forceinline__ int64_t resid_rows(int64_t rows_cap, const int32_t *offsets, int32_t E) {
    if (!offsets) return rows_cap;
    const int64_t r = offsets[E];
    return r < 0 ? 0 : (r > rows_cap ? rows_cap : r);
}

__global__ void __launch_bounds__(256) resid_amax_kernel(const uint16_t *resid, int64_t rows_cap, int32_t k,
                                                        const int32_t *offsets, int32_t E, float *out) {
    const int64_t total = resid_rows(rows_cap, offsets, E) * (k >> 3);  // 8 BF16 per 16-byte load
    const uint4 *p = reinterpret_cast<const uint4 *>(resid);
    uint32_t mx = 0u;
    for (int64_t i = (int64_t)blockIdx.x * blockDim.x + threadIdx.x; i < total; i += (int64_t)gridDim.x * blockDim.x) {
        const uint4 v = __ldg(p + i);
        mx = __vmaxu2(mx, v.x & 0x7fff7fffu);
        mx = __vmaxu2(mx, v.y & 0x7fff7fffu);
        mx = __vmaxu2(mx, v.z & 0x7fff7fffu);
        mx = __vmaxu2(mx, v.w & 0x7fff7fffu);
    }
    uint32_t m16 = max(mx & 0xffffu, mx >> 16);
#pragma unroll
    for (int o = 16; o > 0; o >>= 1) m16 = max(m16, __shfl_xor_sync(0xffffffffu, m16, o));
    __shared__ uint32_t red[8];
    if ((threadIdx.x & 31) == 0) red[threadIdx.x >> 5] = m16;
    __syncthreads();
    if (threadIdx.x == 0) {
        uint32_t r = 0;
        for (int w = 0; w < (int)(blockDim.x >> 5); ++w) r = max(r, red[w]);
        atomicMax(reinterpret_cast<unsigned int *>(out), r << 16);
    }
}

__global__ void __launch_bounds__(256) resid_qdq_kernel(uint16_t *resid, int64_t rows_cap, int32_t k,
                                                       const int32_t *offsets, int32_t E, const float *amax,
                                                       float *gs_out, int32_t *dev_status) {
    __shared__ QTables tb;
    fill_tables(tb);
    __syncthreads();
    const float am = *amax;
    if (!isfinite(am)) {
        if (blockIdx.x == 0 && threadIdx.x == 0) report(dev_status, NVFP4_ERR_NONFINITE);
        return;
    }
    const float gs = tensor_scale(am);
    const float p6 = __fmul_rn(gs, 6.0f);
    const float inv_gs = __frcp_rn(gs);  // exact: gs is a power of two
    if (gs_out && blockIdx.x == 0 && threadIdx.x == 0) *gs_out = gs;
    const int64_t nblk = resid_rows(rows_cap, offsets, E) * (k >> 4);
    uint4 *p = reinterpret_cast<uint4 *>(resid);
    for (int64_t b = (int64_t)blockIdx.x * blockDim.x + threadIdx.x; b < nblk; b += (int64_t)gridDim.x * blockDim.x) {
        float v[16];
        unpack_block(p[2 * b], p[2 * b + 1], v);
        BlockQ q;
        quant_block(v, gs, p6, inv_gs, tb, q);
        uint32_t o[8];
        dequant_block_bf16(q, gs, o);
        p[2 * b] = make_uint4(o[0], o[1], o[2], o[3]);
        p[2 * b + 1] = make_uint4(o[4], o[5], o[6], o[7]);
    }
}

// ---- online per-forward channel selection (QUADS §3.3 Eq. 23-24 on the
// batch at hand).  Scores of the rows [0, offsets[E]) (all rows_cap rows when
// offsets is null): a (row chunk, 512-column segment) per block, one 16-element
// block per lane as the quantizer sees it, 8 warps striding over the chunk's
// rows.  The squared error of an element, (code*sb*gs - x)^2, is exact in
// binary32 (both terms have few significant bits and lie within a factor of a
// block scale of each other); a lane adds four rows' squared errors of each of
// its 16 channels in binary32 and the four-row partials into compensated
// binary32 sums, the warps' sums are added in binary64 in warp order, and the
// chunks' in chunk order -- deterministic, within a few ulp of binary32 of the
// exact sums (all terms are nonnegative).
constexpr int kOnlineChunks = 256;  // row chunks of the score pass, at most
// Row chunks of the score pass: one wave of blocks (two resident per SM) over the
// (chunk, 512-column segment) grid, so that no partial last wave idles the GPU; at
// least 512 rows per chunk when the rows are few.
static int64_t online_chunks(int64_t rows_cap, int64_t K) {
    const int64_t colblocks = (K + 511) / 512;
    int64_t c = (int64_t)sm_count() * 2 / colblocks;
    const int64_t by_rows = (rows_cap + 511) / 512;
    if (c > by_rows) c = by_rows;
    return c < 1 ? 1 : (c > kOnlineChunks ? kOnlineChunks : c);
}

__global__ void __launch_bounds__(256) online_score_kernel(const uint16_t *x, int64_t rows_cap, int64_t K,
                                                          const int32_t *offsets, int32_t E, const float *amax,
                                                          double *part) {
    const int64_t nchunks = gridDim.x;
    __shared__ QTables tb;
    __shared__ double red[8][512];
    fill_tables(tb);
    __syncthreads();
    const float gs = tensor_scale(*amax);
    const float p6 = __fmul_rn(gs, 6.0f);
    const float inv_gs = __frcp_rn(gs);
    const int64_t rows = resid_rows(rows_cap, offsets, E);
    const int c = blockIdx.x, lane = threadIdx.x & 31, w = threadIdx.x >> 5;
    const int64_t r0 = rows * c / nchunks, r1 = rows * (c + 1) / nchunks;
    const int64_t col = (int64_t)blockIdx.y * 512 + 16 * lane;  // this lane's block
    const bool valid = col < K;
    float sum[16], comp[16];
#pragma unroll
    for (int t = 0; t < 16; ++t) sum[t] = comp[t] = 0.0f;
    if (valid) {
        // four rows' loads in flight per warp (rows r, r+8, r+16, r+24), added in row order
        for (int64_t rb = r0 + w; rb < r1; rb += 32) {
            uint4 raw[4][2];
#pragma unroll
            for (int u = 0; u < 4; ++u) {
                const int64_t r = rb + 8 * u;
                if (r < r1) {
                    const uint4 *p = reinterpret_cast<const uint4 *>(x + r * K + col);
                    raw[u][0] = __ldg(p);
                    raw[u][1] = __ldg(p + 1);
                } else {
                    raw[u][0] = raw[u][1] = make_uint4(0, 0, 0, 0);  // adds exact zeros
                }
            }
            // the four rows' squared errors in binary32 (a sum of four nonnegative terms, within
            // 3 ulp), then that partial into the compensated sum
            float pz[16];
#pragma unroll
            for (int t = 0; t < 16; ++t) pz[t] = 0.0f;
#pragma unroll
            for (int u = 0; u < 4; ++u) {
                float v[16];
                unpack_block(raw[u][0], raw[u][1], v);
                BlockQ q;
                quant_block(v, gs, p6, inv_gs, tb, q);
                float dq[16];
                dequant_block_f32(q, gs, dq);
#pragma unroll
                for (int t = 0; t < 16; t += 2) {  // d = dq - v, pz += d * d (pairs of channels)
                    float d0, d1;
                    fsub2_rn(dq[t], dq[t + 1], v[t], v[t + 1], d0, d1);
                    ffma2_rn(d0, d1, d0, d1, pz[t], pz[t + 1], pz[t], pz[t + 1]);
                }
            }
#pragma unroll
            for (int t = 0; t < 16; t += 2) {  // compensated sum += pz
                float y0, y1, s0, s1, e0, e1;
                fsub2_rn(pz[t], pz[t + 1], comp[t], comp[t + 1], y0, y1);
                fadd2_rn(sum[t], sum[t + 1], y0, y1, s0, s1);
                fsub2_rn(s0, s1, sum[t], sum[t + 1], e0, e1);
                fsub2_rn(e0, e1, y0, y1, comp[t], comp[t + 1]);
                sum[t] = s0;
                sum[t + 1] = s1;
            }
        }
    }
#pragma unroll
    for (int t = 0; t < 16; ++t) red[w][16 * lane + t] = (double)sum[t] - (double)comp[t];
    __syncthreads();
    for (int i = threadIdx.x; i < 512; i += blockDim.x) {
        const int64_t j = (int64_t)blockIdx.y * 512 + i;
        if (j >= K) continue;
        double acc = 0.0;
        for (int ww = 0; ww < 8; ++ww) acc = __dadd_rn(acc, red[ww][i]);
        part[(int64_t)c * K + j] = acc;
    }
}

// ssq[j] = the sum over chunks of part[c, j]: a block per 32 channels, warp w
// adding chunks w, w + 8, ... in order (eight loads in flight), then the
// warps' sums in warp order.
__global__ void __launch_bounds__(256) online_score_finish_kernel(const double *part, int64_t K, int nchunks,
                                                                  double *ssq) {
    __shared__ double red[8][32];
    const int lane = threadIdx.x & 31, w = threadIdx.x >> 5;
    const int64_t j = (int64_t)blockIdx.x * 32 + lane;
    double acc = 0.0;
    if (j < K) {
        for (int c0 = w; c0 < nchunks; c0 += 64) {
            double v[8];
#pragma unroll
            for (int u = 0; u < 8; ++u) v[u] = c0 + 8 * u < nchunks ? __ldg(part + (int64_t)(c0 + 8 * u) * K + j) : 0.0;
#pragma unroll
            for (int u = 0; u < 8; ++u) acc = __dadd_rn(acc, v[u]);
        }
    }
    red[w][lane] = acc;
    __syncthreads();
    if (w == 0 && j < K) {
        double sum = 0.0;
        for (int i = 0; i < 8; ++i) sum = __dadd_rn(sum, red[i][lane]);
        ssq[j] = sum;
    }
}

// W_sel[e, n, s] = bf16(code * sb) of packed weight element (n, S[s]) of
// expert e -- the unscaled dequantized value nvfp4_prepare_weights stores for
// the channels S -- gathered for a new S.  A block covers one 128-row tile of
// one expert (blockIdx.x, blockIdx.y); its block scales (the tile's 512-byte
// scale groups) and its rows' packed codes arrive by bulk copies -- the scale
// groups once, each 16 bytes further along the banks than the last, the rows
// through a ring of kGatherSlots row slots per warp.  A warp takes 16 rows; a
// lane emits channels 4l + 128u .. 4l + 128u + 3 of each.  A row's scale
// words (4 blocks each) are all in one bank of a scale group, so lane g reads
// word g of the row once (the skew spreads the groups over 8 banks) and the
// lanes that need a block take its word by shuffle.
constexpr int kGatherWarps = 8;
constexpr int kGatherSlots = 4;                     // rows in flight per warp
constexpr int kGatherRowsPerWarp = 128 / kGatherWarps;
constexpr int kGatherGroupPitch = 512 + 16;         // a scale group's place in shared memory
constexpr uint64_t kGatherWaitNs = 2000000000ull;  // 2 s per wait

__host__ __device__ constexpr int64_t gather_groups(int64_t K) { return ((K / 16 + 15) / 16) * 4; }
__host__ __device__ constexpr int64_t gather_smem_bytes(int64_t K, int32_t k) {
    return gather_groups(K) * kGatherGroupPitch + (int64_t)kGatherWarps * kGatherSlots * (K / 2) +
           (((int64_t)k * 4 + 15) / 16) * 16;
}

__global__ void __launch_bounds__(32 * kGatherWarps) gather_wsel_kernel(const uint8_t *codes, const uint8_t *scales,
                                                                      int64_t N, int64_t K, const int32_t *S,
                                                                      int32_t k, uint16_t *wsel, int32_t *dev_status) {
    extern __shared__ __align__(128) uint8_t gsm[];
    __shared__ uint64_t s_bar[1 + kGatherWarps * kGatherSlots];
    const int lane = threadIdx.x & 31, w = threadIdx.x >> 5;
    const int64_t e = blockIdx.y, tile = blockIdx.x;
    const int ngroups = (int)gather_groups(K);  // 512-byte scale groups of the tile: 4 per 256-element K-slice
    const uint32_t rowb = (uint32_t)(K / 2);
    uint8_t *s_sc = gsm;                                                 // the scale groups, skewed
    uint8_t *ring = gsm + (size_t)ngroups * kGatherGroupPitch + (size_t)w * kGatherSlots * rowb;
    int32_t *s_S = reinterpret_cast<int32_t *>(gsm + (size_t)ngroups * kGatherGroupPitch +
                                               (size_t)kGatherWarps * kGatherSlots * rowb);
    uint64_t *bars = s_bar + 1 + w * kGatherSlots;
    if (threadIdx.x == 0) {
        for (int i = 0; i < 1 + kGatherWarps * kGatherSlots; ++i) mbar_init(&s_bar[i], 1);
        fence_barrier_init();
    }
    __syncthreads();  // the barriers are ready
    const int64_t n0 = tile * 128 + (int64_t)w * kGatherRowsPerWarp;  // this warp's first row
    const uint8_t *crow = codes + (e * N + n0) * rowb;
    if (w == 0) {  // the scale groups, issued by the 32 lanes of warp 0
        const uint8_t *src = scales + (e * (N / 128) + tile) * (int64_t)ngroups * 512;
        if (lane == 0) mbar_arrive_expect_tx(&s_bar[0], (uint32_t)ngroups * 512u);
        __syncwarp();
        for (int g = lane; g < ngroups; g += 32) bulk_load(s_sc + g * kGatherGroupPitch, src + g * 512, 512u, &s_bar[0]);
    }
    if (lane == 0)
        for (int i = 0; i < kGatherSlots; ++i) {
            mbar_arrive_expect_tx(&bars[i], rowb);
            bulk_load(ring + (size_t)i * rowb, crow + (size_t)i * rowb, rowb, &bars[i]);
        }
    for (int i = threadIdx.x; i < k; i += blockDim.x) s_S[i] = min(max(S[i], 0), (int32_t)(K - 1));
    __syncthreads();  // S is ready
    // channels 4 lane .. 4 lane + 3 (k <= 128 in one pass; more come from shared memory per row)
    int cb[4], csh[4], wl[4], wb[4];
#pragma unroll
    for (int t = 0; t < 4; ++t) {
        const int j = 4 * lane + t < k ? s_S[4 * lane + t] : 0;
        cb[t] = j >> 1;             // the code byte
        csh[t] = 4 * (j & 1);       // its nibble
        wl[t] = j >> 6;             // the lane holding its block's scale word
        wb[t] = 8 * ((j >> 4) & 3); // the scale byte in that word
    }
    bool ok = __all_sync(0xffffffffu, mbar_wait_bounded(&s_bar[0], 0u, kGatherWaitNs));
    int i = 0;
    for (; ok && i < kGatherRowsPerWarp; ++i) {
        const int slot = i % kGatherSlots;
        if (!__all_sync(0xffffffffu, mbar_wait_bounded(&bars[slot], (uint32_t)(i / kGatherSlots) & 1u, kGatherWaitNs))) {
            ok = false;
            break;
        }
        const uint8_t *rc = ring + (size_t)slot * rowb;
        const int64_t n = n0 + i;
        const int srow = (int)((n & 31) * 16 + ((n & 127) >> 5) * 4);  // the row's word in each scale group
        uint16_t *out = wsel + (e * N + n) * k;
        for (int s0 = 0; s0 < k; s0 += 128) {
            uint32_t sw = 0u;  // lane g: the row's scale word of group g, then of group 32 + g, ...
            uint32_t h[4];
            for (int g0 = 0; g0 < ngroups; g0 += 32) {
                if (g0 + lane < ngroups)
                    sw = *reinterpret_cast<const uint32_t *>(s_sc + (g0 + lane) * kGatherGroupPitch + srow);
#pragma unroll
                for (int t = 0; t < 4; ++t) {
                    int j = 0, cbt = cb[t], csht = csh[t], wlt = wl[t], wbt = wb[t];
                    if (s0 > 0) {  // channels past the first 128: from shared memory
                        j = s0 + 4 * lane + t < k ? s_S[s0 + 4 * lane + t] : 0;
                        cbt = j >> 1;
                        csht = 4 * (j & 1);
                        wlt = j >> 6;
                        wbt = 8 * ((j >> 4) & 3);
                    }
                    const uint32_t word = __shfl_sync(0xffffffffu, sw, wlt & 31);
                    if ((wlt >> 5) == (g0 >> 5)) {
                        const uint32_t c = (rc[cbt] >> csht) & 15u;
                        const uint32_t sb = (word >> wbt) & 0xffu;
                        h[t] = __bfloat16_as_ushort(__float2bfloat16_rn(__fmul_rn(e2m1_to_f32_hw(c), e4m3_to_f32(sb))));
                    }
                }
            }
            if (s0 + 4 * lane < k)
                *reinterpret_cast<uint2 *>(out + s0 + 4 * lane) = make_uint2(h[0] | (h[1] << 16), h[2] | (h[3] << 16));
        }
        __syncwarp();  // every lane is done with the slot
        if (lane == 0 && i + kGatherSlots < kGatherRowsPerWarp) {
            mbar_arrive_expect_tx(&bars[slot], rowb);
            bulk_load(ring + (size_t)slot * rowb, crow + (size_t)(i + kGatherSlots) * rowb, rowb, &bars[slot]);
        }
    }
    if (!ok && lane == 0) {
        // a copy never arrived: report it, and let every copy still in flight land before the block exits
        report(dev_status, NVFP4_ERR_TIMEOUT);
        for (int ii = i; ii < kGatherRowsPerWarp && ii < i + kGatherSlots; ++ii)
            (void)mbar_wait_bounded(&bars[ii % kGatherSlots], (uint32_t)(ii / kGatherSlots) & 1u, kGatherWaitNs);
        if (w == 0) (void)mbar_wait_bounded(&s_bar[0], 0u, kGatherWaitNs);
    }
}

// The same gather reading the code and scale bytes straight from global
// memory (only the sectors that hold selected channels are read): a block
// covers 32 rows of one expert (blockIdx.y), a warp 4 of them, the 4 rows'
// loads all issued before the first is used.  For rows of 4096 channels and
// more this beats the staged kernel (whose 128-row blocks wait for 32 KB of
// scales before the first row); for shorter rows the staged one wins.
constexpr int kGatherDirectRows = 4;  // rows per warp
__global__ void __launch_bounds__(32 * kGatherWarps) gather_wsel_direct_kernel(const uint8_t *codes,
                                                                             const uint8_t *scales, int64_t N,
                                                                             int64_t K, const int32_t *S, int32_t k,
                                                                             uint16_t *wsel) {
    const int lane = threadIdx.x & 31, w = threadIdx.x >> 5;
    const int64_t e = blockIdx.y;
    const int64_t n0 = ((int64_t)blockIdx.x * kGatherWarps + w) * kGatherDirectRows;  // N % 128 == 0: all rows exist
    const int64_t nb = K >> 4, kslices = (nb + 15) >> 4;
    const uint8_t *sten = scales + e * (N >> 7) * kslices * 2048;  // the expert's scales
    const uint8_t *cten = codes + e * N * (K >> 1);
    for (int s0 = 4 * lane; s0 < k; s0 += 128) {  // k % 8 == 0: channels s0 .. s0 + 3 all exist
        int32_t co[4];
        uint32_t sh[4];
        int64_t so[4];
#pragma unroll
        for (int t = 0; t < 4; ++t) {
            const int32_t j = min(max(__ldg(S + s0 + t), 0), (int32_t)(K - 1));
            co[t] = j >> 1;
            sh[t] = 4u * (uint32_t)(j & 1);
            so[t] = scale_block_offset(j >> 4) + ((j >> 4) & 3);
        }
        uint32_t cv[kGatherDirectRows][4], sv[kGatherDirectRows][4];
#pragma unroll
        for (int r = 0; r < kGatherDirectRows; ++r) {
            const uint8_t *crow = cten + (n0 + r) * (K >> 1);
            const uint8_t *srow = sten + scale_row_offset(n0 + r, kslices);
#pragma unroll
            for (int t = 0; t < 4; ++t) {
                cv[r][t] = __ldg(crow + co[t]);
                sv[r][t] = __ldg(srow + so[t]);
            }
        }
#pragma unroll
        for (int r = 0; r < kGatherDirectRows; ++r) {
            uint32_t h[4];
#pragma unroll
            for (int t = 0; t < 4; ++t)
                h[t] = __bfloat16_as_ushort(
                    __float2bfloat16_rn(__fmul_rn(e2m1_to_f32_hw((cv[r][t] >> sh[t]) & 15u), e4m3_to_f32(sv[r][t]))));
            *reinterpret_cast<uint2 *>(wsel + (e * N + n0 + r) * k + s0) = make_uint2(h[0] | (h[1] << 16), h[2] | (h[3] << 16));
        }
    }
}

// Channel-major copy of a weight pack, for the online gather: per expert e,
// codes_t[e][j][n/2] holds channel j of rows n and n+1 (row n in the low
// nibble) and scales_t[e][kb][n] the block scale of row n, block kb.  A block
// transposes a 64-row x 64-channel tile of codes through shared memory (one
// code per byte there) and the matching 64 x 4 block scales.
__global__ void __launch_bounds__(256) pack_transpose_kernel(const uint8_t *codes, const uint8_t *scales, int64_t N,
                                                             int64_t K, uint8_t *codes_t, uint8_t *scales_t) {
    __shared__ uint8_t tile[64][64 + 4];  // [row][channel]
    const int64_t e = blockIdx.z, n0 = (int64_t)blockIdx.y * 64, j0 = (int64_t)blockIdx.x * 64;
    const int64_t nb = K >> 4, kslices = (nb + 15) >> 4;
    const uint8_t *ce = codes + e * N * (K >> 1);
    // read: 64 rows x 32 bytes (64 channels), 8 bytes per thread
    {
        const int r = threadIdx.x >> 2, q = threadIdx.x & 3;  // row, 8-byte quarter
        const uint2 v = *reinterpret_cast<const uint2 *>(ce + (n0 + r) * (K >> 1) + (j0 >> 1) + 8 * q);
        const uint32_t w[2] = {v.x, v.y};
#pragma unroll
        for (int b = 0; b < 8; ++b) {
            const uint32_t byte = (w[b >> 2] >> (8 * (b & 3))) & 0xffu;
            tile[r][16 * q + 2 * b] = (uint8_t)(byte & 15u);
            tile[r][16 * q + 2 * b + 1] = (uint8_t)(byte >> 4);
        }
    }
    __syncthreads();
    // write: 64 channels x 32 bytes (64 rows, two per byte), 8 bytes per thread
    {
        const int c = threadIdx.x >> 2, q = threadIdx.x & 3;  // channel, 8-byte quarter of the rows
        uint32_t w[2] = {0u, 0u};
#pragma unroll
        for (int b = 0; b < 8; ++b) {
            const int r = 16 * q + 2 * b;
            w[b >> 2] |= ((uint32_t)tile[r][c] | ((uint32_t)tile[r + 1][c] << 4)) << (8 * (b & 3));
        }
        *reinterpret_cast<uint2 *>(codes_t + (e * K + j0 + c) * (N >> 1) + (n0 >> 1) + 8 * q) = make_uint2(w[0], w[1]);
    }
    // the tile's 4 blocks of scales (K % 64 == 0: all of them exist): scales_t[e][kb][n0 .. n0 + 64),
    // one byte per thread
    {
        const int kb = (int)(j0 >> 4) + (threadIdx.x >> 6), r = threadIdx.x & 63;
        const int64_t n = n0 + r;
        const uint8_t *se = scales + e * (N >> 7) * kslices * 2048;
        scales_t[(e * nb + kb) * N + n] = se[scale_row_offset(n, kslices) + scale_block_offset(kb & ~3) + (kb & 3)];
    }
}

// w_sel[e, n, s] from the channel-major pack: a block covers 128 rows x 64
// selected channels of one expert; thread (s, quarter) reads the 32 rows'
// codes of channel S[s] (16 bytes) and their 32 block scales, writes the 32
// values into a shared tile, and the tile leaves as 128-byte row pieces.  The
// tile's 16-byte column groups are swizzled by the row's quarter (group g of
// row r sits at g ^ (r / 32)), so the four quarters' writes of one column fall
// in different banks.
__global__ void __launch_bounds__(256) gather_wsel_t_kernel(const uint8_t *codes_t, const uint8_t *scales_t, int64_t N,
                                                           int64_t K, const int32_t *S, int32_t k, uint16_t *wsel) {
    __shared__ __align__(16) uint16_t tile[128][64];  // [row][selected channel, groups swizzled]
    const int64_t e = blockIdx.z, n0 = (int64_t)blockIdx.y * 128;
    const int s0 = blockIdx.x * 64;
    const int64_t nb = K >> 4;
    {
        const int sl = threadIdx.x >> 2, q = threadIdx.x & 3;  // channel in the tile, 32-row quarter
        const int s = s0 + sl;
        if (s < k) {
            const int32_t j = min(max(__ldg(S + s), 0), (int32_t)(K - 1));
            const uint4 c = __ldg(reinterpret_cast<const uint4 *>(codes_t + (e * K + j) * (N >> 1) + (n0 >> 1)) + q);
            const uint8_t *sc = scales_t + (e * nb + (j >> 4)) * N + n0 + 32 * q;
            const uint4 s_lo = __ldg(reinterpret_cast<const uint4 *>(sc)), s_hi = __ldg(reinterpret_cast<const uint4 *>(sc) + 1);
            const uint32_t cw[4] = {c.x, c.y, c.z, c.w};
            const uint32_t sw[8] = {s_lo.x, s_lo.y, s_lo.z, s_lo.w, s_hi.x, s_hi.y, s_hi.z, s_hi.w};
            const int col = sl ^ (8 * q);  // this channel's column in the swizzled rows of quarter q
#pragma unroll
            for (int i = 0; i < 32; ++i) {
                const uint32_t code = (cw[i >> 3] >> (4 * (i & 7))) & 15u;
                const uint32_t sb = (sw[i >> 2] >> (8 * (i & 3))) & 0xffu;
                tile[32 * q + i][col] =
                    __bfloat16_as_ushort(__float2bfloat16_rn(__fmul_rn(e2m1_to_f32_hw(code), e4m3_to_f32(sb))));
            }
        }
    }
    __syncthreads();
    // 128 rows x (up to) 64 channels = 128 bytes per row: 8 lanes x 16 bytes per row
    const int nsel = min(64, k - s0);
    for (int i = threadIdx.x; i < 128 * 8; i += blockDim.x) {
        const int r = i >> 3, p = i & 7;
        if (8 * p < nsel) {  // k % 8 == 0: whole 16-byte pieces
            const uint4 v = *reinterpret_cast<const uint4 *>(&tile[r][8 * (p ^ (r >> 5))]);
            *reinterpret_cast<uint4 *>(wsel + (e * N + n0 + r) * k + s0 + 8 * p) = v;
        }
    }
}

// QDQ_W (QUADS §3.2 Eq. 12) that also writes the transpose, for the learner's
// backward (dX = W_hat^T dY needs W_hat^T with the reduction axis contiguous):
// a block owns a 64 x 64 tile of one tensor; each thread quantizes one
// 16-element block exactly as fake_quant_fused_kernel does (quant_block, the
// tensor's gs), writes it to w_hat, and leaves it in shared memory; the tile
// then leaves transposed, 16 bytes per thread.
__global__ void __launch_bounds__(256) fake_quant_t_kernel(const uint16_t *w, int64_t rows, int64_t cols,
                                                          const float *amax, float *gs_out, uint16_t *w_hat,
                                                          uint16_t *w_hat_t, int32_t *dev_status) {
    __shared__ QTables tb;
    __shared__ uint32_t tile[64][33];  // 64 rows x 64 BF16 (two per word) + 1 word of pad
    fill_tables(tb);
    __syncthreads();
    const int64_t tensor = blockIdx.z;
    const float am = amax[tensor];
    const float gs = tensor_scale(am);
    const float p6 = __fmul_rn(gs, 6.0f);
    const float inv_gs = __frcp_rn(gs);
    if (blockIdx.x == 0 && blockIdx.y == 0 && threadIdx.x == 0) {
        if (gs_out) gs_out[tensor] = gs;
        if (!isfinite(am)) report(dev_status, NVFP4_ERR_NONFINITE);
    }
    const int64_t off = tensor * rows * cols;
    const int64_t r0 = (int64_t)blockIdx.y * 64, c0 = (int64_t)blockIdx.x * 64;
    {
        const int r = threadIdx.x >> 2, b = threadIdx.x & 3;  // row in the tile, 16-element block
        const int64_t gi = off + (r0 + r) * cols + c0 + 16 * b;
        const uint4 *src = reinterpret_cast<const uint4 *>(w + gi);
        float v[16];
        unpack_block(__ldg(src), __ldg(src + 1), v);
        BlockQ q;
        quant_block(v, gs, p6, inv_gs, tb, q);
        uint32_t o[8];
        dequant_block_bf16(q, gs, o);
        uint4 *dst = reinterpret_cast<uint4 *>(w_hat + gi);
        dst[0] = make_uint4(o[0], o[1], o[2], o[3]);
        dst[1] = make_uint4(o[4], o[5], o[6], o[7]);
#pragma unroll
        for (int i = 0; i < 8; ++i) tile[r][8 * b + i] = o[i];
    }
    __syncthreads();
    // w_hat_t[tensor][c][r]: output row c0 + cc holds input rows r0 .. r0+63; a thread writes
    // 8 consecutive of them (16 bytes), two such pieces per thread
#pragma unroll
    for (int k = 0; k < 2; ++k) {
        const int idx = threadIdx.x + 256 * k;  // 64 output rows x 8 pieces
        const int cc = idx >> 3, piece = idx & 7;
        uint32_t o[4];
#pragma unroll
        for (int u = 0; u < 4; ++u) {
            const int ra = 8 * piece + 2 * u;
            const uint32_t a0 = tile[ra][cc >> 1], a1 = tile[ra + 1][cc >> 1];
            const uint32_t lo = (cc & 1) ? (a0 >> 16) : (a0 & 0xffffu);
            const uint32_t hi = (cc & 1) ? (a1 >> 16) : (a1 & 0xffffu);
            o[u] = lo | (hi << 16);
        }
        *reinterpret_cast<uint4 *>(w_hat_t + off + (c0 + cc) * rows + r0 + 8 * piece) = make_uint4(o[0], o[1], o[2], o[3]);
    }
}

// Blocks for `rows` rows (one warp per row): as many as are resident at once.
template <int MODE>
static int quant_grid(int64_t rows) {
    int64_t blocks = (rows + kQWarps - 1) / kQWarps;
    int64_t cap = (int64_t)sm_count() * q_blocks_per_sm<MODE>();
    if (blocks > cap) blocks = cap;
    return (int)(blocks < 1 ? 1 : blocks);
}

// The segment ring is dynamic shared memory above the static arrays.
template <int MODE>
static int launch_quantize(dim3 grid, const QuantArgs &a, cudaStream_t st, const char *name) {
    static bool attr_done = false;
    if (!attr_done) {
        const cudaError_t e =
            cudaFuncSetAttribute(quantize_kernel<MODE>, cudaFuncAttributeMaxDynamicSharedMemorySize, (int)kQRingBytes);
        if (e != cudaSuccess) {
            set_last_error("cudaFuncSetAttribute(quantize_kernel)", e);
            return NVFP4_ERR_CUDA;
        }
        attr_done = true;
    }
    quantize_kernel<MODE><<<grid, kQThreads, kQRingBytes, st>>>(a);
    return launch_status(name);
}

// QDQ_W of many weight tensors (QUADS §3.2 Eq. 12) in one persistent launch
// that reads every tensor from HBM once: its amax and its quantize-dequantize
// are two kinds of work items of `rpi` rows, taken from one counter in the
// order A(0), A(1), B(0), A(2), B(1), ..., B(nt-1) -- A(t) the amax of tensor
// t, B(t) its QDQ -- so that B(t) re-reads rows that A(t) read shortly before
// and that still sit in L2.  A B(t) item starts once every A(t) item has
// added its maximum (a per-tensor count of finished A items, waited on with a
// bound); no A item ever waits, and every A(t) item is taken before any B(t)
// item, so the wait always ends.  Scratch (32-bit words, zeroed by the
// caller's stream before the launch): amax[nt], done[nt], the work counter.
// Items are kept near 64 KB (rpi a multiple of 8 rows, at least 8) so that
// the items in flight at once -- one per resident block -- span only about
// two tensors, whose rows then fit in L2 between their two reads.
constexpr int kFQItemBytes = 65536;
__host__ __device__ constexpr int64_t fq_rows_per_item(int64_t cols) {
    const int64_t r = (kFQItemBytes / 2 / (cols > 0 ? cols : 1) + 4) / 8 * 8;
    return r < 8 ? 8 : r;
}
constexpr uint64_t kFQWaitNs = 2000000000ull;

// 16-byte global load / store with an L2 eviction-priority policy (createpolicy):
// the amax pass keeps a tensor's lines in L2 for the second read, which then
// lets them go, as does the output stream.
__device__ __forceinline__ uint64_t l2_policy_evict_last() {
    uint64_t pol;
    asm volatile("createpolicy.fractional.L2::evict_last.b64 %0, 1.0;" : "=l"(pol));
    return pol;
}
__device__ __forceinline__ uint64_t l2_policy_evict_first() {
    uint64_t pol;
    asm volatile("createpolicy.fractional.L2::evict_first.b64 %0, 1.0;" : "=l"(pol));
    return pol;
}
__device__ __forceinline__ uint4 ld_hint(const uint4 *p, uint64_t pol) {
    uint4 v;
    asm volatile("ld.global.nc.L2::cache_hint.v4.u32 {%0, %1, %2, %3}, [%4], %5;"
                 : "=r"(v.x), "=r"(v.y), "=r"(v.z), "=r"(v.w)
                 : "l"(p), "l"(pol));
    return v;
}
__device__ __forceinline__ void st_hint(uint4 *p, const uint4 &v, uint64_t pol) {
    asm volatile("st.global.L2::cache_hint.v4.u32 [%0], {%1, %2, %3, %4}, %5;" ::"l"(p), "r"(v.x), "r"(v.y), "r"(v.z),
                 "r"(v.w), "l"(pol)
                 : "memory");
}

struct FQArgs {
    const uint16_t *w;
    uint16_t *w_hat;
    int64_t rows, cols;
    int32_t nt, per;  // tensors, items per tensor and kind
    int32_t rpi;      // rows per item (a multiple of 8)
    uint32_t *ws;     // amax bits [nt], done [nt], counter
    float *gs_out;
    int32_t *dev_status;
};

__global__ void __launch_bounds__(256, 4) fake_quant_fused_kernel(FQArgs a) {
    __shared__ QTables tb;
    __shared__ int64_t s_next[2];  // the item after the current one, by iteration parity
    __shared__ uint32_t s_red[8];
    __shared__ int s_ok;
    fill_tables(tb);
    const int lane = threadIdx.x & 31, wid = threadIdx.x >> 5;
    const int64_t total = 2ll * a.nt * a.per;
    const int nb = (int)(a.cols >> 4), segs = (nb + 31) >> 5;
    uint32_t *amax_bits = a.ws, *done = a.ws + a.nt, *counter = a.ws + 2 * a.nt;
    const uint64_t keep = l2_policy_evict_last(), drop = l2_policy_evict_first();
    if (threadIdx.x == 0) s_next[0] = (int64_t)atomicAdd(counter, 1u);
    __syncthreads();  // the first item, and the tables, are ready
    int64_t item = s_next[0];
    for (int iter = 0; item < total; ++iter) {
        // group gi: 0 -> A(0); 2nt-1 -> B(nt-1); odd -> A((gi+1)/2); even -> B(gi/2 - 1)
        const int64_t gi = (int64_t)((uint32_t)item / (uint32_t)a.per);  // items fit in 32 bits
        const int chunk = (int)(item - gi * a.per);
        const bool is_a = gi == 0 || (gi != 2ll * a.nt - 1 && (gi & 1));
        const int t = gi == 0 ? 0 : (gi == 2ll * a.nt - 1 ? a.nt - 1 : (int)((gi & 1) ? (gi + 1) / 2 : gi / 2 - 1));
        const int64_t r0 = (int64_t)chunk * a.rpi;
        const int64_t r1 = min(a.rows, r0 + (int64_t)a.rpi);
        const uint16_t *wt = a.w + (int64_t)t * a.rows * a.cols;
        if (is_a) {
            // max |w| of the rows: bit patterns of |bf16| order like the values (NaN above Inf)
            const uint4 *p = reinterpret_cast<const uint4 *>(wt + r0 * a.cols);
            const int64_t nvec = (r1 - r0) * (a.cols >> 3);
            uint32_t mx = 0u;
            int64_t i = threadIdx.x;
            for (; i + 7 * 256 < nvec; i += 8 * 256) {  // eight 16-byte loads in flight per thread
                uint4 v[8];
#pragma unroll
                for (int u = 0; u < 8; ++u) v[u] = ld_hint(p + i + 256 * u, keep);
#pragma unroll
                for (int u = 0; u < 8; ++u) {
                    mx = __vmaxu2(mx, v[u].x & 0x7fff7fffu);
                    mx = __vmaxu2(mx, v[u].y & 0x7fff7fffu);
                    mx = __vmaxu2(mx, v[u].z & 0x7fff7fffu);
                    mx = __vmaxu2(mx, v[u].w & 0x7fff7fffu);
                }
            }
            for (; i < nvec; i += 256) {
                const uint4 v = ld_hint(p + i, keep);
                mx = __vmaxu2(mx, v.x & 0x7fff7fffu);
                mx = __vmaxu2(mx, v.y & 0x7fff7fffu);
                mx = __vmaxu2(mx, v.z & 0x7fff7fffu);
                mx = __vmaxu2(mx, v.w & 0x7fff7fffu);
            }
            uint32_t m16 = max(mx & 0xffffu, mx >> 16);
#pragma unroll
            for (int o = 16; o > 0; o >>= 1) m16 = max(m16, __shfl_xor_sync(0xffffffffu, m16, o));
            if (lane == 0) s_red[wid] = m16;
            __syncthreads();
            if (threadIdx.x == 0) {
                uint32_t r = 0u;
                for (int q = 0; q < 8; ++q) r = max(r, s_red[q]);
                atomicMax(amax_bits + t, r << 16);
                __threadfence();  // the maximum is visible before the item counts as done
                atomicAdd(done + t, 1u);
            }
        } else {
            // B(t): this warp's rows r0 + wid + 8 i (i < nrw), their segments in order; the
            // loads run two segments ahead, across row ends.  The weights are inputs, so the
            // first loads go out before the wait for the tensor's amax.
            const int nrw = r1 - r0 > wid ? (int)((r1 - r0 - wid + 7) >> 3) : 0;
            auto load = [&](int i, int sg, uint4 &x0, uint4 &x1) {
                const int b = sg * 32 + lane;
                if (i < nrw && b < nb) {
                    const uint4 *p = reinterpret_cast<const uint4 *>(wt + (r0 + wid + 8 * i) * a.cols + b * 16);
                    x0 = ld_hint(p, drop);
                    x1 = ld_hint(p + 1, drop);
                }
            };
            int li = 0, lsg = 0;  // the next segment to load
            auto step = [&](int &i, int &sg) {
                if (++sg == segs) {
                    sg = 0;
                    ++i;
                }
            };
            uint4 n0a = make_uint4(0, 0, 0, 0), n0b = n0a, n1a = n0a, n1b = n0a;
            load(li, lsg, n0a, n0b);
            step(li, lsg);
            load(li, lsg, n1a, n1b);
            step(li, lsg);
            // wait for every A(t) item
            if (threadIdx.x == 0) {
                const volatile uint32_t *d = done + t;
                bool ok = *d >= (uint32_t)a.per;
                const uint64_t t0 = global_ns();
                while (!ok) {
                    __nanosleep(200);
                    ok = *d >= (uint32_t)a.per;
                    if (!ok && global_ns() - t0 > kFQWaitNs) break;
                }
                __threadfence();
                s_ok = ok;
                if (!ok) report(a.dev_status, NVFP4_ERR_TIMEOUT);
            }
            __syncthreads();
            if (s_ok) {
                const float amax_t = __uint_as_float(*(const volatile uint32_t *)(amax_bits + t));
                const float gs = tensor_scale(amax_t);
                const float p6 = __fmul_rn(gs, 6.0f);
                const float inv_gs = __frcp_rn(gs);
                if (chunk == 0 && threadIdx.x == 0) {
                    if (a.gs_out) a.gs_out[t] = gs;
                    if (!isfinite(amax_t)) report(a.dev_status, NVFP4_ERR_NONFINITE);
                }
                uint16_t *ot = a.w_hat + (int64_t)t * a.rows * a.cols;
                for (int ci = 0, csg = 0; ci < nrw; step(ci, csg)) {
                    const uint4 ca = n0a, cb = n0b;
                    n0a = n1a;
                    n0b = n1b;
                    load(li, lsg, n1a, n1b);
                    step(li, lsg);
                    const int b = csg * 32 + lane;
                    if (b < nb) {
                        float v[16];
                        BlockQ q;
                        unpack_block(ca, cb, v);
                        quant_block(v, gs, p6, inv_gs, tb, q);
                        uint32_t o[8];
                        dequant_block_bf16(q, gs, o);
                        uint4 *dst = reinterpret_cast<uint4 *>(ot + (r0 + wid + 8 * ci) * a.cols + b * 16);
                        st_hint(dst, make_uint4(o[0], o[1], o[2], o[3]), drop);
                        st_hint(dst + 1, make_uint4(o[4], o[5], o[6], o[7]), drop);
                    }
                }
            }
        }
        // thread 0 takes the next item once its own share is done, so the counter's round trip
        // overlaps the other warps' tail (s_next by parity: every thread read the other slot
        // before this iteration's barriers)
        if (threadIdx.x == 0) s_next[(iter + 1) & 1] = (int64_t)atomicAdd(counter, 1u);
        __syncthreads();  // the item is done: s_next is visible, s_red and s_ok may be rewritten
        item = s_next[(iter + 1) & 1];
    }
}

static int amax_launch(const void *x, int64_t M, int64_t K, int64_t ldx, int32_t nt, int64_t tstride, float *out,
                       cudaStream_t st) {
    cudaError_t e = cudaMemsetAsync(out, 0, sizeof(float) * (size_t)nt, st);
    if (e != cudaSuccess) {
        set_last_error("cudaMemsetAsync(amax)", e);
        return NVFP4_ERR_CUDA;
    }
    if (M == 0 || K == 0) return NVFP4_OK;
    int64_t vecs = M * (K / 8);
    int64_t blocks = (vecs + 255) / 256;
    int64_t cap = (int64_t)sm_count() * 8 / (nt > 8 ? 8 : (nt < 1 ? 1 : nt));
    if (cap < 1) cap = 1;
    if (blocks > cap) blocks = cap;
    amax_kernel<<<dim3((unsigned)blocks, (unsigned)nt), 256, 0, st>>>((const uint16_t *)x, M, K, ldx, tstride, out);
    return launch_status("amax_kernel");
}

}  // namespace nvfp4

using namespace nvfp4;

extern "C" int nvfp4_amax(const void *x, int64_t M, int64_t K, int64_t ldx, int32_t ntensors, int64_t tensor_stride,
                          float *amax_out, void *stream) {
    if (missing(x, M * K) || !amax_out || M < 0 || K < 0 || ldx < K || ntensors < 1 || tensor_stride < 0)
        return NVFP4_ERR_INVALID_ARG;
    if (ntensors > 65535) return NVFP4_ERR_UNSUPPORTED;
    if (K % 8) return NVFP4_ERR_UNSUPPORTED;
    if (!aligned16(x) || ldx % 8 || tensor_stride % 8) return NVFP4_ERR_ALIGNMENT;
    NVFP4_CHECK_INIT();
    return amax_launch(x, M, K, ldx, ntensors, tensor_stride, amax_out, (cudaStream_t)stream);
}

extern "C" int nvfp4_quantize(const void *x, int64_t M, int64_t K, int64_t ldx, const float *amax, float *gs_out,
                              const int32_t *S, int32_t k, const int32_t *dst_row, int32_t fanout, int64_t rows_out,
                              uint8_t *codes, uint8_t *scales, void *resid, const int32_t *row_limit,
                              int32_t *dev_status, void *stream) {
    if (missing(x, M * K) || !amax || missing(codes, rows_out * K) || missing(scales, rows_out * K) || M < 0 || K < 0 ||
        ldx < K || k < 0 || k > K || fanout < 1)
        return NVFP4_ERR_INVALID_ARG;
    if (k > 0 && (!S || missing(resid, rows_out))) return NVFP4_ERR_INVALID_ARG;
    if (!dst_row && M > 0 && (fanout != 1 || rows_out < M)) return NVFP4_ERR_INVALID_ARG;
    // a row's destinations are resolved into 32 per-warp slots
    if (K % 32 || k % 8 || K / 16 > kMaxBlocksPerRow || fanout > 32 || M > INT32_MAX || rows_out > INT32_MAX)
        return NVFP4_ERR_UNSUPPORTED;
    if (!aligned16(x) || ldx % 8 || !aligned16(codes) || !aligned16(scales) || (resid && !aligned16(resid)))
        return NVFP4_ERR_ALIGNMENT;
    if (M == 0) return NVFP4_OK;
    NVFP4_CHECK_INIT();
    QuantArgs a{};
    a.x = (const uint16_t *)x;
    a.M = M;
    a.K = K;
    a.ldx = ldx;
    a.amax = amax;
    a.gs_out = gs_out;
    a.S = S;
    a.k = k;
    a.dst_row = dst_row;
    a.fanout = fanout;
    a.rows_out = rows_out;
    a.codes = codes;
    a.scales = scales;
    a.resid = (uint16_t *)resid;
    a.row_limit = row_limit;
    a.dev_status = dev_status;
    return launch_quantize<kModeAct>(dim3(quant_grid<kModeAct>(M)), a, (cudaStream_t)stream, "quantize_kernel");
}

extern "C" int nvfp4_fake_quant(const void *w, int32_t nt, int64_t rows, int64_t cols, void *w_hat, float *gs_out,
                                float *amax_ws, int32_t *dev_status, void *stream) {
    if (!w || !w_hat || !amax_ws || nt < 1 || rows < 0 || cols < 0) return NVFP4_ERR_INVALID_ARG;
    // items are counted in 32 bits
    const int64_t rpi = fq_rows_per_item(cols);
    if (cols % 32 || cols / 16 > kMaxBlocksPerRow || nt > 65535 || 2 * (int64_t)nt * ((rows + rpi - 1) / rpi) > (1ll << 31))
        return NVFP4_ERR_UNSUPPORTED;
    if (!aligned16(w) || !aligned16(w_hat)) return NVFP4_ERR_ALIGNMENT;
    NVFP4_CHECK_INIT();
    cudaStream_t st = (cudaStream_t)stream;
    // scratch: amax[nt], done[nt], the work counter -- all start at zero
    const cudaError_t e = cudaMemsetAsync(amax_ws, 0, sizeof(float) * (2 * (size_t)nt + 1), st);
    if (e != cudaSuccess) {
        set_last_error("cudaMemsetAsync(fake-quant scratch)", e);
        return NVFP4_ERR_CUDA;
    }
    if (rows == 0 || cols == 0) return NVFP4_OK;
    FQArgs a{};
    a.w = (const uint16_t *)w;
    a.w_hat = (uint16_t *)w_hat;
    a.rows = rows;
    a.cols = cols;
    a.nt = nt;
    a.per = (int32_t)((rows + rpi - 1) / rpi);
    a.rpi = (int32_t)rpi;
    a.ws = reinterpret_cast<uint32_t *>(amax_ws);
    a.gs_out = gs_out;
    a.dev_status = dev_status;
    const int64_t items = 2ll * nt * a.per;
    int64_t grid = (int64_t)sm_count() * 4;
    if (grid > items) grid = items;
    fake_quant_fused_kernel<<<(unsigned)grid, 256, 0, st>>>(a);
    return launch_status("fake_quant_fused_kernel");
}

extern "C" int nvfp4_fake_quant_transposed(const void *w, int32_t nt, int64_t rows, int64_t cols, void *w_hat,
                                           void *w_hat_t, float *gs_out, float *amax_ws, int32_t *dev_status,
                                           void *stream) {
    if (!w || !w_hat || !w_hat_t || !amax_ws || nt < 1 || rows < 0 || cols < 0) return NVFP4_ERR_INVALID_ARG;
    if (rows % 64 || cols % 64 || nt > 65535 || rows / 64 > 65535) return NVFP4_ERR_UNSUPPORTED;
    if (!aligned16(w) || !aligned16(w_hat) || !aligned16(w_hat_t)) return NVFP4_ERR_ALIGNMENT;
    NVFP4_CHECK_INIT();
    cudaStream_t st = (cudaStream_t)stream;
    int s = amax_launch(w, rows, cols, cols, nt, rows * cols, amax_ws, st);
    if (s != NVFP4_OK || rows == 0 || cols == 0) return s;
    fake_quant_t_kernel<<<dim3((unsigned)(cols / 64), (unsigned)(rows / 64), (unsigned)nt), 256, 0, st>>>(
        (const uint16_t *)w, rows, cols, amax_ws, gs_out, (uint16_t *)w_hat, (uint16_t *)w_hat_t, dev_status);
    return launch_status("fake_quant_t_kernel");
}

extern "C" int nvfp4_prepare_weights(const void *w, int32_t E, int64_t N, int64_t K, const int32_t *S, int32_t k,
                                     int32_t interleave, uint8_t *w_codes, uint8_t *w_scales, float *gs_w,
                                     void *w_sel, float *amax_ws, int32_t *dev_status, void *stream) {
    if (!w || !w_codes || !w_scales || !gs_w || !amax_ws || E < 1 || N < 0 || K < 0 || k < 0 || k > K)
        return NVFP4_ERR_INVALID_ARG;
    if (k > 0 && (!S || !w_sel)) return NVFP4_ERR_INVALID_ARG;
    if (K % 64 || N % 128 || (interleave && N % 256) || k % 8 || K / 16 > kMaxBlocksPerRow || E > 65535 || N > INT32_MAX)
        return NVFP4_ERR_UNSUPPORTED;
    if (!aligned16(w) || !aligned16(w_codes) || !aligned16(w_scales) || (w_sel && !aligned16(w_sel)))
        return NVFP4_ERR_ALIGNMENT;
    NVFP4_CHECK_INIT();
    cudaStream_t st = (cudaStream_t)stream;
    int s = amax_launch(w, N, K, K, E, N * K, amax_ws, st);
    if (s != NVFP4_OK || N == 0) return s;
    QuantArgs a{};
    a.x = (const uint16_t *)w;
    a.M = N;
    a.K = K;
    a.ldx = K;
    a.x_tstride = N * K;
    a.amax = amax_ws;
    a.gs_out = gs_w;
    a.S = S;
    a.k = k;
    a.fanout = 1;
    a.codes = w_codes;
    a.codes_tstride = N * K / 2;
    a.scales = w_scales;
    a.scales_tstride = N * ((K / 16 + 15) / 16) * 16;  // an expert's scales
    a.wsel = (uint16_t *)w_sel;
    a.wsel_tstride = N * (int64_t)k;
    a.interleave = interleave;
    a.dev_status = dev_status;
    int g = quant_grid<kModeWeight>(N) / (E > 8 ? 8 : E);
    return launch_quantize<kModeWeight>(dim3(g < 1 ? 1 : g, E), a, st, "quantize_kernel<weight>");
}

extern "C" int nvfp4_rac_requant_residual(void *resid, int64_t rows_cap, int32_t k, const int32_t *offsets, int32_t E,
                                          float *amax_ws, float *gs_out, int32_t *dev_status, void *stream) {
    if (!resid || !amax_ws || rows_cap < 0 || k < 0 || (offsets && E < 1)) return NVFP4_ERR_INVALID_ARG;
    if (k % 16) return NVFP4_ERR_UNSUPPORTED;
    if (!aligned16(resid)) return NVFP4_ERR_ALIGNMENT;
    NVFP4_CHECK_INIT();
    cudaStream_t st = (cudaStream_t)stream;
    const cudaError_t e = cudaMemsetAsync(amax_ws, 0, sizeof(float), st);
    if (e != cudaSuccess) {
        set_last_error("cudaMemsetAsync(residual amax)", e);
        return NVFP4_ERR_CUDA;
    }
    if (rows_cap == 0 || k == 0) return NVFP4_OK;
    // sized for all rows_cap rows; the kernels stop at offsets[E]
    int64_t blocks = (rows_cap * (k / 8) + 255) / 256;
    const int64_t cap = (int64_t)sm_count() * 8;
    if (blocks > cap) blocks = cap;
    resid_amax_kernel<<<(unsigned)blocks, 256, 0, st>>>((const uint16_t *)resid, rows_cap, k, offsets, E, amax_ws);
    int s = launch_status("resid_amax_kernel");
    if (s != NVFP4_OK) return s;
    blocks = (rows_cap * (k / 16) + 255) / 256;
    if (blocks > cap) blocks = cap;
    resid_qdq_kernel<<<(unsigned)blocks, 256, 0, st>>>((uint16_t *)resid, rows_cap, k, offsets, E, amax_ws, gs_out,
                                                      dev_status);
    return launch_status("resid_qdq_kernel");
}

extern "C" int nvfp4_rac_select_channels_online(const void *x, int64_t rows_cap, int64_t K, const int32_t *offsets,
                                                int32_t E, const float *amax, int32_t k, int32_t *S_out,
                                                double *score_ws, void *stream) {
    if (missing(x, rows_cap * K) || !amax || !score_ws || rows_cap < 0 || K < 0 || k < 0 || (offsets && E < 1))
        return NVFP4_ERR_INVALID_ARG;
    if (k > 0 && !S_out) return NVFP4_ERR_INVALID_ARG;
    if (K % 16 || K > 16384 || k > K) return NVFP4_ERR_UNSUPPORTED;
    if (!aligned16(x) || !aligned16(score_ws)) return NVFP4_ERR_ALIGNMENT;
    if (K == 0) return NVFP4_OK;
    NVFP4_CHECK_INIT();
    cudaStream_t st = (cudaStream_t)stream;
    double *part = score_ws + K;  // [kOnlineChunks][K]
    const int nchunks = (int)online_chunks(rows_cap, K);
    online_score_kernel<<<dim3((unsigned)nchunks, (unsigned)((K + 511) / 512)), 256, 0, st>>>(
        (const uint16_t *)x, rows_cap, K, offsets, E, amax, part);
    int s = launch_status("online_score_kernel");
    if (s != NVFP4_OK) return s;
    online_score_finish_kernel<<<(unsigned)((K + 31) / 32), 256, 0, st>>>(part, K, nchunks, score_ws);
    s = launch_status("online_score_finish_kernel");
    if (s != NVFP4_OK || k == 0) return s;
    select_topk_kernel<<<1, 1024, 0, st>>>(score_ws, K, k, S_out);
    return launch_status("select_topk_kernel");
}

extern "C" int nvfp4_gather_selected_weights(const uint8_t *w_codes, const uint8_t *w_scales, int32_t E, int64_t N,
                                             int64_t K, const int32_t *S, int32_t k, void *w_sel,
                                             int32_t *dev_status, void *stream) {
    if (!w_codes || !w_scales || !S || !w_sel || E < 1 || N < 0 || K < 0 || k < 1 || k > K)
        return NVFP4_ERR_INVALID_ARG;
    if (K % 64 || N % 128 || k % 8 || E > 65535 || K > 16384 || N / 128 > 0x7fffffff) return NVFP4_ERR_UNSUPPORTED;
    if (!aligned16(w_sel) || !aligned16(w_codes) || !aligned16(w_scales)) return NVFP4_ERR_ALIGNMENT;
    if (N == 0) return NVFP4_OK;
    NVFP4_CHECK_INIT();
    if (K >= 4096) {  // long rows: straight from global memory (measured faster there)
        gather_wsel_direct_kernel<<<dim3((unsigned)(N / (kGatherWarps * kGatherDirectRows)), (unsigned)E),
                                    32 * kGatherWarps, 0, (cudaStream_t)stream>>>(w_codes, w_scales, N, K, S, k,
                                                                                 (uint16_t *)w_sel);
        return launch_status("gather_wsel_direct_kernel");
    }
    const int64_t smem = gather_smem_bytes(K, k);
    if (smem > 227 * 1024) return NVFP4_ERR_UNSUPPORTED;
    if (smem > 48 * 1024) {
        const cudaError_t e = cudaFuncSetAttribute(gather_wsel_kernel, cudaFuncAttributeMaxDynamicSharedMemorySize,
                                                   (int)smem);
        if (e != cudaSuccess) {
            set_last_error("cudaFuncSetAttribute(gather_wsel_kernel)", e);
            return NVFP4_ERR_CUDA;
        }
    }
    gather_wsel_kernel<<<dim3((unsigned)(N / 128), (unsigned)E), 32 * kGatherWarps, (size_t)smem,
                         (cudaStream_t)stream>>>(w_codes, w_scales, N, K, S, k, (uint16_t *)w_sel, dev_status);
    return launch_status("gather_wsel_kernel");
}

extern "C" int nvfp4_transpose_weight_pack(const uint8_t *w_codes, const uint8_t *w_scales, int32_t E, int64_t N,
                                           int64_t K, uint8_t *codes_t, uint8_t *scales_t, void *stream) {
    if (!w_codes || !w_scales || !codes_t || !scales_t || E < 1 || N < 0 || K < 0) return NVFP4_ERR_INVALID_ARG;
    if (K % 64 || N % 128 || E > 65535 || K / 64 > 0x7fffffff || N / 64 > 65535) return NVFP4_ERR_UNSUPPORTED;
    if (!aligned16(w_codes) || !aligned16(codes_t)) return NVFP4_ERR_ALIGNMENT;
    if (N == 0 || K == 0) return NVFP4_OK;
    NVFP4_CHECK_INIT();
    pack_transpose_kernel<<<dim3((unsigned)(K / 64), (unsigned)(N / 64), (unsigned)E), 256, 0,
                            (cudaStream_t)stream>>>(w_codes, w_scales, N, K, codes_t, scales_t);
    return launch_status("pack_transpose_kernel");
}

extern "C" int nvfp4_gather_selected_weights_t(const uint8_t *codes_t, const uint8_t *scales_t, int32_t E, int64_t N,
                                               int64_t K, const int32_t *S, int32_t k, void *w_sel, void *stream) {
    if (!codes_t || !scales_t || !S || !w_sel || E < 1 || N < 0 || K < 0 || k < 1 || k > K)
        return NVFP4_ERR_INVALID_ARG;
    if (K % 64 || N % 128 || k % 8 || E > 65535 || N / 128 > 65535) return NVFP4_ERR_UNSUPPORTED;
    if (!aligned16(codes_t) || !aligned16(scales_t) || !aligned16(w_sel)) return NVFP4_ERR_ALIGNMENT;
    if (N == 0) return NVFP4_OK;
    NVFP4_CHECK_INIT();
    gather_wsel_t_kernel<<<dim3((unsigned)((k + 63) / 64), (unsigned)(N / 128), (unsigned)E), 256, 0,
                           (cudaStream_t)stream>>>(codes_t, scales_t, N, K, S, k, (uint16_t *)w_sel);
    return launch_status("gather_wsel_t_kernel");
}

extern "C" int nvfp4_moe_clear_padding(const int32_t *counts, const int32_t *offsets, int32_t E, int64_t rows_cap,
                                       int64_t K, int32_t k, uint8_t *codes, uint8_t *scales, void *resid,
                                       void *stream) {
    if (!counts || !offsets || !codes || !scales || E < 1 || K < 0 || k < 0 || rows_cap < 0)
        return NVFP4_ERR_INVALID_ARG;
    if (k > 0 && !resid) return NVFP4_ERR_INVALID_ARG;
    if (K % 32 || E > 65535) return NVFP4_ERR_UNSUPPORTED;
    NVFP4_CHECK_INIT();
    clear_padding_kernel<<<dim3(127, E), 128, 0, (cudaStream_t)stream>>>(counts, offsets, rows_cap, K, k, codes,
                                                                         scales, (uint16_t *)resid);
    return launch_status("clear_padding_kernel");
}

extern "C" int nvfp4_moe_scatter_rows(const void *x, int32_t T, int64_t K, int32_t topk, const int32_t *dst_row,
                                      const int32_t *counts, const int32_t *offsets, int32_t E, int64_t rows_cap,
                                      void *y, void *stream) {
    if (missing(x, (int64_t)T * K) || missing(dst_row, T) || !counts || !offsets || missing(y, rows_cap * K) || T < 0 ||
        K < 0 || topk < 1 || E < 1 || rows_cap < 0)
        return NVFP4_ERR_INVALID_ARG;
    if (K % 8 || E > 65535) return NVFP4_ERR_UNSUPPORTED;
    if (!aligned16(x) || !aligned16(y)) return NVFP4_ERR_ALIGNMENT;
    NVFP4_CHECK_INIT();
    cudaStream_t st = (cudaStream_t)stream;
    if (T > 0) {
        scatter_rows_kernel<<<T, 256, 0, st>>>((const uint16_t *)x, T, K, topk, dst_row, rows_cap, (uint16_t *)y);
        int s = launch_status("scatter_rows_kernel");
        if (s != NVFP4_OK) return s;
    }
    zero_pad_rows_kernel<<<dim3(127, E), 256, 0, st>>>(counts, offsets, rows_cap, K, (uint16_t *)y);
    return launch_status("zero_pad_rows_kernel");
}

extern "C" int nvfp4_rac_select_channels(const void *x, int64_t M, int64_t K, const float *amax, int32_t k,
                                         int32_t *S_out, double *score_ws, void *stream) {
    if (!x || !amax || !score_ws || M < 0 || K < 0 || k < 0) return NVFP4_ERR_INVALID_ARG;
    if (k > 0 && !S_out) return NVFP4_ERR_INVALID_ARG;
    if (K % 16 || K > 16384 || k > K) return NVFP4_ERR_UNSUPPORTED;
    if (!aligned16(x) || !aligned16(score_ws)) return NVFP4_ERR_ALIGNMENT;
    if (K == 0) return NVFP4_OK;
    NVFP4_CHECK_INIT();
    cudaStream_t st = (cudaStream_t)stream;
    channel_score_kernel<<<(unsigned)((K + 31) / 32), 32 * kScoreWarps, 0, st>>>((const uint16_t *)x, M, K, amax,
                                                                                 score_ws);
    int s = launch_status("channel_score_kernel");
    if (s != NVFP4_OK || k == 0) return s;
    select_topk_kernel<<<1, 1024, 0, st>>>(score_ws, K, k, S_out);
    return launch_status("select_topk_kernel");
}

// ---------------------------------------------------------------------------
// Fake-quant without any allocation by the caller.
//
// Some callers cannot hand the library a scratch buffer: a host framework
// that owns all device memory through its own pool (a raw cudaMalloc would
// bypass its accounting and can fail once the pool has reserved the GPU), or a
// latency-critical loop that must not call cudaMalloc/cudaFree (cudaFree waits
// for the whole device).  nvfp4_fake_quant needs ntensors floats of scratch
// for the per-tensor amax; this variant keeps them in a fixed array in device
// memory that the library itself declares, so nothing is allocated at call time.
namespace nvfp4 {
constexpr int kNoAllocMaxTensors = 4096;
// nvfp4_fake_quant's scratch for that many tensors (amax, done counts, counter): 32 KB per GPU
static __device__ __align__(256) float g_noalloc_amax[2 * kNoAllocMaxTensors + 1];
// device address of the array per device ordinal, and the CUDA context it was looked up in
static float *g_noalloc_addr[64];
static void *g_noalloc_ctx[64];
static std::mutex g_noalloc_mu;

// The array's name in host code is not a device address: look the address up
// with the device current, the first time a device is used, and pass it to
// the kernels.  A device reset gives the device a new context in which the
// array may sit elsewhere, so the cached address is keyed by the context too
// and looked up again when that changes.
static int noalloc_scratch(float **out) {
    int dev = 0;
    cudaError_t e = cudaGetDevice(&dev);
    if (e != cudaSuccess) {
        set_last_error("cudaGetDevice", e);
        return NVFP4_ERR_CUDA;
    }
    if (dev < 0 || dev >= 64) {
        set_last_error_text("nvfp4_fake_quant_noalloc: the library supports device ordinals 0..63");
        return NVFP4_ERR_ARCH;
    }
    void *ctx = current_context();
    std::lock_guard<std::mutex> lock(g_noalloc_mu);
    if (!g_noalloc_addr[dev] || g_noalloc_ctx[dev] != ctx) {
        void *p = nullptr;
        e = cudaGetSymbolAddress(&p, g_noalloc_amax);
        if (e != cudaSuccess || !p) {
            set_last_error("cudaGetSymbolAddress(no-alloc scratch)", e);
            return NVFP4_ERR_CUDA;
        }
        g_noalloc_addr[dev] = static_cast<float *>(p);
        g_noalloc_ctx[dev] = ctx;
    }
    *out = g_noalloc_addr[dev];
    return NVFP4_OK;
}
}  // namespace nvfp4

extern "C" int nvfp4_fake_quant_noalloc(const void *w, int32_t nt, int64_t rows, int64_t cols, void *w_hat,
                                        float *gs_out, int32_t *dev_status, void *stream) {
    if (!w || !w_hat || nt < 1 || rows < 0 || cols < 0) return NVFP4_ERR_INVALID_ARG;
    if (nt > kNoAllocMaxTensors) {
        set_last_error_text("nvfp4_fake_quant_noalloc: more than 4096 tensors in one call");
        return NVFP4_ERR_UNSUPPORTED;
    }
    if (cols % 32 || cols / 16 > kMaxBlocksPerRow) return NVFP4_ERR_UNSUPPORTED;
    if (!aligned16(w) || !aligned16(w_hat)) return NVFP4_ERR_ALIGNMENT;
    NVFP4_CHECK_INIT();
    float *scratch = nullptr;
    const int s = noalloc_scratch(&scratch);
    if (s != NVFP4_OK) return s;
    // the amax slots are cleared on `stream` before use (inside nvfp4_fake_quant)
    return nvfp4_fake_quant(w, nt, rows, cols, w_hat, gs_out, scratch, dev_status, stream);
}
