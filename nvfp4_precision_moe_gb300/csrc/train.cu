// train.cu -- the element-wise and data-movement kernels of the trainer-side
// backward of the asymmetric-QAT MoE layer (QUADS §3.2 Eq. 13: the
// straight-through estimator, dW = dW_hat and dX = W_hat^T dY; the GEMMs
// themselves are the grouped GEMMs of gemm.cu): BF16 batched transposes, the
// SwiGLU forward on saved pre-activations and its backward, and the backward
// of the weighted top-k combine.  All HBM-bound.
#include "common.cuh"

namespace nvfp4 {
namespace {

// y[b][c][r] = x[b][r][c] for a batch of rows x cols BF16 matrices: 32 x 32
// tiles through shared memory, so that both the reads (along c) and the writes
// (along r) are coalesced.
__global__ void __launch_bounds__(256) transpose_kernel(const uint16_t *x, int64_t rows, int64_t cols, uint16_t *y) {
    __shared__ uint16_t t[32][34];
    const int64_t off = (int64_t)blockIdx.z * rows * cols;
    const uint16_t *xb = x + off;
    uint16_t *yb = y + off;
    const int tx = threadIdx.x & 31, ty = threadIdx.x >> 5;  // 32 x 8
    for (int64_t r0 = (int64_t)blockIdx.y * 32; r0 < rows; r0 += (int64_t)gridDim.y * 32) {
        const int64_t c0 = (int64_t)blockIdx.x * 32;
#pragma unroll
        for (int i = 0; i < 32; i += 8) {
            const int64_t r = r0 + ty + i, c = c0 + tx;
            t[ty + i][tx] = (r < rows && c < cols) ? xb[r * cols + c] : (uint16_t)0;
        }
        __syncthreads();
#pragma unroll
        for (int i = 0; i < 32; i += 8) {
            const int64_t c = c0 + ty + i, r = r0 + tx;
            if (c < cols && r < rows) yb[c * rows + r] = t[tx][ty + i];
        }
        __syncthreads();
    }
}

// The same for even rows and cols: 64 x 64 tiles, 4-byte (two-element) reads
// along c and 4-byte writes along r, so a warp moves 128 contiguous bytes on
// both sides.
__global__ void __launch_bounds__(256) transpose64_kernel(const uint16_t *x, int64_t rows, int64_t cols,
                                                          uint16_t *y) {
    __shared__ uint16_t t[64][66];
    const int64_t off = (int64_t)blockIdx.z * rows * cols;
    const uint16_t *xb = x + off;
    uint16_t *yb = y + off;
    const int tx = threadIdx.x & 31, ty = threadIdx.x >> 5;  // 32 x 8
    const int64_t c0 = (int64_t)blockIdx.x * 64;
    for (int64_t r0 = (int64_t)blockIdx.y * 64; r0 < rows; r0 += (int64_t)gridDim.y * 64) {
#pragma unroll
        for (int i = 0; i < 64; i += 8) {
            const int64_t r = r0 + ty + i, c = c0 + 2 * tx;
            uint32_t v = 0u;
            if (r < rows && c < cols) v = *reinterpret_cast<const uint32_t *>(xb + r * cols + c);
            t[ty + i][2 * tx] = (uint16_t)(v & 0xffffu);
            t[ty + i][2 * tx + 1] = (uint16_t)(v >> 16);
        }
        __syncthreads();
#pragma unroll
        for (int i = 0; i < 64; i += 8) {
            const int64_t c = c0 + ty + i, r = r0 + 2 * tx;
            if (c < cols && r < rows)
                *reinterpret_cast<uint32_t *>(yb + c * rows + r) =
                    (uint32_t)t[2 * tx][ty + i] | ((uint32_t)t[2 * tx + 1][ty + i] << 16);
        }
        __syncthreads();
    }
}

// The same for rows and cols multiples of 8 and 16-byte aligned tensors:
// 64 x 64 tiles moved with 16-byte global accesses on both sides -- a thread
// reads 8 consecutive elements of a row and writes 8 consecutive elements of
// a column (gathered from shared memory, whose 33-word row pitch keeps the
// gathers at most 2-way bank-conflicted).
__global__ void __launch_bounds__(256) transpose64v_kernel(const uint16_t *x, int64_t rows, int64_t cols,
                                                           uint16_t *y) {
    __shared__ uint32_t t[64][33];  // 64 rows x 64 BF16 (2 per word) + 1 word of pad
    const int64_t off = (int64_t)blockIdx.z * rows * cols;
    const uint16_t *xb = x + off;
    uint16_t *yb = y + off;
    const int q = threadIdx.x & 7, rr = threadIdx.x >> 3;  // 8-element chunk, row within 32
    const int64_t c0 = (int64_t)blockIdx.x * 64;
    for (int64_t r0 = (int64_t)blockIdx.y * 64; r0 < rows; r0 += (int64_t)gridDim.y * 64) {
#pragma unroll
        for (int h = 0; h < 64; h += 32) {
            const int64_t r = r0 + rr + h, c = c0 + 8 * q;
            uint4 v = make_uint4(0, 0, 0, 0);
            if (r < rows && c < cols) v = __ldg(reinterpret_cast<const uint4 *>(xb + r * cols + c));
            t[rr + h][4 * q] = v.x;
            t[rr + h][4 * q + 1] = v.y;
            t[rr + h][4 * q + 2] = v.z;
            t[rr + h][4 * q + 3] = v.w;
        }
        __syncthreads();
#pragma unroll
        for (int h = 0; h < 64; h += 32) {
            const int cc = rr + h;  // output row = input column c0 + cc
            const int64_t c = c0 + cc, r = r0 + 8 * q;
            uint32_t o[4];
#pragma unroll
            for (int u = 0; u < 4; ++u) {
                const uint32_t a = t[8 * q + 2 * u][cc >> 1], b = t[8 * q + 2 * u + 1][cc >> 1];
                const uint32_t lo = (cc & 1) ? (a >> 16) : (a & 0xffffu);
                const uint32_t hi = (cc & 1) ? (b >> 16) : (b & 0xffffu);
                o[u] = lo | (hi << 16);
            }
            if (c < cols && r < rows) *reinterpret_cast<uint4 *>(yb + c * rows + r) = make_uint4(o[0], o[1], o[2], o[3]);
        }
        __syncthreads();
    }
}

__device__ __forceinline__ float bf(uint16_t h) { return __uint_as_float((uint32_t)h << 16); }
__device__ __forceinline__ uint16_t to_bf(float v) { return __bfloat16_as_ushort(__float2bfloat16_rn(v)); }

// logistic function with the accurate exponential
__device__ __forceinline__ float sigmoid(float g) { return __frcp_rn(__fadd_rn(1.0f, expf(-g))); }

// h = bf16(silu(g) * u) from saved BF16 pre-activations gu = [g | u] (rows x 2I)
__global__ void __launch_bounds__(256) swiglu_kernel(const uint16_t *gu, int64_t rows, int64_t I, uint16_t *h) {
    const int64_t total = rows * I;
    for (int64_t i = (int64_t)blockIdx.x * blockDim.x + threadIdx.x; i < total; i += (int64_t)gridDim.x * blockDim.x) {
        const int64_t r = i / I, c = i - r * I;
        const float g = bf(gu[r * 2 * I + c]), u = bf(gu[r * 2 * I + I + c]);
        h[i] = to_bf(__fmul_rn(__fmul_rn(g, sigmoid(g)), u));
    }
}

// The same with 16-byte accesses (I % 8 == 0): a block strides over rows, its
// threads over a row's 8-element vectors (no per-element index division).
__global__ void __launch_bounds__(256) swiglu8_kernel(const uint16_t *gu, int64_t rows, int64_t I, uint16_t *h) {
    for (int64_t r = blockIdx.x; r < rows; r += gridDim.x) {
        const uint16_t *g = gu + r * 2 * I, *u = g + I;
        for (int64_t c = (int64_t)threadIdx.x * 8; c < I; c += (int64_t)blockDim.x * 8) {
            const uint4 gv = __ldg(reinterpret_cast<const uint4 *>(g + c));
            const uint4 uv = __ldg(reinterpret_cast<const uint4 *>(u + c));
            const uint32_t G4[4] = {gv.x, gv.y, gv.z, gv.w}, U4[4] = {uv.x, uv.y, uv.z, uv.w};
            uint32_t o[4];
#pragma unroll
            for (int k = 0; k < 4; ++k) {
                uint32_t p = 0;
#pragma unroll
                for (int hh = 0; hh < 2; ++hh) {
                    const float gf = __uint_as_float(hh ? (G4[k] & 0xffff0000u) : (G4[k] << 16));
                    const float uf = __uint_as_float(hh ? (U4[k] & 0xffff0000u) : (U4[k] << 16));
                    p |= (uint32_t)to_bf(__fmul_rn(__fmul_rn(gf, sigmoid(gf)), uf)) << (16 * hh);
                }
                o[k] = p;
            }
            *reinterpret_cast<uint4 *>(h + r * I + c) = make_uint4(o[0], o[1], o[2], o[3]);
        }
    }
}

// dg = dh * u * silu'(g), du = dh * silu(g); silu'(g) = s (1 + g (1 - s)), s = sigmoid(g)
__global__ void __launch_bounds__(256) swiglu_backward_kernel(const uint16_t *gu, const uint16_t *dh, int64_t rows,
                                                              int64_t I, uint16_t *dgu) {
    const int64_t total = rows * I;
    for (int64_t i = (int64_t)blockIdx.x * blockDim.x + threadIdx.x; i < total; i += (int64_t)gridDim.x * blockDim.x) {
        const int64_t r = i / I, c = i - r * I;
        const float g = bf(gu[r * 2 * I + c]), u = bf(gu[r * 2 * I + I + c]), d = bf(dh[i]);
        const float s = sigmoid(g);
        const float ds = __fmul_rn(s, __fadd_rn(1.0f, __fmul_rn(g, __fsub_rn(1.0f, s))));
        dgu[r * 2 * I + c] = to_bf(__fmul_rn(__fmul_rn(d, u), ds));
        dgu[r * 2 * I + I + c] = to_bf(__fmul_rn(d, __fmul_rn(g, s)));
    }
}

// The SwiGLU backward with 16-byte accesses (I % 8 == 0): 8 elements per thread
__global__ void __launch_bounds__(256) swiglu_backward8_kernel(const uint16_t *gu, const uint16_t *dh, int64_t rows,
                                                               int64_t I, uint16_t *dgu) {
    const int64_t per_row = I >> 3, total = rows * per_row;
    for (int64_t i = (int64_t)blockIdx.x * blockDim.x + threadIdx.x; i < total; i += (int64_t)gridDim.x * blockDim.x) {
        const int64_t r = i / per_row, c = (i - r * per_row) * 8;
        const uint4 gv = __ldg(reinterpret_cast<const uint4 *>(gu + r * 2 * I + c));
        const uint4 uv = __ldg(reinterpret_cast<const uint4 *>(gu + r * 2 * I + I + c));
        const uint4 dv = __ldg(reinterpret_cast<const uint4 *>(dh + r * I + c));
        const uint32_t G4[4] = {gv.x, gv.y, gv.z, gv.w}, U4[4] = {uv.x, uv.y, uv.z, uv.w},
                       D4[4] = {dv.x, dv.y, dv.z, dv.w};
        uint32_t og[4], ou[4];
#pragma unroll
        for (int k = 0; k < 4; ++k) {
            uint32_t pg = 0, pu = 0;
#pragma unroll
            for (int hh = 0; hh < 2; ++hh) {
                const float g = __uint_as_float(hh ? (G4[k] & 0xffff0000u) : (G4[k] << 16));
                const float u = __uint_as_float(hh ? (U4[k] & 0xffff0000u) : (U4[k] << 16));
                const float d = __uint_as_float(hh ? (D4[k] & 0xffff0000u) : (D4[k] << 16));
                const float sg = sigmoid(g);
                const float ds = __fmul_rn(sg, __fadd_rn(1.0f, __fmul_rn(g, __fsub_rn(1.0f, sg))));
                pg |= (uint32_t)to_bf(__fmul_rn(__fmul_rn(d, u), ds)) << (16 * hh);
                pu |= (uint32_t)to_bf(__fmul_rn(d, __fmul_rn(g, sg))) << (16 * hh);
            }
            og[k] = pg;
            ou[k] = pu;
        }
        *reinterpret_cast<uint4 *>(dgu + r * 2 * I + c) = make_uint4(og[0], og[1], og[2], og[3]);
        *reinterpret_cast<uint4 *>(dgu + r * 2 * I + I + c) = make_uint4(ou[0], ou[1], ou[2], ou[3]);
    }
}

// Backward of out[t] = sum_s w[t,s] y[dst[t,s]]: the routed gradient
// dy[dst[t,s]] = bf16(w[t,s] dout[t]) and, when asked, the weights' gradient
// dw[t,s] = <y[dst[t,s]], dout[t]> (binary32 lane sums in element order, a
// warp's lanes by a butterfly, then the block's warps in order; one block per
// token).  H % 8 == 0 and 16-byte aligned rows: NV 8-element vectors per
// thread (dout read once per token into registers, reused for every slot);
// the rows of kCombineBwdGroup slots are loaded together, and the weights'
// gradients of all slots are summed across warps after one barrier.
constexpr int kCombineBwdMaxVec = 4;  // 8-element vectors per thread: H <= 8 * 256 * 4
constexpr int kCombineBwdGroup = 4;
constexpr int kCombineBwdMaxTopk = 32;
template <int NV>
__global__ void __launch_bounds__(256) combine_backward_kernel(const float *dout, const uint16_t *y,
                                                               const int32_t *dst, const float *w, int32_t topk,
                                                               int64_t H, int64_t rows_cap, uint16_t *dy, float *dw) {
    __shared__ float red[kCombineBwdMaxTopk][8];
    const int64_t t = blockIdx.x;
    const int nv = (int)(H >> 3);
    float g[NV][8];
#pragma unroll
    for (int i = 0; i < NV; ++i) {
        const int v = threadIdx.x + 256 * i;
        if (v < nv) {
            const float4 a = __ldg(reinterpret_cast<const float4 *>(dout + t * H) + 2 * v);
            const float4 b = __ldg(reinterpret_cast<const float4 *>(dout + t * H) + 2 * v + 1);
            g[i][0] = a.x, g[i][1] = a.y, g[i][2] = a.z, g[i][3] = a.w;
            g[i][4] = b.x, g[i][5] = b.y, g[i][6] = b.z, g[i][7] = b.w;
        }
    }
    for (int s0 = 0; s0 < topk; s0 += kCombineBwdGroup) {
        int64_t r[kCombineBwdGroup];
        bool ok[kCombineBwdGroup];
        float ws[kCombineBwdGroup];
        uint4 yv[kCombineBwdGroup][NV];
#pragma unroll
        for (int j = 0; j < kCombineBwdGroup; ++j) {
            const bool in = s0 + j < topk;
            r[j] = in ? (int64_t)dst[t * topk + s0 + j] : -1;
            ok[j] = in && r[j] >= 0 && r[j] < rows_cap;
            ws[j] = in ? w[t * topk + s0 + j] : 0.0f;
        }
#pragma unroll
        for (int j = 0; j < kCombineBwdGroup; ++j)
#pragma unroll
            for (int i = 0; i < NV; ++i) {
                const int v = threadIdx.x + 256 * i;
                if (ok[j] && v < nv) yv[j][i] = __ldg(reinterpret_cast<const uint4 *>(y + r[j] * H) + v);
            }
#pragma unroll
        for (int j = 0; j < kCombineBwdGroup; ++j) {
            float acc = 0.0f;
#pragma unroll
            for (int i = 0; i < NV; ++i) {
                const int v = threadIdx.x + 256 * i;
                if (ok[j] && v < nv) {
                    const uint32_t yw[4] = {yv[j][i].x, yv[j][i].y, yv[j][i].z, yv[j][i].w};
                    uint32_t o[4];
#pragma unroll
                    for (int k = 0; k < 4; ++k) {
                        o[k] = (uint32_t)to_bf(__fmul_rn(ws[j], g[i][2 * k])) |
                               ((uint32_t)to_bf(__fmul_rn(ws[j], g[i][2 * k + 1])) << 16);
                        acc = __fmaf_rn(__uint_as_float(yw[k] << 16), g[i][2 * k], acc);
                        acc = __fmaf_rn(__uint_as_float(yw[k] & 0xffff0000u), g[i][2 * k + 1], acc);
                    }
                    reinterpret_cast<uint4 *>(dy + r[j] * H)[v] = make_uint4(o[0], o[1], o[2], o[3]);
                }
            }
            if (dw && s0 + j < topk) {
#pragma unroll
                for (int o = 16; o > 0; o >>= 1) acc += __shfl_xor_sync(0xffffffffu, acc, o);
                if ((threadIdx.x & 31) == 0) red[s0 + j][threadIdx.x >> 5] = acc;
            }
        }
    }
    if (dw) {
        __syncthreads();
        if ((int)threadIdx.x < topk) {
            float sum = 0.0f;
            for (int i = 0; i < 8; ++i) sum += red[threadIdx.x][i];
            dw[t * topk + threadIdx.x] = sum;
        }
    }
}

// zero the padding rows [offsets[e] + counts[e], offsets[e+1]) of a routed BF16 tensor
__global__ void zero_padding_bf16_kernel(const int32_t *counts, const int32_t *offsets, int64_t rows_cap, int64_t H,
                                         uint16_t *y) {
    const int e = blockIdx.y;
    const int64_t row = (int64_t)offsets[e] + counts[e] + blockIdx.x;
    if (row >= offsets[e + 1] || row >= rows_cap || row < 0) return;
    for (int64_t h = threadIdx.x; h < H; h += blockDim.x) y[row * H + h] = 0;
}

int grid_for(int64_t work, int64_t per_block) {
    int64_t b = (work + per_block - 1) / per_block;
    const int64_t cap = (int64_t)sm_count() * 8;
    if (b > cap) b = cap;
    return (int)(b < 1 ? 1 : b);
}

}  // namespace
}  // namespace nvfp4

using namespace nvfp4;

extern "C" int nvfp4_transpose_bf16(const void *x, int32_t batch, int64_t rows, int64_t cols, void *y, void *stream) {
    if (!x || !y || batch < 1 || rows < 0 || cols < 0) return NVFP4_ERR_INVALID_ARG;
    if (batch > 65535 || (cols + 31) / 32 > 0x7fffffff) return NVFP4_ERR_UNSUPPORTED;
    if (rows == 0 || cols == 0) return NVFP4_OK;
    NVFP4_CHECK_INIT();
    if (rows % 8 == 0 && cols % 8 == 0 && reinterpret_cast<uintptr_t>(x) % 16 == 0 &&
        reinterpret_cast<uintptr_t>(y) % 16 == 0) {
        const int64_t gy = (rows + 63) / 64;
        transpose64v_kernel<<<dim3((unsigned)((cols + 63) / 64), (unsigned)(gy < 65535 ? gy : 65535),
                                   (unsigned)batch),
                              256, 0, (cudaStream_t)stream>>>((const uint16_t *)x, rows, cols, (uint16_t *)y);
        return launch_status("transpose64v_kernel");
    }
    if (rows % 2 == 0 && cols % 2 == 0 && reinterpret_cast<uintptr_t>(x) % 4 == 0 &&
        reinterpret_cast<uintptr_t>(y) % 4 == 0) {
        const int64_t gy = (rows + 63) / 64;
        transpose64_kernel<<<dim3((unsigned)((cols + 63) / 64), (unsigned)(gy < 65535 ? gy : 65535), (unsigned)batch),
                             256, 0, (cudaStream_t)stream>>>((const uint16_t *)x, rows, cols, (uint16_t *)y);
        return launch_status("transpose64_kernel");
    }
    const int64_t gy = (rows + 31) / 32;
    transpose_kernel<<<dim3((unsigned)((cols + 31) / 32), (unsigned)(gy < 65535 ? gy : 65535), (unsigned)batch), 256,
                       0, (cudaStream_t)stream>>>((const uint16_t *)x, rows, cols, (uint16_t *)y);
    return launch_status("transpose_kernel");
}

extern "C" int nvfp4_swiglu(const void *gu, int64_t rows, int64_t I, void *h, void *stream) {
    if (!gu || !h || rows < 0 || I < 0) return NVFP4_ERR_INVALID_ARG;
    if (rows == 0 || I == 0) return NVFP4_OK;
    NVFP4_CHECK_INIT();
    if (I % 8 == 0 && aligned16(gu) && aligned16(h)) {
        int64_t blocks = rows, cap = (int64_t)sm_count() * 8;
        if (blocks > cap) blocks = cap;
        swiglu8_kernel<<<(unsigned)blocks, 256, 0, (cudaStream_t)stream>>>((const uint16_t *)gu, rows, I,
                                                                           (uint16_t *)h);
        return launch_status("swiglu8_kernel");
    }
    swiglu_kernel<<<grid_for(rows * I, 256), 256, 0, (cudaStream_t)stream>>>((const uint16_t *)gu, rows, I,
                                                                            (uint16_t *)h);
    return launch_status("swiglu_kernel");
}

extern "C" int nvfp4_swiglu_backward(const void *gu, const void *dh, int64_t rows, int64_t I, void *dgu,
                                     void *stream) {
    if (!gu || !dh || !dgu || rows < 0 || I < 0) return NVFP4_ERR_INVALID_ARG;
    if (rows == 0 || I == 0) return NVFP4_OK;
    NVFP4_CHECK_INIT();
    if (I % 8 == 0 && reinterpret_cast<uintptr_t>(gu) % 16 == 0 && reinterpret_cast<uintptr_t>(dh) % 16 == 0 &&
        reinterpret_cast<uintptr_t>(dgu) % 16 == 0) {
        swiglu_backward8_kernel<<<grid_for(rows * I / 8, 256), 256, 0, (cudaStream_t)stream>>>(
            (const uint16_t *)gu, (const uint16_t *)dh, rows, I, (uint16_t *)dgu);
        return launch_status("swiglu_backward8_kernel");
    }
    swiglu_backward_kernel<<<grid_for(rows * I, 256), 256, 0, (cudaStream_t)stream>>>(
        (const uint16_t *)gu, (const uint16_t *)dh, rows, I, (uint16_t *)dgu);
    return launch_status("swiglu_backward_kernel");
}

extern "C" int nvfp4_moe_combine_backward(const float *dout, const void *y, const int32_t *dst_row,
                                          const float *weights, int32_t T, int32_t topk, int64_t H,
                                          const int32_t *counts, const int32_t *offsets, int32_t E, int64_t rows_cap,
                                          void *dy, float *dweights, void *stream) {
    if (missing(dout, (int64_t)T * H) || missing(y, rows_cap * H) || missing(dst_row, T) || missing(weights, T) || !counts ||
        !offsets || missing(dy, rows_cap * H) || T < 0 || topk < 1 || H < 0 || E < 1 || rows_cap < 0)
        return NVFP4_ERR_INVALID_ARG;
    if (E > 65535 || H % 8 || H > 8 * 256 * kCombineBwdMaxVec || topk > kCombineBwdMaxTopk)
        return NVFP4_ERR_UNSUPPORTED;
    if (!aligned16(dout) || !aligned16(y) || !aligned16(dy)) return NVFP4_ERR_ALIGNMENT;
    if (H == 0) return NVFP4_OK;
    NVFP4_CHECK_INIT();
    cudaStream_t st = (cudaStream_t)stream;
    zero_padding_bf16_kernel<<<dim3(127, E), 256, 0, st>>>(counts, offsets, rows_cap, H, (uint16_t *)dy);
    int s = launch_status("zero_padding_bf16_kernel");
    if (s != NVFP4_OK || T == 0) return s;
    const int nv = (int)((H / 8 + 255) / 256);  // 8-element vectors per thread
    auto kern = nv <= 1 ? combine_backward_kernel<1>
                        : nv == 2 ? combine_backward_kernel<2> : nv == 3 ? combine_backward_kernel<3> : combine_backward_kernel<4>;
    kern<<<(unsigned)T, 256, 0, st>>>(dout, (const uint16_t *)y, dst_row, weights, topk, H, rows_cap, (uint16_t *)dy,
                                      dweights);
    return launch_status("combine_backward_kernel");
}
