// moe.cu -- MoE routing (top-k softmax), routed-row layout and combine.
//
// The paper's MoE layers (QUADS §4.1, MoE 25B-A2.8B) do not spell out the
// router; this is the plainest top-k softmax router: FP32 softmax over the
// experts, the k largest logits (ties to the lower expert index), their
// probabilities as combine weights without renormalization.  Routed rows are
// grouped by expert, tokens in order inside an expert, and every expert
// segment starts at a multiple of 128 rows (one GEMM M-tile).
#include "common.cuh"

namespace nvfp4 {

// A logit as an unsigned key whose integer order is the float order (-0
// counts as +0, so the two tie as floats do), and back.
__device__ __forceinline__ uint32_t order_key(float f) {
    uint32_t u = __float_as_uint(f);
    if (u == 0x80000000u) u = 0u;
    return (u & 0x80000000u) ? ~u : (u | 0x80000000u);
}
__device__ __forceinline__ float key_value(uint32_t k) { return __uint_as_float((k & 0x80000000u) ? (k & 0x7fffffffu) : ~k); }

// One warp per token.  Lane l holds the keys of experts l + 32i (kPer of them,
// E <= 32 kPer) in registers.  Each of the topk selections is two warp
// reductions: the largest key among the lanes' best untaken ones, then the
// lowest expert index holding it (ties go to the lower expert).  The softmax
// sum adds a lane's experts in order, then across lanes by a butterfly.  Each
// block counts the experts its tokens chose in shared memory and adds its
// counts into `counts` (zeroed on the stream before the launch).
template <int kPer>
__global__ void __launch_bounds__(256) topk_kernel(const float *logits, int32_t T, int32_t E, int32_t topk,
                                                   int32_t *ids, float *weights, int32_t *counts) {
    __shared__ int32_t s_hist[1024];
    for (int e = threadIdx.x; e < E; e += blockDim.x) s_hist[e] = 0;
    __syncthreads();
    const int lane = threadIdx.x & 31;
    const int64_t warps = (int64_t)gridDim.x * (blockDim.x >> 5);
    for (int64_t t = (int64_t)blockIdx.x * (blockDim.x >> 5) + (threadIdx.x >> 5); t < T; t += warps) {
        const float *l = logits + t * E;
        uint32_t key[kPer];
        uint32_t lmax = 0u;
#pragma unroll
        for (int i = 0; i < kPer; ++i) {
            const int e = lane + 32 * i;
            key[i] = e < E ? order_key(__ldg(l + e)) : 0u;
            lmax = max(lmax, key[i]);
        }
        const float mx = key_value(__reduce_max_sync(0xffffffffu, lmax));
        float sum = 0.0f;
#pragma unroll
        for (int i = 0; i < kPer; ++i)
            if (lane + 32 * i < E) sum += expf(key_value(key[i]) - mx);
#pragma unroll
        for (int o = 16; o > 0; o >>= 1) sum += __shfl_xor_sync(0xffffffffu, sum, o);
        uint32_t taken = 0u;  // bit i: expert lane + 32i is chosen
        uint32_t my_id = 0u, my_key = 0u;
        for (int s = 0; s < topk; ++s) {
            // this lane's best untaken expert (strict >: the lower index of equal keys); with
            // topk <= E some lane always has one, so the chosen index is always < E
            uint32_t bk = 0u;
            int bi = -1;
#pragma unroll
            for (int i = 0; i < kPer; ++i)
                if (lane + 32 * i < E && !((taken >> i) & 1u) && (bi < 0 || key[i] > bk)) {
                    bk = key[i];
                    bi = i;
                }
            const uint32_t gk = __reduce_max_sync(0xffffffffu, bk);
            const uint32_t ge =
                __reduce_min_sync(0xffffffffu, bi >= 0 && bk == gk ? (uint32_t)(lane + 32 * bi) : 0xffffffffu);
            if ((int)(ge & 31u) == lane) taken |= 1u << (ge >> 5);
            if (lane == s) {
                my_id = ge;
                my_key = gk;
            }
        }
        if (lane < topk) {
            ids[t * topk + lane] = (int32_t)my_id;
            weights[t * topk + lane] = expf(key_value(my_key) - mx) / sum;
            if (my_id < (uint32_t)E) atomicAdd(&s_hist[my_id], 1);
        }
    }
    __syncthreads();
    for (int e = threadIdx.x; e < E; e += blockDim.x)
        if (s_hist[e]) atomicAdd(&counts[e], s_hist[e]);
}

// Block per expert: the padded segment start (from all experts' counts), then
// the ranks of its tokens in token order.  Thread i owns a contiguous run of
// tokens.  A run of at most 128 ids (read 16 bytes at a time, eight loads in
// flight) keeps its matches as a 128-bit mask, so the ids are read once
// however many of them match; a longer run counts its matches and reads the
// run again to write them.  A block-wide scan gives each run its first rank.
constexpr int kMaskIds = 128;

__global__ void __launch_bounds__(1024) dst_row_kernel(const int32_t *ids, int32_t T, int32_t E, int32_t topk,
                                                       const int32_t *counts, int32_t *offsets, int32_t *dst_row) {
    const int e = blockIdx.x;
    __shared__ int32_t s_part[32];
    __shared__ int32_t s_base;
    const int lane = threadIdx.x & 31, wid = threadIdx.x >> 5, nw = blockDim.x >> 5;
    if (wid == 0) {  // segment start: sum of the padded counts of experts < e
        int64_t off = 0;
        for (int i = lane; i < e; i += 32) off += (counts[i] + 127) / 128 * 128;
#pragma unroll
        for (int o = 16; o > 0; o >>= 1) off += __shfl_xor_sync(0xffffffffu, off, o);
        if (lane == 0) {
            s_base = (int32_t)off;
            offsets[e] = (int32_t)off;
            if (e == E - 1) offsets[E] = (int32_t)(off + (counts[e] + 127) / 128 * 128);
        }
    }
    const int64_t per = (T + (int64_t)blockDim.x - 1) / blockDim.x;
    const int64_t t0 = (int64_t)threadIdx.x * per;
    const int64_t t1 = min((int64_t)T, t0 + per);
    const int64_t n = t1 > t0 ? (t1 - t0) * topk : 0;  // ids in the run
    const int32_t *run = ids + t0 * topk;
    // the run's ids are contiguous: read them 16 bytes at a time when rows are whole int4s
    const bool vec = (topk & 3) == 0 && (reinterpret_cast<uintptr_t>(ids) & 15) == 0;
    const bool masked = vec && n <= kMaskIds;
    const int4 *p = reinterpret_cast<const int4 *>(run);
    uint32_t mk[kMaskIds / 32] = {0u, 0u, 0u, 0u};  // bit j: id j of the run is e
    int c = 0;
    if (masked) {
        const int n4 = (int)(n / 4);
#pragma unroll
        for (int i0 = 0; i0 < kMaskIds / 4; i0 += 8) {
            int4 q[8];
#pragma unroll
            for (int u = 0; u < 8; ++u) q[u] = i0 + u < n4 ? __ldg(p + i0 + u) : make_int4(-1, -1, -1, -1);
#pragma unroll
            for (int u = 0; u < 8; ++u) {
                const int i = i0 + u;
                const uint32_t b = (uint32_t)(q[u].x == e) | ((uint32_t)(q[u].y == e) << 1) |
                                   ((uint32_t)(q[u].z == e) << 2) | ((uint32_t)(q[u].w == e) << 3);
                mk[i >> 3] |= b << (4 * (i & 7));
            }
        }
#pragma unroll
        for (int w = 0; w < kMaskIds / 32; ++w) c += __popc(mk[w]);
    } else if (vec) {
        const int64_t n4 = n / 4;
        int64_t i = 0;
        for (; i + 8 <= n4; i += 8) {  // eight 16-byte loads in flight
            int4 q[8];
#pragma unroll
            for (int u = 0; u < 8; ++u) q[u] = __ldg(p + i + u);
#pragma unroll
            for (int u = 0; u < 8; ++u) c += (q[u].x == e) + (q[u].y == e) + (q[u].z == e) + (q[u].w == e);
        }
        for (; i < n4; ++i) {
            const int4 q = __ldg(p + i);
            c += (q.x == e) + (q.y == e) + (q.z == e) + (q.w == e);
        }
    } else {
        for (int64_t i = 0; i < n; ++i) c += run[i] == e;
    }
    // block-wide exclusive scan of c (thread order = token order)
    int incl = c;
#pragma unroll
    for (int o = 1; o < 32; o <<= 1) {
        const int v = __shfl_up_sync(0xffffffffu, incl, o);
        if (lane >= o) incl += v;
    }
    if (lane == 31) s_part[wid] = incl;
    __syncthreads();
    if (wid == 0) {
        int v = lane < nw ? s_part[lane] : 0;
        int w = v;
#pragma unroll
        for (int o = 1; o < 32; o <<= 1) {
            const int u = __shfl_up_sync(0xffffffffu, w, o);
            if (lane >= o) w += u;
        }
        if (lane < nw) s_part[lane] = w - v;  // exclusive prefix of the warps
    }
    __syncthreads();
    int r = s_base + s_part[wid] + incl - c;
    if (c == 0) return;  // nothing of this expert in the run
    int32_t *d = dst_row + t0 * topk;
    if (masked) {
#pragma unroll
        for (int w = 0; w < kMaskIds / 32; ++w)
            for (uint32_t m = mk[w]; m; m &= m - 1u) d[32 * w + __ffs((int)m) - 1] = r++;
    } else if (vec) {  // a second pass over the run, 16 bytes at a time
        const int64_t n4 = n / 4;
        for (int64_t i = 0; i < n4; ++i) {
            const int4 q = __ldg(p + i);
            if (q.x == e) d[4 * i] = r++;
            if (q.y == e) d[4 * i + 1] = r++;
            if (q.z == e) d[4 * i + 2] = r++;
            if (q.w == e) d[4 * i + 3] = r++;
        }
    } else {
        for (int64_t i = 0; i < n; ++i)
            if (run[i] == e) d[i] = r++;
    }
}

// out[t, c:c+8] = sum_s w[t,s] * y[row(t,s), c:c+8] in FP32, slots in order
template <bool BF16>
__global__ void combine_kernel(const void *y, int64_t ldy, const int32_t *dst_row, const float *weights,
                               int32_t T, int32_t topk, int64_t H, float *out) {
    const int64_t per_row = H >> 3;
    const int64_t total = (int64_t)T * per_row;
    for (int64_t i = (int64_t)blockIdx.x * blockDim.x + threadIdx.x; i < total; i += (int64_t)gridDim.x * blockDim.x) {
        const int64_t t = i / per_row, c = (i - t * per_row) * 8;
        float acc[8] = {0, 0, 0, 0, 0, 0, 0, 0};
        for (int s = 0; s < topk; ++s) {
            const int64_t row = dst_row[t * topk + s];
            const float w = weights[t * topk + s];
            float v[8];
            if (BF16) {
                uint4 q = __ldg(reinterpret_cast<const uint4 *>(reinterpret_cast<const uint16_t *>(y) + row * ldy + c));
                uint32_t ww[4] = {q.x, q.y, q.z, q.w};
#pragma unroll
                for (int j = 0; j < 4; ++j) {
                    v[2 * j] = __uint_as_float(ww[j] << 16);
                    v[2 * j + 1] = __uint_as_float(ww[j] & 0xffff0000u);
                }
            } else {
                const float4 *p = reinterpret_cast<const float4 *>(reinterpret_cast<const float *>(y) + row * ldy + c);
                float4 a = __ldg(p), b = __ldg(p + 1);
                v[0] = a.x; v[1] = a.y; v[2] = a.z; v[3] = a.w;
                v[4] = b.x; v[5] = b.y; v[6] = b.z; v[7] = b.w;
            }
#pragma unroll
            for (int j = 0; j < 8; ++j) acc[j] = __fadd_rn(acc[j], __fmul_rn(w, v[j]));
        }
        float4 *o = reinterpret_cast<float4 *>(out + t * H + c);
        o[0] = make_float4(acc[0], acc[1], acc[2], acc[3]);
        o[1] = make_float4(acc[4], acc[5], acc[6], acc[7]);
    }
}

// BF16 routed rows, topk <= kCombineMaxK: every slot's 16 bytes are loaded
// before the slots are summed (in slot order, as above), so a thread keeps
// topk loads in flight instead of one.
constexpr int kCombineMaxK = 8;
__global__ void combine_bf16_kernel(const uint16_t *y, int64_t ldy, const int32_t *dst_row, const float *weights,
                                    int32_t T, int32_t topk, int64_t H, float *out) {
    const int64_t per_row = H >> 3;
    const int64_t total = (int64_t)T * per_row;
    for (int64_t i = (int64_t)blockIdx.x * blockDim.x + threadIdx.x; i < total; i += (int64_t)gridDim.x * blockDim.x) {
        const int64_t t = i / per_row, c = (i - t * per_row) * 8;
        uint4 q[kCombineMaxK];
        float w[kCombineMaxK];
#pragma unroll
        for (int s = 0; s < kCombineMaxK; ++s) {
            if (s < topk) {
                const int64_t row = __ldg(dst_row + t * topk + s);
                w[s] = __ldg(weights + t * topk + s);
                q[s] = __ldg(reinterpret_cast<const uint4 *>(y + row * ldy + c));
            }
        }
        float acc[8] = {0, 0, 0, 0, 0, 0, 0, 0};
#pragma unroll
        for (int s = 0; s < kCombineMaxK; ++s) {
            if (s < topk) {
                const uint32_t ww[4] = {q[s].x, q[s].y, q[s].z, q[s].w};
#pragma unroll
                for (int j = 0; j < 4; ++j) {
                    acc[2 * j] = __fadd_rn(acc[2 * j], __fmul_rn(w[s], __uint_as_float(ww[j] << 16)));
                    acc[2 * j + 1] = __fadd_rn(acc[2 * j + 1], __fmul_rn(w[s], __uint_as_float(ww[j] & 0xffff0000u)));
                }
            }
        }
        float4 *o = reinterpret_cast<float4 *>(out + t * H + c);
        o[0] = make_float4(acc[0], acc[1], acc[2], acc[3]);
        o[1] = make_float4(acc[4], acc[5], acc[6], acc[7]);
    }
}

// QUADS §3.1 Eq. 11: sum (a - b)^2 and sum b^2, each thread in binary64 over
// its grid-stride share (FP32 products of FP32 values are exact in binary64),
// then a warp reduction and one atomic add per warp.
__global__ void mismatch_kernel(const float *a, const float *b, int64_t n, double *acc) {
    double d2 = 0.0, b2 = 0.0;
    for (int64_t i = (int64_t)blockIdx.x * blockDim.x + threadIdx.x; i < n; i += (int64_t)gridDim.x * blockDim.x) {
        const double x = (double)a[i], y = (double)b[i];
        d2 = __dadd_rn(d2, __dmul_rn(__dsub_rn(x, y), __dsub_rn(x, y)));
        b2 = __dadd_rn(b2, __dmul_rn(y, y));
    }
#pragma unroll
    for (int o = 16; o > 0; o >>= 1) {
        d2 += __shfl_xor_sync(0xffffffffu, d2, o);
        b2 += __shfl_xor_sync(0xffffffffu, b2, o);
    }
    if ((threadIdx.x & 31) == 0) {
        atomicAdd(&acc[0], d2);
        atomicAdd(&acc[1], b2);
    }
}

}  // namespace nvfp4

using namespace nvfp4;

extern "C" int nvfp4_mismatch_norm(const float *y_infer, const float *y_train, int64_t n, double *acc, void *stream) {
    if (!y_infer || !y_train || !acc || n < 0) return NVFP4_ERR_INVALID_ARG;
    if (!aligned16(y_infer) || !aligned16(y_train) || !aligned16(acc)) return NVFP4_ERR_ALIGNMENT;
    NVFP4_CHECK_INIT();
    cudaStream_t st = (cudaStream_t)stream;
    const cudaError_t e = cudaMemsetAsync(acc, 0, 2 * sizeof(double), st);
    if (e != cudaSuccess) {
        set_last_error("cudaMemsetAsync(acc)", e);
        return NVFP4_ERR_CUDA;
    }
    if (n == 0) return NVFP4_OK;
    int64_t blocks = (n + 255) / 256, cap = (int64_t)sm_count() * 8;
    if (blocks > cap) blocks = cap;
    mismatch_kernel<<<(unsigned)blocks, 256, 0, st>>>(y_infer, y_train, n, acc);
    return launch_status("mismatch_kernel");
}

extern "C" int nvfp4_route_topk(const float *logits, int32_t T, int32_t E, int32_t topk, int32_t *ids, float *weights,
                                int32_t *counts, int32_t *offsets, int32_t *dst_row, void *stream) {
    if (missing(logits, T) || missing(ids, T) || missing(weights, T) || !counts || !offsets || missing(dst_row, T) ||
        T < 0 || E < 1 || topk < 1)
        return NVFP4_ERR_INVALID_ARG;
    if (topk > 32 || topk > E || E > 1024) return NVFP4_ERR_UNSUPPORTED;
    NVFP4_CHECK_INIT();
    cudaStream_t st = (cudaStream_t)stream;
    const cudaError_t ce = cudaMemsetAsync(counts, 0, sizeof(int32_t) * (size_t)E, st);
    if (ce != cudaSuccess) {
        set_last_error("cudaMemsetAsync(counts)", ce);
        return NVFP4_ERR_CUDA;
    }
    if (T > 0) {
        // a warp per token: the selection passes are latency-bound, so every token gets its own warp
        const unsigned blocks = (unsigned)((T + 7) / 8);
        if (E <= 128) topk_kernel<4><<<blocks, 256, 0, st>>>(logits, T, E, topk, ids, weights, counts);
        else if (E <= 256) topk_kernel<8><<<blocks, 256, 0, st>>>(logits, T, E, topk, ids, weights, counts);
        else topk_kernel<32><<<blocks, 256, 0, st>>>(logits, T, E, topk, ids, weights, counts);
        int s = launch_status("topk_kernel");
        if (s != NVFP4_OK) return s;
    }
    dst_row_kernel<<<E, 1024, 0, st>>>(ids, T, E, topk, counts, offsets, dst_row);
    return launch_status("dst_row_kernel");
}

extern "C" int nvfp4_moe_combine(const void *y, int32_t y_dtype, int64_t ldy, const int32_t *dst_row,
                                 const float *weights, int32_t T, int32_t topk, int64_t H, float *out, void *stream) {
    if (missing(y, (int64_t)T * H) || missing(dst_row, T) || missing(weights, T) || missing(out, (int64_t)T * H) || T < 0 ||
        topk < 1 || H < 0 || ldy < H)
        return NVFP4_ERR_INVALID_ARG;
    if (y_dtype != NVFP4_OUT_F32 && y_dtype != NVFP4_OUT_BF16) return NVFP4_ERR_INVALID_ARG;
    if (H % 8 || ldy % 8) return NVFP4_ERR_UNSUPPORTED;
    if (!aligned16(y) || !aligned16(out)) return NVFP4_ERR_ALIGNMENT;
    if (T == 0 || H == 0) return NVFP4_OK;
    NVFP4_CHECK_INIT();
    int64_t total = (int64_t)T * (H / 8);
    int64_t blocks = (total + 255) / 256, cap = (int64_t)sm_count() * 8;
    if (blocks > cap) blocks = cap;
    cudaStream_t st = (cudaStream_t)stream;
    if (y_dtype == NVFP4_OUT_BF16 && topk <= kCombineMaxK)
        combine_bf16_kernel<<<(unsigned)blocks, 256, 0, st>>>((const uint16_t *)y, ldy, dst_row, weights, T, topk, H,
                                                              out);
    else if (y_dtype == NVFP4_OUT_BF16)
        combine_kernel<true><<<(unsigned)blocks, 256, 0, st>>>(y, ldy, dst_row, weights, T, topk, H, out);
    else
        combine_kernel<false><<<(unsigned)blocks, 256, 0, st>>>(y, ldy, dst_row, weights, T, topk, H, out);
    return launch_status("combine_kernel");
}
