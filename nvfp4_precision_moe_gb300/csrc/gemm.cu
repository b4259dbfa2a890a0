// gemm.cu -- the grouped-GEMM entry points: argument checks, tensor maps, and
// the choice between the two tcgen05 pipelines (gemm_single.cu: one CTA per
// 128x256 tile; gemm_pair.cu: a CTA pair per 256x256 tile).  By default each
// kind runs on the pipeline measured faster for it on GB300 -- FP4 (W4A4 +
// RAC) on the single-CTA pipeline, BF16 on the pair pipeline;
// nvfp4_gemm_pipeline() overrides the choice process-wide.
#include <atomic>

#include "gemm_common.cuh"

using namespace nvfp4;

namespace {
std::atomic<int> g_pipeline{NVFP4_PIPELINE_AUTO};

bool use_pair(bool fp4) {
    const int which = g_pipeline.load(std::memory_order_relaxed);
    if (which == NVFP4_PIPELINE_SINGLE) return false;
    if (which == NVFP4_PIPELINE_PAIR) return true;
    return !fp4;
}
}  // namespace

extern "C" int nvfp4_gemm_pipeline(int32_t which, int32_t *previous) {
    if (which != NVFP4_PIPELINE_AUTO && which != NVFP4_PIPELINE_SINGLE && which != NVFP4_PIPELINE_PAIR)
        return NVFP4_ERR_INVALID_ARG;
    const int prev = g_pipeline.exchange(which);
    if (previous) *previous = prev;
    return NVFP4_OK;
}

extern "C" int nvfp4_w4a4_rac_grouped_gemm(const uint8_t *a_codes, const uint8_t *a_scales, const void *a_resid,
                                           const float *gs_a, const uint8_t *w_codes, const uint8_t *w_scales,
                                           const float *gs_w, const void *w_sel, int32_t k, const int32_t *offsets,
                                           int32_t E, int64_t rows_cap, int64_t N, int64_t K, int32_t epilogue,
                                           int32_t out_dtype, void *y, int64_t ldy, float *amax_out,
                                           int32_t *dev_status, void *stream) {
    if (!a_codes || !a_scales || !gs_a || !w_codes || !w_scales || !gs_w || !offsets || !y || E < 1 ||
        rows_cap < 0 || N < 0 || K < 0 || k < 0)
        return NVFP4_ERR_INVALID_ARG;
    if (k > 0 && (!a_resid || !w_sel)) return NVFP4_ERR_INVALID_ARG;
    if (epilogue != NVFP4_EPI_NONE && epilogue != NVFP4_EPI_SWIGLU) return NVFP4_ERR_INVALID_ARG;
    if (out_dtype != NVFP4_OUT_F32 && out_dtype != NVFP4_OUT_BF16) return NVFP4_ERR_INVALID_ARG;
    if (epilogue == NVFP4_EPI_SWIGLU && out_dtype != NVFP4_OUT_BF16) return NVFP4_ERR_INVALID_ARG;
    const int64_t ncols = epilogue == NVFP4_EPI_SWIGLU ? N / 2 : N;
    if (ldy < ncols) return NVFP4_ERR_INVALID_ARG;
    if (K % 256 || N % 256 || k % 16 || k > K || E > kMaxExperts || rows_cap % 128 || rows_cap > (1ll << 31) ||
        (int64_t)E * N > (1ll << 31))
        return NVFP4_ERR_UNSUPPORTED;
    if (!aligned16(a_codes) || !aligned16(a_scales) || !aligned16(w_codes) || !aligned16(w_scales) || !aligned16(y) ||
        (a_resid && !aligned16(a_resid)) || (w_sel && !aligned16(w_sel)) || ldy % 8)
        return NVFP4_ERR_ALIGNMENT;
    NVFP4_CHECK_INIT();
    if (amax_out) {
        cudaError_t e = cudaMemsetAsync(amax_out, 0, sizeof(float), (cudaStream_t)stream);
        if (e != cudaSuccess) {
            set_last_error("cudaMemsetAsync(amax_out)", e);
            return NVFP4_ERR_CUDA;
        }
    }
    if (rows_cap == 0 || N == 0 || K == 0) return NVFP4_OK;
    const bool pair = use_pair(true);
    const uint32_t brows = pair ? 128 : 256;  // B rows per copy: this CTA's half, or the whole tile

    CUtensorMap tA, tB, tR, tW, tSA, tSB;
    int s = encode_tmap_2d(&tA, CU_TENSOR_MAP_DATA_TYPE_UINT8, (void *)a_codes, K / 2, rows_cap, K / 2, 128, 128,
                           CU_TENSOR_MAP_SWIZZLE_128B);
    if (s == NVFP4_OK)
        s = encode_tmap_2d(&tB, CU_TENSOR_MAP_DATA_TYPE_UINT8, (void *)w_codes, K / 2, (uint64_t)E * N, K / 2, 128,
                           brows, CU_TENSOR_MAP_SWIZZLE_128B);
    if (s == NVFP4_OK && k > 0) {
        s = encode_tmap_2d(&tR, CU_TENSOR_MAP_DATA_TYPE_BFLOAT16, (void *)a_resid, k, rows_cap, 2 * k, 64, 128,
                           CU_TENSOR_MAP_SWIZZLE_128B);
        if (s == NVFP4_OK)
            s = encode_tmap_2d(&tW, CU_TENSOR_MAP_DATA_TYPE_BFLOAT16, (void *)w_sel, k, (uint64_t)E * N, 2 * k, 64,
                               brows, CU_TENSOR_MAP_SWIZZLE_128B);
    } else {
        tR = tA;
        tW = tB;
    }
    // the scale tensors as rows of 256 bytes, a 2048-byte scale tile in 8 rows; the pair
    // pipeline copies them with the operands
    const int64_t kslices = K / 256;
    if (s == NVFP4_OK && pair)
        s = encode_tmap_2d(&tSA, CU_TENSOR_MAP_DATA_TYPE_UINT8, (void *)a_scales, 256,
                           (uint64_t)(rows_cap / 128) * kslices * 8, 256, 256, 8, CU_TENSOR_MAP_SWIZZLE_NONE);
    if (s == NVFP4_OK && pair)
        s = encode_tmap_2d(&tSB, CU_TENSOR_MAP_DATA_TYPE_UINT8, (void *)w_scales, 256,
                           (uint64_t)E * (N / 128) * kslices * 8, 256, 256, 8, CU_TENSOR_MAP_SWIZZLE_NONE);
    if (s != NVFP4_OK) return s;

    GemmParams p{};
    p.a_codes_base = a_codes;
    p.a_scales = a_scales;
    p.w_scales = w_scales;
    p.gs_a = gs_a;
    p.gs_w = gs_w;
    p.offsets = offsets;
    p.rows_cap = (int32_t)rows_cap;
    p.E = E;
    p.k = k;
    p.N = N;
    p.K = K;
    p.epilogue = epilogue;
    p.out_dtype = out_dtype;
    p.y = y;
    p.ldy = ldy;
    p.vec32 = (reinterpret_cast<uintptr_t>(y) % 32 == 0) &&
              (ldy * (out_dtype == NVFP4_OUT_F32 ? 4 : 2)) % 32 == 0;
    p.amax_out = amax_out;
    p.dev_status = dev_status;
    return pair ? launch_pair_gemm<true>(tA, tB, tR, tW, tSA, tSB, p, rows_cap, N, (cudaStream_t)stream)
                : launch_single_gemm<true>(tA, tB, tR, tW, p, rows_cap, N, (cudaStream_t)stream);
}

extern "C" int nvfp4_bf16_grouped_gemm(const void *x, const void *w_hat, const int32_t *offsets, int32_t E,
                                       int64_t rows_cap, int64_t N, int64_t K, int32_t out_dtype, int32_t epilogue,
                                       void *y, int64_t ldy, void *gu, int32_t *dev_status, void *stream) {
    if (!x || !w_hat || !offsets || !y || E < 1 || rows_cap < 0 || N < 0 || K < 0) return NVFP4_ERR_INVALID_ARG;
    if (out_dtype != NVFP4_OUT_F32 && out_dtype != NVFP4_OUT_BF16) return NVFP4_ERR_INVALID_ARG;
    const bool swiglu = epilogue == NVFP4_EPI_SWIGLU || epilogue == NVFP4_EPI_SWIGLU_SAVE;
    if (epilogue != NVFP4_EPI_NONE && !swiglu) return NVFP4_ERR_INVALID_ARG;
    if (swiglu && out_dtype != NVFP4_OUT_BF16) return NVFP4_ERR_INVALID_ARG;
    if ((epilogue == NVFP4_EPI_SWIGLU_SAVE) != (gu != nullptr)) return NVFP4_ERR_INVALID_ARG;
    if (ldy < (swiglu ? N / 2 : N)) return NVFP4_ERR_INVALID_ARG;
    if (K % 64 || N % 256 || E > kMaxExperts || rows_cap % 128 || rows_cap > (1ll << 31) || (int64_t)E * N > (1ll << 31))
        return NVFP4_ERR_UNSUPPORTED;
    if (!aligned16(x) || !aligned16(w_hat) || !aligned16(y) || ldy % 8 || !aligned16(gu)) return NVFP4_ERR_ALIGNMENT;
    if (rows_cap == 0 || N == 0 || K == 0) return NVFP4_OK;
    NVFP4_CHECK_INIT();
    CUtensorMap tA, tB;
    int s = encode_tmap_2d(&tA, CU_TENSOR_MAP_DATA_TYPE_BFLOAT16, (void *)x, K, rows_cap, 2 * K, 64, 128,
                       CU_TENSOR_MAP_SWIZZLE_128B);
    if (s == NVFP4_OK)
        s = encode_tmap_2d(&tB, CU_TENSOR_MAP_DATA_TYPE_BFLOAT16, (void *)w_hat, K, (uint64_t)E * N, 2 * K, 64, 128,
                           CU_TENSOR_MAP_SWIZZLE_128B);
    if (s != NVFP4_OK) return s;
    GemmParams p{};
    p.a_codes_base = (const uint8_t *)x;
    p.epilogue = epilogue;
    p.offsets = offsets;
    p.rows_cap = (int32_t)rows_cap;
    p.E = E;
    p.N = N;
    p.K = K;
    p.out_dtype = out_dtype;
    p.y = y;
    p.ldy = ldy;
    p.vec32 = (reinterpret_cast<uintptr_t>(y) % 32 == 0) &&
              (ldy * (out_dtype == NVFP4_OUT_F32 ? 4 : 2)) % 32 == 0;
    p.gu_out = (uint16_t *)gu;
    p.gu_vec32 = (reinterpret_cast<uintptr_t>(gu) % 32 == 0) && (N * 2) % 32 == 0;
    p.dev_status = dev_status;
    return use_pair(false) ? launch_pair_gemm<false>(tA, tB, tA, tB, tA, tB, p, rows_cap, N, (cudaStream_t)stream)
                           : launch_single_gemm<false>(tA, tB, tA, tB, p, rows_cap, N, (cudaStream_t)stream);
}

extern "C" int nvfp4_bf16_grouped_gemm_dgrad(const void *dy, const void *w_hat, const int32_t *offsets, int32_t E,
                                             int64_t rows_cap, int64_t N, int64_t K, int32_t out_dtype,
                                             int32_t epilogue, const void *gu, void *y, int64_t ldy,
                                             int32_t *dev_status, void *stream) {
    if (!dy || !w_hat || !offsets || !y || E < 1 || rows_cap < 0 || N < 0 || K < 0) return NVFP4_ERR_INVALID_ARG;
    if (out_dtype != NVFP4_OUT_F32 && out_dtype != NVFP4_OUT_BF16) return NVFP4_ERR_INVALID_ARG;
    if (epilogue != NVFP4_EPI_NONE && epilogue != NVFP4_EPI_SWIGLU_BWD) return NVFP4_ERR_INVALID_ARG;
    const bool bwd = epilogue == NVFP4_EPI_SWIGLU_BWD;
    if (bwd && (!gu || out_dtype != NVFP4_OUT_BF16)) return NVFP4_ERR_INVALID_ARG;
    if (ldy < (bwd ? 2 * N : N)) return NVFP4_ERR_INVALID_ARG;
    if (K % 64 || N % 256 || E > kMaxExperts || rows_cap % 128 || rows_cap > (1ll << 31) || (int64_t)E * K > (1ll << 31))
        return NVFP4_ERR_UNSUPPORTED;
    if (!aligned16(dy) || !aligned16(w_hat) || !aligned16(y) || ldy % 8 || (bwd && !aligned16(gu)))
        return NVFP4_ERR_ALIGNMENT;
    if (rows_cap == 0 || N == 0 || K == 0) return NVFP4_OK;
    NVFP4_CHECK_INIT();
    // A: dy rows, K-major; B: the experts' [K, N] blocks stacked, MN-major boxes of 64 columns x 64 K-rows
    CUtensorMap tA, tB;
    int s = encode_tmap_2d(&tA, CU_TENSOR_MAP_DATA_TYPE_BFLOAT16, (void *)dy, K, rows_cap, 2 * K, 64, 128,
                           CU_TENSOR_MAP_SWIZZLE_128B);
    if (s == NVFP4_OK)
        s = encode_tmap_2d(&tB, CU_TENSOR_MAP_DATA_TYPE_BFLOAT16, (void *)w_hat, N, (uint64_t)E * K, 2 * N, 64, 64,
                           CU_TENSOR_MAP_SWIZZLE_128B);
    if (s != NVFP4_OK) return s;
    GemmParams p{};
    p.a_codes_base = (const uint8_t *)dy;
    p.epilogue = epilogue;
    p.gu = bwd ? (const uint16_t *)gu : nullptr;
    p.offsets = offsets;
    p.rows_cap = (int32_t)rows_cap;
    p.E = E;
    p.N = N;
    p.K = K;
    p.b_mn = 1;
    p.out_dtype = out_dtype;
    p.y = y;
    p.ldy = ldy;
    p.vec32 = (reinterpret_cast<uintptr_t>(y) % 32 == 0) &&
              (ldy * (out_dtype == NVFP4_OUT_F32 ? 4 : 2)) % 32 == 0;
    p.dev_status = dev_status;
    return use_pair(false) ? launch_pair_gemm<false>(tA, tB, tA, tB, tA, tB, p, rows_cap, N, (cudaStream_t)stream)
                           : launch_single_gemm<false>(tA, tB, tA, tB, p, rows_cap, N, (cudaStream_t)stream);
}

namespace {
// The weight-gradient GEMM with its operands either transposed (K-major: a [M, R], b [N, R]) or
// as the routed rows themselves (MN-major: a [R, M], b [R, N]).
int wgrad_gemm(const void *a, const void *b, bool rows_major, const int32_t *offsets, int32_t E, int64_t R, int64_t M,
               int64_t N, int32_t out_dtype, void *dw, int32_t *dev_status, void *stream) {
    if (!a || !b || !offsets || !dw || E < 1 || R < 0 || M < 0 || N < 0) return NVFP4_ERR_INVALID_ARG;
    if (out_dtype != NVFP4_OUT_F32 && out_dtype != NVFP4_OUT_BF16) return NVFP4_ERR_INVALID_ARG;
    if (M % 128 || N % 256 || R % 128 || E > kMaxExperts || R > (1ll << 31) || (int64_t)E * M > (1ll << 31))
        return NVFP4_ERR_UNSUPPORTED;
    if (!aligned16(a) || !aligned16(b) || !aligned16(dw)) return NVFP4_ERR_ALIGNMENT;
    if (M == 0 || N == 0) return NVFP4_OK;
    NVFP4_CHECK_INIT();
    if (R == 0) {  // no routed rows at all: every gradient is zero
        const cudaError_t e = cudaMemsetAsync(dw, 0, (size_t)E * M * N * (out_dtype == NVFP4_OUT_F32 ? 4 : 2),
                                              (cudaStream_t)stream);
        if (e != cudaSuccess) {
            set_last_error("cudaMemsetAsync(dw)", e);
            return NVFP4_ERR_CUDA;
        }
        return NVFP4_OK;
    }
    CUtensorMap tA, tB;
    int s;
    if (rows_major) {  // boxes of 64 columns x 64 rows
        s = encode_tmap_2d(&tA, CU_TENSOR_MAP_DATA_TYPE_BFLOAT16, (void *)a, M, R, 2 * M, 64, 64,
                           CU_TENSOR_MAP_SWIZZLE_128B);
        if (s == NVFP4_OK)
            s = encode_tmap_2d(&tB, CU_TENSOR_MAP_DATA_TYPE_BFLOAT16, (void *)b, N, R, 2 * N, 64, 64,
                               CU_TENSOR_MAP_SWIZZLE_128B);
    } else {  // boxes of 64 reduction elements x 128 rows
        s = encode_tmap_2d(&tA, CU_TENSOR_MAP_DATA_TYPE_BFLOAT16, (void *)a, R, M, 2 * R, 64, 128,
                           CU_TENSOR_MAP_SWIZZLE_128B);
        if (s == NVFP4_OK)
            s = encode_tmap_2d(&tB, CU_TENSOR_MAP_DATA_TYPE_BFLOAT16, (void *)b, R, N, 2 * R, 64, 128,
                               CU_TENSOR_MAP_SWIZZLE_128B);
    }
    if (s != NVFP4_OK) return s;
    GemmParams p{};
    p.wgrad = 1;
    p.wgrad_f32 = out_dtype == NVFP4_OUT_F32 ? 1 : 0;
    p.a_mn = rows_major ? 1 : 0;
    p.b_mn = rows_major ? 1 : 0;
    p.M = M;
    p.offsets = offsets;
    p.rows_cap = (int32_t)R;
    p.E = E;
    p.N = N;
    p.K = R;
    p.epilogue = NVFP4_EPI_NONE;
    p.out_dtype = out_dtype;
    p.y = dw;
    p.ldy = N;
    p.vec32 = (reinterpret_cast<uintptr_t>(dw) % 32 == 0) && (N * (out_dtype == NVFP4_OUT_F32 ? 4 : 2)) % 32 == 0;
    p.dev_status = dev_status;
    // the weight-gradient mode exists on the single-CTA pipeline only
    return launch_single_gemm<false>(tA, tB, tA, tB, p, (int64_t)E * M, N, (cudaStream_t)stream);
}
}  // namespace

extern "C" int nvfp4_bf16_grouped_gemm_wgrad(const void *a_t, const void *b_t, const int32_t *offsets, int32_t E,
                                             int64_t R, int64_t M, int64_t N, int32_t out_dtype, void *dw,
                                             int32_t *dev_status, void *stream) {
    return wgrad_gemm(a_t, b_t, false, offsets, E, R, M, N, out_dtype, dw, dev_status, stream);
}

extern "C" int nvfp4_bf16_grouped_gemm_wgrad_rows(const void *a, const void *b, const int32_t *offsets, int32_t E,
                                                  int64_t R, int64_t M, int64_t N, int32_t out_dtype, void *dw,
                                                  int32_t *dev_status, void *stream) {
    return wgrad_gemm(a, b, true, offsets, E, R, M, N, out_dtype, dw, dev_status, stream);
}
