// abi.cu -- status strings, device check and TMA descriptor encoding.
#include <cudaTypedefs.h>
#include <stdio.h>
#include <string.h>

#include "common.cuh"

namespace nvfp4 {

static thread_local char g_last_error[256] = "";

void set_last_error(const char *what, cudaError_t e) {
    snprintf(g_last_error, sizeof(g_last_error), "%s: %s", what, cudaGetErrorString(e));
}

void set_last_error_text(const char *text) { snprintf(g_last_error, sizeof(g_last_error), "%s", text); }

static PFN_cuTensorMapEncodeTiled_v12000 g_encode = nullptr;
static int g_dev_ok[64];   // 0 unknown, 1 ok, 2 not sm_103
static int g_dev_sms[64];

int ensure_init() {
    int dev = 0;
    cudaError_t e = cudaGetDevice(&dev);
    if (e != cudaSuccess) {
        set_last_error("cudaGetDevice", e);
        return NVFP4_ERR_ARCH;
    }
    if (dev < 0 || dev >= 64) {
        set_last_error_text("the library supports device ordinals 0..63");
        return NVFP4_ERR_ARCH;
    }
    if (g_dev_ok[dev] == 0) {
        int major = 0, minor = 0, sms = 0;
        if (cudaDeviceGetAttribute(&major, cudaDevAttrComputeCapabilityMajor, dev) != cudaSuccess ||
            cudaDeviceGetAttribute(&minor, cudaDevAttrComputeCapabilityMinor, dev) != cudaSuccess ||
            cudaDeviceGetAttribute(&sms, cudaDevAttrMultiProcessorCount, dev) != cudaSuccess) {
            set_last_error("cudaDeviceGetAttribute", cudaGetLastError());
            return NVFP4_ERR_ARCH;
        }
        g_dev_sms[dev] = sms;
        g_dev_ok[dev] = (major == 10 && minor == 3) ? 1 : 2;
    }
    if (g_dev_ok[dev] != 1) return NVFP4_ERR_ARCH;
    if (!g_encode) {
        void *fn = nullptr;
        cudaDriverEntryPointQueryResult q;
        e = cudaGetDriverEntryPointByVersion("cuTensorMapEncodeTiled", &fn, 12000, cudaEnableDefault, &q);
        if (e != cudaSuccess || q != cudaDriverEntryPointSuccess || !fn) {
            set_last_error("cudaGetDriverEntryPointByVersion(cuTensorMapEncodeTiled)", e);
            return NVFP4_ERR_CUDA;
        }
        g_encode = reinterpret_cast<PFN_cuTensorMapEncodeTiled_v12000>(fn);
    }
    return NVFP4_OK;
}

void *current_context() {
    static PFN_cuCtxGetCurrent_v4000 get = nullptr;
    if (!get) {
        void *fn = nullptr;
        cudaDriverEntryPointQueryResult q;
        if (cudaGetDriverEntryPointByVersion("cuCtxGetCurrent", &fn, 4000, cudaEnableDefault, &q) != cudaSuccess ||
            q != cudaDriverEntryPointSuccess || !fn)
            return nullptr;
        get = reinterpret_cast<PFN_cuCtxGetCurrent_v4000>(fn);
    }
    CUcontext c = nullptr;
    return get(&c) == CUDA_SUCCESS ? (void *)c : nullptr;
}

int sm_count() {
    int dev = 0;
    cudaGetDevice(&dev);
    return (dev >= 0 && dev < 64 && g_dev_sms[dev] > 0) ? g_dev_sms[dev] : 148;
}

int encode_tmap_2d(CUtensorMap *map, CUtensorMapDataType dtype, void *base, uint64_t inner,
                   uint64_t outer, uint64_t row_bytes, uint32_t box_inner, uint32_t box_outer,
                   CUtensorMapSwizzle swz) {
    cuuint64_t dims[2] = {inner, outer};
    cuuint64_t strides[1] = {row_bytes};
    cuuint32_t box[2] = {box_inner, box_outer};
    cuuint32_t estr[2] = {1, 1};
    CUresult r = g_encode(map, dtype, 2, base, dims, strides, box, estr, CU_TENSOR_MAP_INTERLEAVE_NONE,
                          swz, CU_TENSOR_MAP_L2_PROMOTION_L2_256B, CU_TENSOR_MAP_FLOAT_OOB_FILL_NONE);
    if (r != CUDA_SUCCESS) {
        snprintf(g_last_error, sizeof(g_last_error), "cuTensorMapEncodeTiled failed (%d)", (int)r);
        return NVFP4_ERR_CUDA;
    }
    return NVFP4_OK;
}

}  // namespace nvfp4

extern "C" const char *nvfp4_status_str(int s) {
    switch (s) {
        case NVFP4_OK: return "NVFP4_OK";
        case NVFP4_ERR_INVALID_ARG: return "NVFP4_ERR_INVALID_ARG";
        case NVFP4_ERR_UNSUPPORTED: return "NVFP4_ERR_UNSUPPORTED";
        case NVFP4_ERR_ALIGNMENT: return "NVFP4_ERR_ALIGNMENT";
        case NVFP4_ERR_CUDA: return "NVFP4_ERR_CUDA";
        case NVFP4_ERR_TIMEOUT: return "NVFP4_ERR_TIMEOUT";
        case NVFP4_ERR_NONFINITE: return "NVFP4_ERR_NONFINITE";
        case NVFP4_ERR_ARCH: return "NVFP4_ERR_ARCH";
        default: return "NVFP4_ERR_UNKNOWN";
    }
}

extern "C" int nvfp4_init(void) { return nvfp4::ensure_init(); }

extern "C" const char *nvfp4_last_error(void) { return nvfp4::g_last_error; }

// ---------------------------------------------------------------- self test

namespace nvfp4 {
__global__ void wait_timeout_kernel(uint64_t limit_ns, int32_t *dev_status) {
    __shared__ uint64_t bar;
    if (threadIdx.x == 0) {
        mbar_init(&bar, 1);
        fence_barrier_init();
    }
    __syncthreads();
    if (threadIdx.x == 0) {
        // Nothing ever arrives on `bar`: phase 0 never completes.
        if (!mbar_wait_bounded(&bar, 0, limit_ns)) report(dev_status, NVFP4_ERR_TIMEOUT);
    }
}
}  // namespace nvfp4

extern "C" int nvfp4_selftest_wait_timeout(int32_t limit_us, int32_t *dev_status, void *stream) {
    if (limit_us < 1 || limit_us > 10000000 || !dev_status) return NVFP4_ERR_INVALID_ARG;
    NVFP4_CHECK_INIT();
    nvfp4::wait_timeout_kernel<<<1, 32, 0, (cudaStream_t)stream>>>((uint64_t)limit_us * 1000u, dev_status);
    return nvfp4::launch_status("wait_timeout_kernel");
}
