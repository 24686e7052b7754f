// Library-wide pieces of the C ABI: status strings, the device error word and
// the TMA descriptor encoder shared by the kernels.
#include <mutex>

#include "bi_internal.h"
#include "bi_ptx.cuh"

namespace {

// One error word per device.  Kernels record the first device-side problem
// here (see bi_get_device_error); it is a flag, not part of any arithmetic.
__device__ uint32_t g_bi_error_word = 0;

constexpr int kMaxDevices = 64;
std::mutex g_mu;
uint32_t* g_err_ptr[kMaxDevices] = {};
int g_sm_count[kMaxDevices] = {};

using EncodeTiledFn = CUresult (*)(CUtensorMap*, CUtensorMapDataType, cuuint32_t, void*,
                                   const cuuint64_t*, const cuuint64_t*, const cuuint32_t*,
                                   const cuuint32_t*, CUtensorMapInterleave, CUtensorMapSwizzle,
                                   CUtensorMapL2promotion, CUtensorMapFloatOOBfill);
EncodeTiledFn g_encode = nullptr;

int current_device() {
    int dev = -1;
    if (cudaGetDevice(&dev) != cudaSuccess) return -1;
    return (dev >= 0 && dev < kMaxDevices) ? dev : -1;
}

// One thread waits, through the same bounded wait every kernel uses, on an
// mbarrier that nothing will ever arrive on; the wait must give up after
// `limit_ns` and record BI_ERR_DEVICE_TIMEOUT.
__global__ void selftest_wait_kernel(uint32_t* err, uint64_t limit_ns) {
    __shared__ uint64_t bar;
    if (threadIdx.x == 0) {
        bi::mbar_init(&bar, 1);
        bi::fence_mbar_init();
    }
    __syncthreads();
    if (threadIdx.x == 0 && !bi::mbar_wait_for(&bar, 0, limit_ns))
        bi::report_error(err, bi::kErrTimeout | bi::kWhereSelftest);
}

}  // namespace

namespace bi {

uint32_t* device_error_word() {
    int dev = current_device();
    if (dev < 0) return nullptr;
    std::lock_guard<std::mutex> lk(g_mu);
    if (!g_err_ptr[dev]) {
        void* p = nullptr;
        if (cudaGetSymbolAddress(&p, g_bi_error_word) != cudaSuccess) return nullptr;
        g_err_ptr[dev] = static_cast<uint32_t*>(p);
    }
    return g_err_ptr[dev];
}

int sm_count() {
    int dev = current_device();
    if (dev < 0) return 0;
    std::lock_guard<std::mutex> lk(g_mu);
    if (!g_sm_count[dev]) {
        int n = 0;
        if (cudaDeviceGetAttribute(&n, cudaDevAttrMultiProcessorCount, dev) != cudaSuccess)
            return 0;
        g_sm_count[dev] = n;
    }
    return g_sm_count[dev];
}

CUresult encode_tensor_map_2d(CUtensorMap* map, const void* base, uint64_t inner_elems,
                              uint64_t outer_rows, uint64_t row_stride_bytes, uint32_t box_inner,
                              uint32_t box_outer) {
    {
        std::lock_guard<std::mutex> lk(g_mu);
        if (!g_encode) {
            void* fn = nullptr;
            cudaDriverEntryPointQueryResult q{};
            if (cudaGetDriverEntryPointByVersion("cuTensorMapEncodeTiled", &fn, 12000,
                                                 cudaEnableDefault, &q) != cudaSuccess ||
                q != cudaDriverEntryPointSuccess || !fn)
                return CUDA_ERROR_NOT_FOUND;
            g_encode = reinterpret_cast<EncodeTiledFn>(fn);
        }
    }
    cuuint64_t dims[2] = {inner_elems, outer_rows};
    cuuint64_t strides[1] = {row_stride_bytes};
    cuuint32_t box[2] = {box_inner, box_outer};
    cuuint32_t estr[2] = {1, 1};
    return g_encode(map, CU_TENSOR_MAP_DATA_TYPE_BFLOAT16, 2, const_cast<void*>(base), dims,
                    strides, box, estr, CU_TENSOR_MAP_INTERLEAVE_NONE,
                    CU_TENSOR_MAP_SWIZZLE_128B, CU_TENSOR_MAP_L2_PROMOTION_L2_256B,
                    CU_TENSOR_MAP_FLOAT_OOB_FILL_NONE);
}

CUresult encode_page_map(CUtensorMap* map, const void* base, uint64_t rows) {
    CUtensorMap probe;
    const CUresult r = encode_tensor_map_2d(&probe, base, 128, rows, 256, 64, 16);  // resolves the entry point
    if (r != CUDA_SUCCESS) return r;
    // dims: 64 dims of a half-row (inner), token rows (256-byte stride), the
    // two halves of a row (128-byte stride); one box = a 16-row page block,
    // stored half 0 then half 1, as two 16 x 64 boxes would be
    cuuint64_t dims[3] = {64, rows, 2};
    cuuint64_t strides[2] = {256, 128};
    cuuint32_t box[3] = {64, 16, 2};
    cuuint32_t estr[3] = {1, 1, 1};
    return g_encode(map, CU_TENSOR_MAP_DATA_TYPE_BFLOAT16, 3, const_cast<void*>(base), dims,
                    strides, box, estr, CU_TENSOR_MAP_INTERLEAVE_NONE,
                    CU_TENSOR_MAP_SWIZZLE_128B, CU_TENSOR_MAP_L2_PROMOTION_L2_256B,
                    CU_TENSOR_MAP_FLOAT_OOB_FILL_NONE);
}

CUresult encode_q_map(CUtensorMap* map, const void* base, uint64_t T, uint64_t Hq,
                      uint32_t box_heads, uint32_t box_rows) {
    CUtensorMap probe;
    const CUresult r = encode_tensor_map_2d(&probe, base, 128, T * Hq, 256, 64, 1);  // resolves the entry point
    if (r != CUDA_SUCCESS) return r;
    cuuint64_t dims[3] = {128, Hq, T};
    cuuint64_t strides[2] = {256, Hq * 256};
    cuuint32_t box[3] = {64, box_heads, box_rows};
    cuuint32_t estr[3] = {1, 1, 1};
    return g_encode(map, CU_TENSOR_MAP_DATA_TYPE_BFLOAT16, 3, const_cast<void*>(base), dims,
                    strides, box, estr, CU_TENSOR_MAP_INTERLEAVE_NONE,
                    CU_TENSOR_MAP_SWIZZLE_128B, CU_TENSOR_MAP_L2_PROMOTION_L2_256B,
                    CU_TENSOR_MAP_FLOAT_OOB_FILL_NONE);
}

}  // namespace bi

extern "C" {

int bi_abi_version(void) { return BI_ABI_VERSION; }

const char* bi_status_string(bi_status s) {
    switch (s) {
        case BI_OK: return "BI_OK";
        case BI_ERR_INVALID_ARG: return "BI_ERR_INVALID_ARG";
        case BI_ERR_UNSUPPORTED_SHAPE: return "BI_ERR_UNSUPPORTED_SHAPE";
        case BI_ERR_MISALIGNED: return "BI_ERR_MISALIGNED";
        case BI_ERR_WORKSPACE_TOO_SMALL: return "BI_ERR_WORKSPACE_TOO_SMALL";
        case BI_ERR_CUDA: return "BI_ERR_CUDA";
        case BI_ERR_DEVICE_TIMEOUT: return "BI_ERR_DEVICE_TIMEOUT";
        case BI_ERR_DEVICE_BAD_INPUT: return "BI_ERR_DEVICE_BAD_INPUT";
    }
    return "BI_ERR_UNKNOWN";
}

bi_status bi_selftest_wait_timeout(int32_t limit_us, cudaStream_t stream) {
    if (limit_us < 1 || limit_us > 2000000) return BI_ERR_INVALID_ARG;
    uint32_t* err = bi::device_error_word();
    if (!err) return BI_ERR_CUDA;
    selftest_wait_kernel<<<1, 32, 0, stream>>>(err, static_cast<uint64_t>(limit_us) * 1000u);
    return cudaGetLastError() == cudaSuccess ? BI_OK : BI_ERR_CUDA;
}

bi_status bi_get_device_error(cudaStream_t stream) {
    if (cudaStreamSynchronize(stream) != cudaSuccess) return BI_ERR_CUDA;
    uint32_t* p = bi::device_error_word();
    if (!p) return BI_ERR_CUDA;
    uint32_t v = 0;
    if (cudaMemcpy(&v, p, sizeof v, cudaMemcpyDeviceToHost) != cudaSuccess) return BI_ERR_CUDA;
    if (v != 0) {
        uint32_t zero = 0;
        if (cudaMemcpy(p, &zero, sizeof zero, cudaMemcpyHostToDevice) != cudaSuccess)
            return BI_ERR_CUDA;
    }
    switch (v & 0xffu) {
        case 0: return BI_OK;
        case BI_ERR_DEVICE_TIMEOUT: return BI_ERR_DEVICE_TIMEOUT;
        case BI_ERR_DEVICE_BAD_INPUT: return BI_ERR_DEVICE_BAD_INPUT;
    }
    return BI_ERR_CUDA;
}

}  // extern "C"
