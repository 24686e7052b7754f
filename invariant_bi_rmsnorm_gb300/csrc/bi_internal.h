// Declarations shared by the library's translation units (not part of the ABI).
#pragma once
#include <cstdint>

#include <cuda.h>  // CUtensorMap and its enums only; libcuda is not linked
#include <cuda_runtime.h>

#include "bi.h"

namespace bi {

// Limits of every bounded barrier wait: about two seconds of wall clock
// (a healthy wait lasts microseconds), and a poll count as a backstop in case
// the clock does not advance.
constexpr uint64_t kWaitNs = 2000000000ull;
constexpr uint32_t kWaitPollLimit = 1u << 28;
// After a wait has timed out, a kernel gives each copy or MMA it issued and
// never saw complete this much more time before it exits (its shared memory
// and TMEM must not be released under an operation still in flight).
constexpr uint64_t kDrainNs = 20000000ull;

// Device error word values (low byte = bi_status, next byte = where).
enum : uint32_t {
    kErrTimeout = BI_ERR_DEVICE_TIMEOUT,
    kErrBadInput = BI_ERR_DEVICE_BAD_INPUT,
};
enum : uint32_t {
    kWhereRmsnorm = 1u << 8,
    kWhereGemmProducer = 2u << 8,
    kWhereGemmMma = 3u << 8,
    kWhereGemmEpilogue = 4u << 8,
    kWhereAttnSplit = 5u << 8,
    kWhereAttnMerge = 6u << 8,
    kWhereSelftest = 7u << 8,
    kWhereDecoderOps = 8u << 8,
};

// Device address of the current device's error word (nullptr on failure).
uint32_t* device_error_word();

// Multiprocessor count of the current device (cached per device).
int sm_count();

// cuTensorMapEncodeTiled, resolved through the runtime's driver entry point
// so the library does not link libcuda.  Returns CUDA_SUCCESS or an error.
CUresult encode_tensor_map_2d(CUtensorMap* map, const void* base, uint64_t inner_elems,
                              uint64_t outer_rows, uint64_t row_stride_bytes, uint32_t box_inner,
                              uint32_t box_outer);

// The K or V cache [num_pages * Hkv * 16 rows][128] as a 3-D map whose box is
// one 16-row page block in the two-half, 128-byte-swizzled layout of two
// 16 x 64 boxes (one copy instead of two).
CUresult encode_page_map(CUtensorMap* map, const void* base, uint64_t rows);

// Query rows q[T][Hq][128] as a 3-D map (dims, heads, rows) whose box is
// `box_heads` consecutive heads of `box_rows` consecutive rows over 64 dims,
// 128-byte swizzled: one box lands as box_rows * box_heads rows of 128 bytes
// in (row, head) order.
CUresult encode_q_map(CUtensorMap* map, const void* base, uint64_t T, uint64_t Hq,
                      uint32_t box_heads, uint32_t box_rows);

inline bool aligned16(const void* p) { return (reinterpret_cast<uintptr_t>(p) & 15u) == 0; }

// Launch with programmatic stream serialization: the grid may be scheduled
// while the previous kernel in the stream finishes.  Every kernel launched
// this way calls launch_dependents() and grid_dependency_wait() (bi_ptx.cuh)
// before it touches global memory.
template <typename... KArgs, typename... Args>
cudaError_t launch_pdl(void (*kernel)(KArgs...), dim3 grid, dim3 block, size_t smem,
                       cudaStream_t stream, Args... args) {
    cudaLaunchConfig_t cfg = {};
    cfg.gridDim = grid;
    cfg.blockDim = block;
    cfg.dynamicSmemBytes = smem;
    cfg.stream = stream;
    cudaLaunchAttribute attr[1];
    attr[0].id = cudaLaunchAttributeProgrammaticStreamSerialization;
    attr[0].val.programmaticStreamSerializationAllowed = 1;
    cfg.attrs = attr;
    cfg.numAttrs = 1;
    return cudaLaunchKernelEx(&cfg, kernel, args...);
}

}  // namespace bi
