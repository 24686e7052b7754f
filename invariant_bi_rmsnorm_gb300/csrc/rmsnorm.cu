// bi_rmsnorm: data-parallel RMSNorm, one row per CTA.
//
// "Defeating Nondeterminism in LLM Inference: The Core Role of Batch
// Invariance", section "1. Batch-Invariant RMSNorm": keeping each row's whole
// reduction inside one core makes its order independent of the batch size;
// splitting one row over several cores at small batch would change it, so
// that is never done here.
//
// Reduction order (a function of `hidden` only):
//   1. thread t owns the 16-byte vectors t, t+T, t+2T, ... of the row
//      (T = threads per CTA); it sums x^2 over its vectors in that order,
//      each vector's 8 elements left to right, with fused multiply-adds;
//   2. each warp folds its 32 partials with an xor butterfly (16,8,4,2,1) and
//      lane 0's result is taken;
//   3. every thread folds the per-warp sums in warp order 0, 1, 2, ...
// (hidden 4096: T = 256 threads, 2 vectors each.)
// Then r = rsqrt(sum / hidden + eps) and y = bf16_rn((x * r) * w) in fp32.
#include <cuda_bf16.h>

#include "bi_internal.h"
#include "bi_ptx.cuh"

namespace {

// 256 threads per row: each thread keeps two 16-byte loads in flight at
// hidden 4096, and 8 rows (CTAs) fit on an SM, which is what it takes to keep
// HBM busy with one row per CTA (512 threads x 1 load left it latency-bound).
constexpr int kMaxThreads = 256;

// Rows resident at once are few (8 CTAs per SM, 8 KiB each at hidden 4096),
// which leaves HBM short of requests. Each CTA therefore asks L2 to fetch the
// input of the row about kPrefetchAheadBytes of input ahead of its own; that
// row's CTA then finds it in L2. A prefetch moves data only: the arithmetic
// and its order are the same whether it hits or not.
// 16 MiB was the best of 0-40 MiB on GB300 at 16384 x 4096, plain and fused.
constexpr int64_t kPrefetchAheadBytes = int64_t{16} << 20;

__device__ __forceinline__ void prefetch_l2(const void* p, uint32_t bytes) {
    asm volatile("cp.async.bulk.prefetch.L2.global [%0], %1;" ::"l"(p), "r"(bytes) : "memory");
}

__device__ __forceinline__ float bf16_lo(uint32_t v) { return __uint_as_float(v << 16); }
__device__ __forceinline__ float bf16_hi(uint32_t v) { return __uint_as_float(v & 0xffff0000u); }

// kAdd: the fused form -- first res = bf16(res + x) (fp32 add, one rounding),
// stored back, then the RMSNorm of that sum with exactly the reduction below.
template <int VPT, bool kAdd>
__global__ void __launch_bounds__(kMaxThreads)
    rmsnorm_kernel(const __nv_bfloat16* x, const __nv_bfloat16* __restrict__ w, __nv_bfloat16* y,
                   int hidden, int64_t ld_x, int64_t ld_y, float eps, __nv_bfloat16* res,
                   int64_t ld_res, int64_t rows, int64_t ahead) {
    bi::launch_dependents();
    bi::grid_dependency_wait();  // nothing global is touched before the previous kernel ends
    __shared__ float warp_sums[kMaxThreads / 32];
    const int nvec = hidden >> 3;
    const int tid = threadIdx.x;
    const int T = blockDim.x;
    const int64_t row = blockIdx.x;
    const uint4* xr = reinterpret_cast<const uint4*>(x + row * ld_x);
    const uint4* wr = reinterpret_cast<const uint4*>(w);

    if (tid == 0 && ahead > 0 && row + ahead < rows) {
        prefetch_l2(x + (row + ahead) * ld_x, static_cast<uint32_t>(hidden) * 2u);
        if constexpr (kAdd)
            prefetch_l2(res + (row + ahead) * ld_res, static_cast<uint32_t>(hidden) * 2u);
    }

    uint4 xv[VPT];
#pragma unroll
    for (int j = 0; j < VPT; ++j) {
        const int v = tid + j * T;
        xv[j] = (v < nvec) ? __ldcs(xr + v) : make_uint4(0, 0, 0, 0);
    }
    if constexpr (kAdd) {
        uint4* rr = reinterpret_cast<uint4*>(res + row * ld_res);
#pragma unroll
        for (int j = 0; j < VPT; ++j) {
            const int v = tid + j * T;
            if (v >= nvec) continue;
            const uint4 rv = rr[v];
            const uint32_t xu[4] = {xv[j].x, xv[j].y, xv[j].z, xv[j].w};
            const uint32_t ru[4] = {rv.x, rv.y, rv.z, rv.w};
            uint32_t o[4];
#pragma unroll
            for (int e = 0; e < 4; ++e)
                o[e] = bi::pack_bf16x2(__fadd_rn(bf16_lo(ru[e]), bf16_lo(xu[e])),
                                       __fadd_rn(bf16_hi(ru[e]), bf16_hi(xu[e])));
            xv[j] = make_uint4(o[0], o[1], o[2], o[3]);
            rr[v] = xv[j];
        }
    }

    float s = 0.f;
#pragma unroll
    for (int j = 0; j < VPT; ++j) {
        const uint32_t u[4] = {xv[j].x, xv[j].y, xv[j].z, xv[j].w};
#pragma unroll
        for (int e = 0; e < 4; ++e) {
            const float a = bf16_lo(u[e]), b = bf16_hi(u[e]);
            s = __fmaf_rn(a, a, s);
            s = __fmaf_rn(b, b, s);
        }
    }
#pragma unroll
    for (int off = 16; off >= 1; off >>= 1) s += __shfl_xor_sync(0xffffffffu, s, off);
    if ((tid & 31) == 0) warp_sums[tid >> 5] = s;
    __syncthreads();
    const int nwarps = T >> 5;
    float total = warp_sums[0];
    for (int i = 1; i < nwarps; ++i) total += warp_sums[i];
    const float r = rsqrtf(__fdiv_rn(total, static_cast<float>(hidden)) + eps);

    uint4* yr = reinterpret_cast<uint4*>(y + row * ld_y);
#pragma unroll
    for (int j = 0; j < VPT; ++j) {
        const int v = tid + j * T;
        if (v >= nvec) continue;
        const uint4 wv = __ldg(wr + v);
        const uint32_t xu[4] = {xv[j].x, xv[j].y, xv[j].z, xv[j].w};
        const uint32_t wu[4] = {wv.x, wv.y, wv.z, wv.w};
        uint32_t o[4];
#pragma unroll
        for (int e = 0; e < 4; ++e) {
            const float a = __fmul_rn(__fmul_rn(bf16_lo(xu[e]), r), bf16_lo(wu[e]));
            const float b = __fmul_rn(__fmul_rn(bf16_hi(xu[e]), r), bf16_hi(wu[e]));
            o[e] = bi::pack_bf16x2(a, b);
        }
        yr[v] = make_uint4(o[0], o[1], o[2], o[3]);
    }
}

}  // namespace

namespace {

template <bool kAdd>
bi_status launch_rmsnorm(const void* x, const void* w, void* y, int64_t rows, int32_t hidden,
                         int64_t ld_x, int64_t ld_y, float eps, void* res, int64_t ld_res,
                         cudaStream_t stream) {
    if (rows < 0 || rows > 0x7fffffffLL) return BI_ERR_INVALID_ARG;
    if (!(eps >= 0.f) || eps != eps || eps > 3.0e38f) return BI_ERR_INVALID_ARG;
    if (hidden < 8 || hidden > 32768 || (hidden & 7)) return BI_ERR_UNSUPPORTED_SHAPE;
    if (ld_x < hidden || ld_y < hidden) return BI_ERR_INVALID_ARG;
    if ((ld_x & 7) || (ld_y & 7)) return BI_ERR_MISALIGNED;
    if (kAdd && ld_res < hidden) return BI_ERR_INVALID_ARG;
    if (kAdd && (ld_res & 7)) return BI_ERR_MISALIGNED;
    if (rows == 0) return BI_OK;
    if (!x || !w || !y || (kAdd && !res)) return BI_ERR_INVALID_ARG;
    if (!bi::aligned16(x) || !bi::aligned16(w) || !bi::aligned16(y) ||
        (kAdd && !bi::aligned16(res)))
        return BI_ERR_MISALIGNED;

    // Thread count and vectors per thread depend on `hidden` alone.
    const int nvec = hidden / 8;
    int threads, vpt;
    if (nvec <= kMaxThreads) {
        threads = (nvec + 31) / 32 * 32;
        vpt = 1;
    } else {
        threads = kMaxThreads;
        vpt = (nvec + kMaxThreads - 1) / kMaxThreads;  // 2 .. 16
    }
    const auto* xb = static_cast<const __nv_bfloat16*>(x);
    const auto* wb = static_cast<const __nv_bfloat16*>(w);
    auto* yb = static_cast<__nv_bfloat16*>(y);
    auto* rb = static_cast<__nv_bfloat16*>(res);
    const dim3 grid(static_cast<unsigned>(rows));
    cudaError_t err;
    const int64_t ahead = kPrefetchAheadBytes / (int64_t{hidden} * 2 * (kAdd ? 2 : 1));
    if (vpt == 1)
        err = bi::launch_pdl(rmsnorm_kernel<1, kAdd>, grid, dim3(threads), 0, stream, xb, wb, yb, hidden, ld_x, ld_y, eps, rb, ld_res, rows, ahead);
    else if (vpt == 2)
        err = bi::launch_pdl(rmsnorm_kernel<2, kAdd>, grid, dim3(threads), 0, stream, xb, wb, yb, hidden, ld_x, ld_y, eps, rb, ld_res, rows, ahead);
    else if (vpt <= 4)
        err = bi::launch_pdl(rmsnorm_kernel<4, kAdd>, grid, dim3(threads), 0, stream, xb, wb, yb, hidden, ld_x, ld_y, eps, rb, ld_res, rows, ahead);
    else if (vpt <= 8)
        err = bi::launch_pdl(rmsnorm_kernel<8, kAdd>, grid, dim3(threads), 0, stream, xb, wb, yb, hidden, ld_x, ld_y, eps, rb, ld_res, rows, ahead);
    else
        err = bi::launch_pdl(rmsnorm_kernel<16, kAdd>, grid, dim3(threads), 0, stream, xb, wb, yb, hidden, ld_x, ld_y, eps, rb, ld_res, rows, ahead);
    if (err != cudaSuccess) return BI_ERR_CUDA;
    return cudaGetLastError() == cudaSuccess ? BI_OK : BI_ERR_CUDA;
}

}  // namespace

extern "C" bi_status bi_rmsnorm(const void* x, const void* w, void* y, int64_t rows,
                                int32_t hidden, int64_t ld_x, int64_t ld_y, float eps,
                                cudaStream_t stream) {
    return launch_rmsnorm<false>(x, w, y, rows, hidden, ld_x, ld_y, eps, nullptr, hidden, stream);
}

extern "C" bi_status bi_add_rmsnorm(const void* x, void* residual, const void* w, void* y,
                                    int64_t rows, int32_t hidden, int64_t ld_x, int64_t ld_res,
                                    int64_t ld_y, float eps, cudaStream_t stream) {
    return launch_rmsnorm<true>(x, w, y, rows, hidden, ld_x, ld_y, eps, residual, ld_res, stream);
}
