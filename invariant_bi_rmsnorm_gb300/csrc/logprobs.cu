// bi_logprobs: per-row log-sum-exp of a logits row and the log-probability
// of one target token, with a reduction order fixed by the vocabulary size.
//
// "Defeating Nondeterminism in LLM Inference: The Core Role of Batch
// Invariance", section "Experimental Validation and Future Prospects" (true
// on-policy RL): the sampler and the trainer must agree bit for bit on the
// log-probabilities of the sampled tokens.  The softmax denominator is a
// reduction over the vocabulary, so it gets the same treatment as RMSNorm:
// one row per CTA and an order that depends only on the row length.
//
//   pass 1:  m = max_j x_j                      (exact, order-free)
//   pass 2:  s = sum_j exp(x_j - m) in fp32:    thread t adds its 16-byte
//            vectors t, t+256, ... in order, each left to right; then an xor
//            butterfly over the warp; then the 8 warp sums in warp order
//   lse = m + log(s);   logprob = x_target - lse
#include <cuda_bf16.h>

#include <cmath>

#include "bi_internal.h"
#include "bi_ptx.cuh"

namespace {

constexpr int kThreads = 256;

__device__ __forceinline__ float lo16(uint32_t v) { return __uint_as_float(v << 16); }
__device__ __forceinline__ float hi16(uint32_t v) { return __uint_as_float(v & 0xffff0000u); }

__global__ void __launch_bounds__(kThreads)
    logprobs_kernel(const __nv_bfloat16* __restrict__ logits, int64_t ld, int vocab,
                    const int32_t* __restrict__ targets, float* __restrict__ logprob_out,
                    float* __restrict__ lse_out, uint32_t* err) {
    __shared__ float red[kThreads / 32];
    const int64_t row = blockIdx.x;
    const int tid = threadIdx.x;
    const __nv_bfloat16* x = logits + row * ld;
    const uint4* xv = reinterpret_cast<const uint4*>(x);
    const int nvec = vocab / 8;

    float m = -INFINITY;
    for (int v = tid; v < nvec; v += kThreads) {
        const uint4 u = xv[v];
        const uint32_t w[4] = {u.x, u.y, u.z, u.w};
#pragma unroll
        for (int e = 0; e < 4; ++e) m = fmaxf(m, fmaxf(lo16(w[e]), hi16(w[e])));
    }
#pragma unroll
    for (int o = 16; o >= 1; o >>= 1) m = fmaxf(m, __shfl_xor_sync(0xffffffffu, m, o));
    if ((tid & 31) == 0) red[tid >> 5] = m;
    __syncthreads();
    float M = red[0];
    for (int i = 1; i < kThreads / 32; ++i) M = fmaxf(M, red[i]);
    __syncthreads();

    float s = 0.f;
    for (int v = tid; v < nvec; v += kThreads) {
        const uint4 u = xv[v];
        const uint32_t w[4] = {u.x, u.y, u.z, u.w};
#pragma unroll
        for (int e = 0; e < 4; ++e) {
            s = __fadd_rn(s, expf(__fsub_rn(lo16(w[e]), M)));
            s = __fadd_rn(s, expf(__fsub_rn(hi16(w[e]), M)));
        }
    }
#pragma unroll
    for (int o = 16; o >= 1; o >>= 1) s += __shfl_xor_sync(0xffffffffu, s, o);
    if ((tid & 31) == 0) red[tid >> 5] = s;
    __syncthreads();
    if (tid != 0) return;
    float S = red[0];
    for (int i = 1; i < kThreads / 32; ++i) S = __fadd_rn(S, red[i]);
    const float lse = __fadd_rn(M, logf(S));
    if (lse_out) lse_out[row] = lse;
    if (targets && logprob_out) {
        const int t = targets[row];
        if (t < 0 || t >= vocab) {
            bi::report_error(err, bi::kErrBadInput | bi::kWhereDecoderOps);
            logprob_out[row] = NAN;
        } else {
            logprob_out[row] = __fsub_rn(__bfloat162float(x[t]), lse);
        }
    }
}

}  // namespace

extern "C" bi_status bi_logprobs(const void* logits, int64_t rows, int32_t vocab, int64_t ld,
                                 const int32_t* targets, float* logprob_out, float* lse_out,
                                 cudaStream_t stream) {
    if (rows < 0 || rows > 0x7fffffffLL) return BI_ERR_INVALID_ARG;
    if (vocab < 8 || (vocab & 7)) return BI_ERR_UNSUPPORTED_SHAPE;
    if (ld < vocab) return BI_ERR_INVALID_ARG;
    if (ld & 7) return BI_ERR_MISALIGNED;
    if (rows == 0) return BI_OK;
    if (!logits || (!lse_out && !(targets && logprob_out))) return BI_ERR_INVALID_ARG;
    if (!bi::aligned16(logits) || (reinterpret_cast<uintptr_t>(targets) & 3) ||
        (reinterpret_cast<uintptr_t>(logprob_out) & 3) || (reinterpret_cast<uintptr_t>(lse_out) & 3))
        return BI_ERR_MISALIGNED;
    logprobs_kernel<<<static_cast<unsigned>(rows), kThreads, 0, stream>>>(
        static_cast<const __nv_bfloat16*>(logits), ld, vocab, targets, logprob_out, lse_out,
        bi::device_error_word());
    return cudaGetLastError() == cudaSuccess ? BI_OK : BI_ERR_CUDA;
}
