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
// One pass over the row (read once from HBM).  Thread t owns the 16-byte
// vectors t, t+256, t+512, ... and folds them in that order into a running
// (m, s) pair with sum_j exp(x_j - m) = s, exponentials taken base 2 with
// c = log2(e) rounded to fp32 and mc = fp32(m * c):
//     m' = max(m, max of the vector's 8 values);  s = s * 2^((m - m') c);
//     s += 2^(fma(x_e, c, -mc')) for e = 0..7 in element order     (fp32)
// Then an xor butterfly over the warp and the 8 warp pairs in warp order,
// each step  M = max(m1, m2);  s = s1 2^((m1 - M) c) + s2 2^((m2 - M) c).
//   lse = M + log(s);   logprob = x_target - lse
// Every step depends only on the vocabulary size, never on the row count.
#include <cuda_bf16.h>

#include <cmath>

#include "bi_internal.h"
#include "bi_ptx.cuh"

namespace {

constexpr int kThreads = 256;

__device__ __forceinline__ float lo16(uint32_t v) { return __uint_as_float(v << 16); }
__device__ __forceinline__ float hi16(uint32_t v) { return __uint_as_float(v & 0xffff0000u); }

constexpr float kLog2e = 1.4426950408889634f;

// exp(a - b) for a <= b, as 2^((a - b) c); 0 when a is -inf
__device__ __forceinline__ float rescale(float a, float b) {
    return exp2f(__fmul_rn(__fsub_rn(a, b), kLog2e));
}

// 2^x as one ex2.approx.ftz.f32 (bi::ex2_approx; subnormal results flushed
// to zero) for the per-element terms: exp2f() takes about three more
// instructions, and the kernel is issue-bound as much as it is HBM-bound.  A
// flushed term is below 2^-126.  The vector that sets the running maximum also
// adds that maximum's own term (about 1), so by the end of every vector the
// sum is near 1 or more, and terms that small round away: the row's (m, s) is
// unchanged.
__device__ __forceinline__ float ex2_term(float x) { return bi::ex2_approx(x); }

// (m, s) after folding one vector of 8 values in element order; mc = m * c
__device__ __forceinline__ void fold_vec(float& m, float& mc, float& s, const uint4& u) {
    const float x[8] = {lo16(u.x), hi16(u.x), lo16(u.y), hi16(u.y),
                        lo16(u.z), hi16(u.z), lo16(u.w), hi16(u.w)};
    float vm = x[0];
#pragma unroll
    for (int e = 1; e < 8; ++e) vm = fmaxf(vm, x[e]);
    if (vm == -INFINITY) return;  // nothing visible in this vector
    if (vm > m) {
        s = __fmul_rn(s, rescale(m, vm));  // m = -inf: s is 0 and stays 0
        m = vm;
        mc = __fmul_rn(vm, kLog2e);
    }
#pragma unroll
    for (int e = 0; e < 8; ++e) s = __fadd_rn(s, ex2_term(__fmaf_rn(x[e], kLog2e, -mc)));
}

// (m1, s1) <- (m1, s1) combined with (m2, s2); symmetric in its operands
__device__ __forceinline__ void combine(float& m1, float& s1, float m2, float s2) {
    const float M = fmaxf(m1, m2);
    if (M == -INFINITY) return;  // both empty
    s1 = __fadd_rn(__fmul_rn(s1, rescale(m1, M)), __fmul_rn(s2, rescale(m2, M)));
    m1 = M;
}

constexpr int kUnroll = 4;

__global__ void __launch_bounds__(kThreads)
    logprobs_kernel(const __nv_bfloat16* __restrict__ logits, int64_t ld, int vocab,
                    const int32_t* __restrict__ targets, float* __restrict__ logprob_out,
                    float* __restrict__ lse_out, uint32_t* err) {
    bi::launch_dependents();
    bi::grid_dependency_wait();  // nothing global is touched before the previous kernel ends
    __shared__ float red_m[kThreads / 32], red_s[kThreads / 32];
    const int64_t row = blockIdx.x;
    const int tid = threadIdx.x;
    const __nv_bfloat16* x = logits + row * ld;
    const uint4* xv = reinterpret_cast<const uint4*>(x);
    const int nvec = vocab / 8;

    float m = -INFINITY, mc = -INFINITY, s = 0.f;
    int v = tid;
    // kUnroll vectors in flight per thread; folded in ascending order
    for (; v + (kUnroll - 1) * kThreads < nvec; v += kUnroll * kThreads) {
        uint4 u[kUnroll];
#pragma unroll
        for (int i = 0; i < kUnroll; ++i) u[i] = __ldcs(xv + v + i * kThreads);
#pragma unroll
        for (int i = 0; i < kUnroll; ++i) fold_vec(m, mc, s, u[i]);
    }
    for (; v < nvec; v += kThreads) fold_vec(m, mc, s, __ldcs(xv + v));
#pragma unroll
    for (int o = 16; o >= 1; o >>= 1) {
        const float m2 = __shfl_xor_sync(0xffffffffu, m, o);
        const float s2 = __shfl_xor_sync(0xffffffffu, s, o);
        combine(m, s, m2, s2);
    }
    if ((tid & 31) == 0) {
        red_m[tid >> 5] = m;
        red_s[tid >> 5] = s;
    }
    __syncthreads();
    if (tid != 0) return;
    float M = red_m[0], S = red_s[0];
    for (int i = 1; i < kThreads / 32; ++i) combine(M, S, red_m[i], red_s[i]);
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
    return bi::launch_pdl(logprobs_kernel, dim3(static_cast<unsigned>(rows)), dim3(kThreads), 0,
                          stream, static_cast<const __nv_bfloat16*>(logits), ld, vocab, targets,
                          logprob_out, lse_out, bi::device_error_word()) == cudaSuccess
               ? BI_OK
               : BI_ERR_CUDA;
}
