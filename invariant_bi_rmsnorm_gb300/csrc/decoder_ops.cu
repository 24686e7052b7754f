// Pointwise and per-head steps a decoder layer needs around the three
// reduction kernels: per-head q/k RMSNorm + rotary embedding + append of the
// new tokens' K/V into the paged cache, and the SwiGLU product.
//
// "Defeating Nondeterminism in LLM Inference: The Core Role of Batch
// Invariance", section "Achieving Batch-Invariant Kernels": pointwise
// operations are batch-invariant by construction; the per-head RMSNorm here
// reduces over one head's 128 values in an order fixed by the head size.  The
// KV append follows "3. Batch-Invariant Attention": the new tokens' K/V go
// into the same paged cache as every earlier token before attention runs.
#include <cuda_bf16.h>

#include <algorithm>
#include <cmath>

#include "bi_internal.h"
#include "bi_ptx.cuh"

namespace {

constexpr int kD = 128;
constexpr int kHalf = kD / 2;

__device__ __forceinline__ float bf(const __nv_bfloat16 v) { return __bfloat162float(v); }

struct RopeArgs {
    const __nv_bfloat16* qkv;
    int64_t ld_qkv;
    int T, Hq, Hkv;
    const int32_t* positions;
    const int32_t* slots;
    const float* rope;  // [max_pos][128]: cos(pos * f_i) at i, sin(pos * f_i) at 64 + i
    int max_pos;
    const __nv_bfloat16* q_norm_w;  // [128] or null
    const __nv_bfloat16* k_norm_w;  // [128] or null
    float eps;
    __nv_bfloat16* q_out;  // [T][Hq][128]
    __nv_bfloat16* k_cache;
    __nv_bfloat16* v_cache;  // [num_pages][Hkv][16][128]
    int64_t num_slots;       // num_pages * 16
    int page_size;
    uint32_t* err;
};

// One CTA of 8 warps per token.  A warp works on two heads at once, one per
// half-warp: warp w takes head pairs w, w+8, w+16 (heads 2p and 2p+1) and
// issues the loads of all its pairs before computing any, so enough bytes
// are in flight to cover HBM latency.  Per head, lane l of its half (l =
// lane & 15) holds dims 4l .. 4l+3 and their rotation partners 64+4l ..
// 64+4l+3:
//   q, k heads:  x -> bf16(x * rsqrt(mean(x^2) + eps) * w)   (if a norm weight is given;
//                    sum of squares: per lane in the order 4l .. 4l+3, 64+4l .. 64+4l+3,
//                    then an xor butterfly over the 16 lanes of the half, strides 8, 4, 2, 1)
//                -> rotate-half RoPE in fp32: y_i = x_i c_i - x_{64+i} s_i,
//                   y_{64+i} = x_{64+i} c_i + x_i s_i, rounded once to bf16
//   v heads:     copied.
// q goes to q_out; k and v to their token's cache slot.  Each head's
// arithmetic depends only on its own 128 values, the position and the weights.
constexpr int kRopeWarps = 8;
constexpr int kPairsPerPass = 3;

__device__ __forceinline__ uint2 ld_b64(const __nv_bfloat16* p) {
    return *reinterpret_cast<const uint2*>(p);
}

__device__ __forceinline__ void load_pairs(const __nv_bfloat16* row, int p0, int heads, int half,
                                           int i0, uint2 (&lo)[kPairsPerPass],
                                           uint2 (&hi)[kPairsPerPass]) {
#pragma unroll
    for (int j = 0; j < kPairsPerPass; ++j) {
        const int h = 2 * (p0 + j * kRopeWarps) + half;
        if (h < heads) {
            lo[j] = ld_b64(row + static_cast<int64_t>(h) * kD + i0);
            hi[j] = ld_b64(row + static_cast<int64_t>(h) * kD + kHalf + i0);
        }
    }
}

__device__ __forceinline__ void unpack4(uint2 v, float* x) {
    x[0] = __uint_as_float(v.x << 16);
    x[1] = __uint_as_float(v.x & 0xffff0000u);
    x[2] = __uint_as_float(v.y << 16);
    x[3] = __uint_as_float(v.y & 0xffff0000u);
}

__global__ void __launch_bounds__(kRopeWarps * 32, 4) qk_norm_rope_append_kernel(const RopeArgs a) {
    bi::launch_dependents();
    bi::grid_dependency_wait();  // nothing global is touched before the previous kernel ends
    const int t = blockIdx.x;
    const int warp = threadIdx.x >> 5;
    const int lane = threadIdx.x & 31;
    const int half = lane >> 4;
    const int heads = a.Hq + 2 * a.Hkv;
    const int pairs = (heads + 1) / 2;
    const int i0 = 4 * (lane & 15);
    const __nv_bfloat16* row = a.qkv + static_cast<int64_t>(t) * a.ld_qkv;
    // the first pass's q/k/v loads go out before the position is known, so
    // their latency overlaps that of the position -> RoPE-table chain
    uint2 lo[kPairsPerPass], hi[kPairsPerPass];
    load_pairs(row, warp, heads, half, i0, lo, hi);
    const int pos = a.positions[t];
    const int64_t slot = a.slots[t];
    if (pos < 0 || pos >= a.max_pos || slot < 0 || slot >= a.num_slots) {
        if (threadIdx.x == 0) bi::report_error(a.err, bi::kErrBadInput | bi::kWhereDecoderOps);
        return;
    }
    const float* cs = a.rope + static_cast<int64_t>(pos) * kD;
    const float4 cosv = *reinterpret_cast<const float4*>(cs + i0);
    const float4 sinv = *reinterpret_cast<const float4*>(cs + kHalf + i0);
    const float c[4] = {cosv.x, cosv.y, cosv.z, cosv.w};
    const float sn[4] = {sinv.x, sinv.y, sinv.z, sinv.w};
    // the norm weights of this lane's 8 dims, as bf16 pairs (unpacked where used)
    const uint2 zero2 = make_uint2(0u, 0u);
    const uint2 qw_lo = a.q_norm_w ? ld_b64(a.q_norm_w + i0) : zero2;
    const uint2 qw_hi = a.q_norm_w ? ld_b64(a.q_norm_w + kHalf + i0) : zero2;
    const uint2 kw_lo = a.k_norm_w ? ld_b64(a.k_norm_w + i0) : zero2;
    const uint2 kw_hi = a.k_norm_w ? ld_b64(a.k_norm_w + kHalf + i0) : zero2;
    // the token's slot in every kv-head's page block (page size fixed at BI_PAGE_SIZE)
    const int64_t page = slot / BI_PAGE_SIZE, off = slot % BI_PAGE_SIZE;
    const int64_t kv_slot = (page * a.Hkv * BI_PAGE_SIZE + off) * kD;

    for (int p0 = warp; p0 < pairs; p0 += kRopeWarps * kPairsPerPass) {
        if (p0 != warp) load_pairs(row, p0, heads, half, i0, lo, hi);
#pragma unroll
        for (int j = 0; j < kPairsPerPass; ++j) {
            const int pr = p0 + j * kRopeWarps;  // the same for every lane
            if (pr >= pairs) break;
            const int h = 2 * pr + half;        // this half's head
            const bool live = h < heads;
            const bool is_v = h >= a.Hq + a.Hkv;
            const bool is_q = h < a.Hq;
            float x[8];
            unpack4(lo[j], x);
            unpack4(hi[j], x + 4);
            // every lane takes part in the butterfly (both halves, any head kind)
            const bool norm = is_q ? a.q_norm_w != nullptr : a.k_norm_w != nullptr;
            float ss = 0.f;
#pragma unroll
            for (int e = 0; e < 8; ++e) ss = __fmaf_rn(x[e], x[e], ss);
#pragma unroll
            for (int o = 8; o >= 1; o >>= 1) ss += __shfl_xor_sync(0xffffffffu, ss, o);
            if (!live) continue;
            if (is_v) {  // v: copy into the cache
                const int hv = h - a.Hq - a.Hkv;
                __nv_bfloat16* dst = a.v_cache + kv_slot + hv * (BI_PAGE_SIZE * kD);
                *reinterpret_cast<uint2*>(dst + i0) = lo[j];
                *reinterpret_cast<uint2*>(dst + kHalf + i0) = hi[j];
                continue;
            }
            if (norm) {
                // ss / 128 computed as ss * 2^-7: the same correctly rounded value
                const float r = rsqrtf(__fmul_rn(ss, 1.f / kD) + a.eps);
                float w[8];
                unpack4(is_q ? qw_lo : kw_lo, w);
                unpack4(is_q ? qw_hi : kw_hi, w + 4);
#pragma unroll
                for (int e = 0; e < 8; ++e)
                    x[e] = __bfloat162float(__float2bfloat16_rn(__fmul_rn(__fmul_rn(x[e], r), w[e])));
            }
            float y[8];
#pragma unroll
            for (int e = 0; e < 4; ++e) {
                y[e] = __fsub_rn(__fmul_rn(x[e], c[e]), __fmul_rn(x[4 + e], sn[e]));
                y[4 + e] = __fadd_rn(__fmul_rn(x[4 + e], c[e]), __fmul_rn(x[e], sn[e]));
            }
            __nv_bfloat16* dst;
            if (is_q) {
                dst = a.q_out + (static_cast<int64_t>(t) * a.Hq + h) * kD;
            } else {
                dst = a.k_cache + kv_slot + (h - a.Hq) * (BI_PAGE_SIZE * kD);
            }
            *reinterpret_cast<uint2*>(dst + i0) =
                make_uint2(bi::pack_bf16x2(y[0], y[1]), bi::pack_bf16x2(y[2], y[3]));
            *reinterpret_cast<uint2*>(dst + kHalf + i0) =
                make_uint2(bi::pack_bf16x2(y[4], y[5]), bi::pack_bf16x2(y[6], y[7]));
        }
    }
}

// h[t][j] = bf16( silu(g) * u ),  g = gu[t][j], u = gu[t][F + j],
// silu(g) = g / (1 + exp(-g)), all in fp32.  8 outputs per thread.  The grid
// is 2-D (vector blocks of a row on x, rows on y) so that no thread divides a
// flat index by the row length.
__global__ void silu_mul_kernel(const __nv_bfloat16* __restrict__ gu, int64_t ld_gu,
                                __nv_bfloat16* __restrict__ out, int64_t ld_out, int T, int F) {
    bi::launch_dependents();
    bi::grid_dependency_wait();  // nothing global is touched before the previous kernel ends
    const int j = (blockIdx.x * blockDim.x + threadIdx.x) * 8;
    if (j >= F) return;
    for (int64_t t = blockIdx.y; t < T; t += gridDim.y) {
        const uint4 gv = *reinterpret_cast<const uint4*>(gu + t * ld_gu + j);
        const uint4 uv = *reinterpret_cast<const uint4*>(gu + t * ld_gu + F + j);
        const __nv_bfloat162* g2 = reinterpret_cast<const __nv_bfloat162*>(&gv);
        const __nv_bfloat162* u2 = reinterpret_cast<const __nv_bfloat162*>(&uv);
        uint32_t o[4];
#pragma unroll
        for (int e = 0; e < 4; ++e) {
            o[e] = bi::pack_bf16x2(bi::swiglu(__low2float(g2[e]), __low2float(u2[e])),
                                   bi::swiglu(__high2float(g2[e]), __high2float(u2[e])));
        }
        *reinterpret_cast<uint4*>(out + t * ld_out + j) = make_uint4(o[0], o[1], o[2], o[3]);
    }
}

}  // namespace

extern "C" bi_status bi_qk_norm_rope_append(const void* qkv, int64_t ld_qkv, int32_t T, int32_t Hq,
                                            int32_t Hkv, int32_t D, const int32_t* positions,
                                            const int32_t* slots, const float* rope_table,
                                            int32_t max_pos, const void* q_norm_w,
                                            const void* k_norm_w, float eps, void* q_out,
                                            void* k_cache, void* v_cache, int32_t num_pages,
                                            int32_t page_size, cudaStream_t stream) {
    if (T < 0 || Hq <= 0 || Hkv <= 0 || max_pos < 1 || num_pages < 1) return BI_ERR_INVALID_ARG;
    if (D != kD || page_size != BI_PAGE_SIZE) return BI_ERR_UNSUPPORTED_SHAPE;
    if (ld_qkv < static_cast<int64_t>(Hq + 2 * Hkv) * kD) return BI_ERR_INVALID_ARG;
    if (ld_qkv & 7) return BI_ERR_MISALIGNED;
    if (!(eps >= 0.f) || !std::isfinite(eps)) return BI_ERR_INVALID_ARG;
    if (T == 0) return BI_OK;
    if (!qkv || !positions || !slots || !rope_table || !q_out || !k_cache || !v_cache)
        return BI_ERR_INVALID_ARG;
    if (!bi::aligned16(qkv) || !bi::aligned16(q_out) || !bi::aligned16(k_cache) ||
        !bi::aligned16(v_cache) || (reinterpret_cast<uintptr_t>(rope_table) & 15) ||
        (reinterpret_cast<uintptr_t>(positions) & 3) || (reinterpret_cast<uintptr_t>(slots) & 3))
        return BI_ERR_MISALIGNED;
    RopeArgs a;
    a.qkv = static_cast<const __nv_bfloat16*>(qkv);
    a.ld_qkv = ld_qkv;
    a.T = T;
    a.Hq = Hq;
    a.Hkv = Hkv;
    a.positions = positions;
    a.slots = slots;
    a.rope = rope_table;
    a.max_pos = max_pos;
    a.q_norm_w = static_cast<const __nv_bfloat16*>(q_norm_w);
    a.k_norm_w = static_cast<const __nv_bfloat16*>(k_norm_w);
    a.eps = eps;
    a.q_out = static_cast<__nv_bfloat16*>(q_out);
    a.k_cache = static_cast<__nv_bfloat16*>(k_cache);
    a.v_cache = static_cast<__nv_bfloat16*>(v_cache);
    a.num_slots = static_cast<int64_t>(num_pages) * page_size;
    a.page_size = page_size;
    a.err = bi::device_error_word();
    return bi::launch_pdl(qk_norm_rope_append_kernel, dim3(static_cast<unsigned>(T)),
                          dim3(kRopeWarps * 32), 0, stream, a) == cudaSuccess
               ? BI_OK
               : BI_ERR_CUDA;
}

extern "C" bi_status bi_silu_mul(const void* gate_up, int64_t ld_gate_up, int32_t T, int32_t F,
                                 void* out, int64_t ld_out, cudaStream_t stream) {
    if (T < 0 || F < 8 || (F & 7) || F > (1 << 30))
        return T < 0 ? BI_ERR_INVALID_ARG : BI_ERR_UNSUPPORTED_SHAPE;
    if (ld_gate_up < 2 * static_cast<int64_t>(F) || ld_out < F) return BI_ERR_INVALID_ARG;
    if ((ld_gate_up & 7) || (ld_out & 7)) return BI_ERR_MISALIGNED;
    if (T == 0) return BI_OK;
    if (!gate_up || !out) return BI_ERR_INVALID_ARG;
    if (!bi::aligned16(gate_up) || !bi::aligned16(out)) return BI_ERR_MISALIGNED;
    const int threads = 256;
    const dim3 grid(static_cast<unsigned>((F / 8 + threads - 1) / threads),
                    static_cast<unsigned>(std::min(T, 65535)));
    return bi::launch_pdl(silu_mul_kernel, grid, dim3(threads), 0, stream,
                          static_cast<const __nv_bfloat16*>(gate_up), ld_gate_up,
                          static_cast<__nv_bfloat16*>(out), ld_out, T, F) == cudaSuccess
               ? BI_OK
               : BI_ERR_CUDA;
}
