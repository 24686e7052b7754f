// bi_prefill_attention: attention for many query rows of the same sequence at
// once (prompt prefill, chunked prefill), with causal visibility, and per row
// exactly the arithmetic bi_decode_attention uses.
//
// "Defeating Nondeterminism in LLM Inference: The Core Role of Batch
// Invariance", section "3. Batch-Invariant Attention": the FlashAttention2
// strategy parallelises over queries and reduces over keys inside one core,
// and a token's reduction order must not depend on how many other tokens of
// its sequence are processed with it (chunked prefill, prefix caching).  So a
// query row here reduces over its keys exactly as a decode row does: 256-token
// chunks in ascending order, one online softmax over each chunk's pages
// 0, 1, 2, ... (attn_common.cuh), the chunk partials folded in ascending
// chunk order.  A token's output is therefore bit-identical whether it is
// computed here, in a prefill chunk of any size, or by bi_decode_attention.
//
// One CTA per (sequence, kv-head, tile of query rows).  The tile's columns
// (query row x query head) are spread over 8 consumer warps, 8 columns each;
// a producer warp streams the pages the tile needs (chunk by chunk, pages in
// order) through a 6-stage TMA ring that all consumer warps read.  A page a
// row cannot see (past its causal length) leaves that row's state unchanged.
#include <cuda_bf16.h>

#include <algorithm>
#include <atomic>
#include <cmath>

#include "attn_common.cuh"
#include "bi_internal.h"
#include "bi_ptx.cuh"

namespace {

using bi_attn::kChunk;
using bi_attn::kD;
using bi_attn::kHalfBytes;
using bi_attn::kMatBytes;
using bi_attn::kMaxGroup;
using bi_attn::kPage;
using bi_attn::kPagesPerChunk;
using bi_attn::kStageBytes;

constexpr int kConsumerWarps = 8;
constexpr int kThreads = (kConsumerWarps + 1) * 32;  // + one producer warp
constexpr int kCols = kConsumerWarps * 8;             // 64 columns per tile
constexpr int kStages = 6;
constexpr int kSmemBytes = kStages * kStageBytes + 16 * kStages + 1024 /*align*/;

struct PrefillArgs {
    const __nv_bfloat16* q;
    const int32_t* block_table;
    const int32_t* seq_lens;
    const int32_t* q_indptr;
    __nv_bfloat16* out;
    uint32_t* err;
    int max_pages_per_seq;
    int Hq, Hkv, group;
    int rows_per_tile;
    int num_pages;
    int max_seq_len;
    int max_q_len;
    int T;
    float scale_log2;
};

__device__ __forceinline__ void consumer_bar_sync() {
    asm volatile("bar.sync 1, %0;" ::"n"(kConsumerWarps * 32) : "memory");
}

// two CTAs per SM (96 registers, a small spill) ran 12 % faster than one
// (138 registers, no spill): the consumers are latency-bound, not spill-bound
__global__ void __launch_bounds__(kThreads, 2)
    prefill_attn_kernel(const __grid_constant__ CUtensorMap tmap_k,
                        const __grid_constant__ CUtensorMap tmap_v, const PrefillArgs a) {
    bi::launch_dependents();
    bi::grid_dependency_wait();  // nothing global is touched before the previous kernel ends
    const int tile = blockIdx.x;
    const int g = blockIdx.y;
    const int s = blockIdx.z;
    const int tid = threadIdx.x;
    const int warp = tid >> 5;
    const int lane = tid & 31;

    const int q0 = a.q_indptr[s];
    const int nq = a.q_indptr[s + 1] - q0;
    const int Ls = a.seq_lens[s];
    if (q0 < 0 || nq < 0 || q0 + nq > a.T || nq > a.max_q_len ||
        (nq > 0 && (Ls < nq || Ls > a.max_seq_len))) {
        if (tid == 0 && tile == 0 && g == 0) bi::report_error(a.err, bi::kErrBadInput | bi::kWhereAttnSplit);
        return;
    }
    const int r0 = tile * a.rows_per_tile;
    if (r0 >= nq) return;
    const int nr = min(a.rows_per_tile, nq - r0);
    // query row r (0-based among the sequence's nq rows) sees the first
    // Ls - nq + 1 + r tokens
    const int Lbase = Ls - nq + 1;
    const int Lmax = Lbase + r0 + nr - 1;
    const int npg = (Lmax + kPage - 1) / kPage;
    const int nch = (Lmax + kChunk - 1) / kChunk;

    extern __shared__ uint8_t smem_raw[];
    uint8_t* smem = reinterpret_cast<uint8_t*>(
        (reinterpret_cast<uintptr_t>(smem_raw) + 1023) & ~static_cast<uintptr_t>(1023));
    uint64_t* full = reinterpret_cast<uint64_t*>(smem + kStages * kStageBytes);
    uint64_t* empty = full + kStages;
    __shared__ int bad_page;

    const int32_t* bt = a.block_table + static_cast<int64_t>(s) * a.max_pages_per_seq;
    if (tid == 0) {
        bad_page = 0;
        for (int i = 0; i < kStages; ++i) {
            bi::mbar_init(&full[i], 1);
            bi::mbar_init(&empty[i], kConsumerWarps);
        }
        bi::fence_mbar_init();
        bi::tma_prefetch_desc(&tmap_k);
        bi::tma_prefetch_desc(&tmap_v);
    }
    __syncthreads();
    for (int i = tid; i < npg; i += kThreads) {
        const int pg = bt[i];
        if (pg < 0 || pg >= a.num_pages) bad_page = 1;
    }
    __syncthreads();
    if (bad_page) {
        if (tid == 0) bi::report_error(a.err, bi::kErrBadInput | bi::kWhereAttnSplit);
        return;
    }

    if (warp == kConsumerWarps) {
        // ---------------- producer: every page the tile needs, in order ----
        if (lane == 0) {
            int k = 0;
            for (; k < npg; ++k) {
                const int st = k % kStages;
                if (!bi::mbar_wait(&empty[st], ((k / kStages) & 1) ^ 1)) {
                    bi::report_error(a.err, bi::kErrTimeout | bi::kWhereAttnSplit);
                    break;
                }
                uint8_t* kd = smem + st * kStageBytes;
                uint8_t* vd = kd + kMatBytes;
                const int row = (bt[k] * a.Hkv + g) * kPage;
                bi::mbar_arrive_expect_tx(&full[st], kStageBytes);
                bi::tma_load_3d(kd, &tmap_k, &full[st], 0, row, 0);
                bi::tma_load_3d(vd, &tmap_v, &full[st], 0, row, 0);
            }
            // the CTA's shared memory outlives no copy: wait (bounded) for the
            // last copy issued into each stage -- on a healthy run the
            // consumers wait for the same copies
            for (int i = max(0, k - kStages); i < k; ++i)
                bi::mbar_wait_for(&full[i % kStages], (i / kStages) & 1, bi::kDrainNs);
        }
        return;
    }

    // ---------------- consumers: 8 columns per warp -------------------------
    // column n of the tile = query row n / group, head n % group
    const int G = a.group;
    auto col_row = [&](int n) { return n / G; };
    uint32_t qb0[8], qb1[8];
    {
        const int n = warp * 8 + (lane >> 2);
        const int rr = col_row(n);
        const bool ok = n < a.rows_per_tile * G && rr < nr;
        bi_attn::load_q_frags(
            ok ? a.q + (static_cast<int64_t>(q0 + r0 + rr) * a.Hq + g * G + n % G) * kD : nullptr,
            lane, qb0, qb1);
    }
    // this lane's two columns and the tokens their rows see
    int Lcol[2];
    int rrcol[2];
#pragma unroll
    for (int e = 0; e < 2; ++e) {
        const int n = warp * 8 + 2 * (lane & 3) + e;
        rrcol[e] = col_row(n);
        const bool ok = n < a.rows_per_tile * G && rrcol[e] < nr;
        Lcol[e] = ok ? Lbase + r0 + rrcol[e] : 0;
    }

    float Mr[2] = {-INFINITY, -INFINITY}, Lr[2] = {0.f, 0.f};
    float Ar[8][4];
#pragma unroll
    for (int mt = 0; mt < 8; ++mt) Ar[mt][0] = Ar[mt][1] = Ar[mt][2] = Ar[mt][3] = 0.f;

    bool timed_out = false;
    int k = 0;  // page counter over the whole tile
    for (int c = 0; c < nch; ++c) {
        bi_attn::ColState st;
        bi_attn::colstate_init(st);
        const int np = min(kPagesPerChunk, npg - c * kPagesPerChunk);
        for (int p = 0; p < np; ++p, ++k) {
            const int stg = k % kStages;
            const bool ok = !timed_out && bi::mbar_wait(&full[stg], (k / kStages) & 1);
            if (!ok) timed_out = true;
            const int t0 = (c * kPagesPerChunk + p) * kPage;
            uint8_t* kd = smem + stg * kStageBytes;
            const int vmax = min(kPage, Lmax - t0);
            if (vmax < kPage) {
                // tokens past the longest row: zero their V rows once, for all warps
                if (warp == 0 && ok) bi_attn::zero_v_tail(kd + kMatBytes, vmax, lane);
                consumer_bar_sync();
            }
            if (ok) {
                const int v0 = max(0, min(kPage, Lcol[0] - t0));
                const int v1 = max(0, min(kPage, Lcol[1] - t0));
                const uint32_t kb = bi::smem_u32(kd);
                bi_attn::attend_page(st, kb, kb + kMatBytes, qb0, qb1, v0, v1, a.scale_log2, lane);
            }
            bi::fence_proxy_async_smem();
            __syncwarp();
            // a warp that timed out stops handing stages back, so the producer
            // stops too (its own wait on the stage runs out) and drains
            if (lane == 0 && !timed_out) bi::mbar_arrive(&empty[stg]);
        }
        // fold chunk c into each column whose row sees it, as the decode path does
#pragma unroll
        for (int e = 0; e < 2; ++e) {
            if (Lcol[e] <= c * kChunk) continue;
            if (c == 0) {
                Mr[e] = st.m[e];
                Lr[e] = st.l[e];
#pragma unroll
                for (int mt = 0; mt < 8; ++mt) {
                    Ar[mt][e] = st.acc[mt][e];
                    Ar[mt][2 + e] = st.acc[mt][2 + e];
                }
            } else {
                float Mn, fo, fc;
                bi_attn::fold_scalars(Mr[e], st.m[e], Mn, fo, fc);
                Lr[e] = bi_attn::fold_value(Lr[e], fo, st.l[e], fc);
#pragma unroll
                for (int mt = 0; mt < 8; ++mt) {
                    Ar[mt][e] = bi_attn::fold_value(Ar[mt][e], fo, st.acc[mt][e], fc);
                    Ar[mt][2 + e] = bi_attn::fold_value(Ar[mt][2 + e], fo, st.acc[mt][2 + e], fc);
                }
                Mr[e] = Mn;
            }
        }
    }
    if (timed_out) {
        if (lane == 0) bi::report_error(a.err, bi::kErrTimeout | bi::kWhereAttnSplit);
        return;
    }
#pragma unroll
    for (int e = 0; e < 2; ++e) {
        if (Lcol[e] == 0) continue;
        const int n = warp * 8 + 2 * (lane & 3) + e;
        const int64_t row = static_cast<int64_t>(q0 + r0 + rrcol[e]) * a.Hq + g * G + n % G;
#pragma unroll
        for (int mt = 0; mt < 8; ++mt) {
            const int d = 16 * mt + (lane >> 2);
            a.out[row * kD + d] = __float2bfloat16_rn(__fdiv_rn(Ar[mt][e], Lr[e]));
            a.out[row * kD + d + 8] = __float2bfloat16_rn(__fdiv_rn(Ar[mt][2 + e], Lr[e]));
        }
    }
}

// set once per device; any thread may race to set it, the attribute is idempotent
std::atomic<bool> g_attr_set[64] = {};

}  // namespace

extern "C" bi_status bi_prefill_attention(const void* q, const void* k_cache, const void* v_cache,
                                          const int32_t* block_table, int32_t max_pages_per_seq,
                                          const int32_t* seq_lens, const int32_t* q_indptr,
                                          int32_t S, int32_t T, int32_t Hq, int32_t Hkv, int32_t D,
                                          int32_t page_size, int32_t num_pages,
                                          int32_t max_q_len, int32_t max_seq_len, float scale,
                                          void* out, cudaStream_t stream) {
    if (S < 0 || T < 0 || Hq <= 0 || Hkv <= 0 || max_pages_per_seq < 1 || num_pages < 1 ||
        max_seq_len < 1 || max_q_len < 0)
        return BI_ERR_INVALID_ARG;
    if (!(scale > 0.f) || !std::isfinite(scale)) return BI_ERR_INVALID_ARG;
    if (D != kD || page_size != kPage) return BI_ERR_UNSUPPORTED_SHAPE;
    if (Hq % Hkv != 0 || Hq / Hkv > kMaxGroup) return BI_ERR_UNSUPPORTED_SHAPE;
    if (S > 65535) return BI_ERR_UNSUPPORTED_SHAPE;
    if (static_cast<int64_t>(num_pages) * Hkv * kPage >= (int64_t{1} << 31))
        return BI_ERR_UNSUPPORTED_SHAPE;
    if (static_cast<int64_t>(max_seq_len) > static_cast<int64_t>(max_pages_per_seq) * kPage)
        return BI_ERR_INVALID_ARG;
    if (max_q_len > max_seq_len) return BI_ERR_INVALID_ARG;
    if (S == 0 || T == 0 || max_q_len == 0) return BI_OK;
    if (!q || !k_cache || !v_cache || !block_table || !seq_lens || !q_indptr || !out)
        return BI_ERR_INVALID_ARG;
    if (!bi::aligned16(q) || !bi::aligned16(k_cache) || !bi::aligned16(v_cache) ||
        !bi::aligned16(out) || (reinterpret_cast<uintptr_t>(block_table) & 3) ||
        (reinterpret_cast<uintptr_t>(seq_lens) & 3) || (reinterpret_cast<uintptr_t>(q_indptr) & 3))
        return BI_ERR_MISALIGNED;

    CUtensorMap tk, tv;
    const uint64_t rows = static_cast<uint64_t>(num_pages) * Hkv * kPage;
    if (bi::encode_page_map(&tk, k_cache, rows) != CUDA_SUCCESS ||
        bi::encode_page_map(&tv, v_cache, rows) != CUDA_SUCCESS)
        return BI_ERR_CUDA;

    int dev = 0;
    if (cudaGetDevice(&dev) != cudaSuccess) return BI_ERR_CUDA;
    if (dev >= 0 && dev < 64 && !g_attr_set[dev]) {
        if (cudaFuncSetAttribute(prefill_attn_kernel, cudaFuncAttributeMaxDynamicSharedMemorySize,
                                 kSmemBytes) != cudaSuccess)
            return BI_ERR_CUDA;
        g_attr_set[dev] = true;
    }

    PrefillArgs args;
    args.q = static_cast<const __nv_bfloat16*>(q);
    args.block_table = block_table;
    args.seq_lens = seq_lens;
    args.q_indptr = q_indptr;
    args.out = static_cast<__nv_bfloat16*>(out);
    args.err = bi::device_error_word();
    args.max_pages_per_seq = max_pages_per_seq;
    args.Hq = Hq;
    args.Hkv = Hkv;
    args.group = Hq / Hkv;
    args.rows_per_tile = kCols / args.group;
    args.num_pages = num_pages;
    args.max_seq_len = max_seq_len;
    args.max_q_len = max_q_len;
    args.T = T;
    args.scale_log2 = static_cast<float>(static_cast<double>(scale) * 1.4426950408889634);
    const int tiles = (max_q_len + args.rows_per_tile - 1) / args.rows_per_tile;
    return bi::launch_pdl(prefill_attn_kernel, dim3(tiles, Hkv, S), dim3(kThreads), kSmemBytes,
                          stream, tk, tv, args) == cudaSuccess
               ? BI_OK
               : BI_ERR_CUDA;
}
