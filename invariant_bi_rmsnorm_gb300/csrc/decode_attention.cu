// bi_decode_attention: paged decode attention with fixed-size KV splits.
//
// "Defeating Nondeterminism in LLM Inference: The Core Role of Batch
// Invariance", section "3. Batch-Invariant Attention" (figures "Fixed Number
// Split KV Strategy" / "Fixed Size Split KV Strategy") and "Batch Invariance
// and Numerical Reproducibility" (a 1,000-token cache = three 256-token
// chunks plus one of 232): decode has too few query rows to fill the GPU, so
// the KV sequence is split -- but by a fixed split SIZE, so the reduction
// order of a sequence depends only on its own length.
//
// Kernel 1 (split): one CTA per (sequence s, kv-head g, group of consecutive
// chunks).  Chunk c is tokens [256c, min(256c + 256, L)), i.e. up to 16 pages
// of 16 tokens.  For each chunk, warp w (of 4) owns the chunk's pages w, w+4,
// w+8, w+12 and runs an online softmax over them in that order, for the
// Hq/Hkv query heads that share kv-head g.  Pages arrive by TMA (2-D tiled
// loads, 128-byte swizzle) into a 2-stage ring per warp that runs on across
// chunk boundaries.  Per page:
//     S^T[16 tok x 8 heads] = K_page[16 x 128] . Q^T[128 x 8]   (8 mma.sync)
//     p = exp2(S * scale * log2 e - m_new), rounded to bf16
//     O^T[128 x 8] = O^T * alpha + V^T[128 x 16] . P^T[16 x 8]   (8 mma.sync)
// At the end of each chunk the four warp states are folded in warp order
// 0..3 into the chunk partial (m, l, O).  If the CTA's group holds every
// chunk of the sequence, it folds the partials in ascending chunk order with
// the log-sum-exp rule and writes bf16(O / l); otherwise the partials go to
// the workspace.
// Kernel 2 (merge): for each (sequence, query head) not finished by one CTA,
// fold the partials in ascending chunk order -- the same fp32 operations in
// the same order -- and write bf16(O / l).
// How many chunks a CTA walks is chosen per launch to fill the GPU; it moves
// work between CTAs but never changes any operation or its order, so it
// cannot change a bit of the result.
//
// Tokens past the sequence end inside its last page are masked to -inf and
// their V rows are zeroed in shared memory before use, so whatever the cache
// holds there (a later token, or uninitialised bits) never reaches the result.
#include <cuda_bf16.h>

#include <algorithm>
#include <cmath>
#include <mutex>

#include "bi_internal.h"
#include "bi_ptx.cuh"

namespace {

constexpr int kD = 128;
constexpr int kPage = BI_PAGE_SIZE;             // 16 tokens
constexpr int kChunk = BI_DECODE_CHUNK;         // 256 tokens
constexpr int kPagesPerChunk = kChunk / kPage;  // 16
constexpr int kWarps = 4;
constexpr int kThreads = kWarps * 32;
constexpr int kStagesPerWarp = 2;
constexpr int kStages = kWarps * kStagesPerWarp;
constexpr int kHalfBytes = kPage * 64 * 2;         // 16 rows x 64 dims: one TMA box
constexpr int kMatBytes = 2 * kHalfBytes;          // one (page, kv-head) K or V block
constexpr int kStageBytes = 2 * kMatBytes;         // K + V
constexpr int kMaxGroup = 8;                       // query heads per kv-head (mma N)
constexpr int kMaxPagesPerCta = 512;                // pages one CTA walks (a chunk group)
constexpr int kMaxChunksPerCta = kMaxPagesPerCta / kPagesPerChunk;  // 32
constexpr int kFoldFloats = kMaxGroup * kD + kWarps * 2 * kMaxGroup;  // chunk-fold buffers
constexpr int kSmemBytes = kStages * kStageBytes + kFoldFloats * 4 + 4 * kMaxPagesPerCta +
                           8 * kStages + 1024 /*align*/;  // 71.2 KB: 3 CTAs per SM

// Byte offset of the 16-byte chunk `ch` (0..15) of row `r` (0..15) inside one
// K or V page block as laid down by two 16x64 TMA boxes with 128-byte
// swizzle: the box for dims [64*(ch/8), +64) starts at (ch/8)*2048, each row
// is 128 bytes, and the 16-byte unit index is XORed with (row % 8).
__device__ __forceinline__ uint32_t swz(int r, int ch) {
    return static_cast<uint32_t>((ch >> 3) * kHalfBytes + r * 128 + (((ch & 7) ^ (r & 7)) << 4));
}

struct SplitArgs {
    const __nv_bfloat16* q;
    const int32_t* block_table;
    const int32_t* seq_lens;
    __nv_bfloat16* out;
    float* ws_acc;  // [B][Hq][max_chunks][D]
    float* ws_ml;   // [B][Hq][max_chunks][2]
    uint32_t* err;
    int max_pages_per_seq;
    int Hq, Hkv, group;
    int num_pages;
    int max_seq_len;
    int max_chunks;
    int num_splits;    // 0: fixed 256-token chunks; > 0: fixed split count (comparison variant)
    int chunks_per_cta;  // consecutive chunks one CTA walks (a schedule choice only)
    float scale_log2;  // scale * log2(e)
};

// Chunk geometry of one sequence of L tokens: pages per chunk and chunk count.
// Fixed split size (num_splits == 0, the batch-invariant method): 16 pages =
// 256 tokens per chunk, whatever L is.  Fixed split count (num_splits > 0),
// the strategy the pages warn against and kept here only as a comparison: the
// sequence's pages are cut into num_splits nearly equal runs, so the chunk
// size, and with it the reduction order, changes as L grows.
__device__ __forceinline__ void chunk_geometry(int L, int num_splits, int& ppc, int& nch) {
    const int npg = (L + kPage - 1) / kPage;
    ppc = num_splits > 0 ? (npg + num_splits - 1) / num_splits : kPagesPerChunk;
    nch = (npg + ppc - 1) / ppc;
}

__global__ void __launch_bounds__(kThreads)
    attn_split_kernel(const __grid_constant__ CUtensorMap tmap_k,
                      const __grid_constant__ CUtensorMap tmap_v, const SplitArgs a) {
    const int cg = blockIdx.x;  // chunk group
    const int g = blockIdx.y;
    const int s = blockIdx.z;
    const int tid = threadIdx.x;
    const int warp = tid >> 5;
    const int lane = tid & 31;

    const int L = a.seq_lens[s];
    if (L < 1 || L > a.max_seq_len) {
        if (tid == 0 && cg == 0 && g == 0) bi::report_error(a.err, bi::kErrBadInput | bi::kWhereAttnSplit);
        return;
    }
    int ppc, nch;
    chunk_geometry(L, a.num_splits, ppc, nch);
    const int c0 = cg * a.chunks_per_cta;
    if (c0 >= nch) return;
    const int c1 = min(nch, c0 + a.chunks_per_cta);
    const bool whole = (c0 == 0 && c1 == nch);  // this CTA folds the whole sequence
    const int npg_total = (L + kPage - 1) / kPage;
    const int pg0 = c0 * ppc;
    const int npg_group = min(c1 * ppc, npg_total) - pg0;

    extern __shared__ uint8_t smem_raw[];
    uint8_t* smem = reinterpret_cast<uint8_t*>(
        (reinterpret_cast<uintptr_t>(smem_raw) + 1023) & ~static_cast<uintptr_t>(1023));
    float* fold_o = reinterpret_cast<float*>(smem + kStages * kStageBytes);  // [8 heads][128]
    float* fold_ml = fold_o + kMaxGroup * kD;                                // [4 warps][m 8, l 8]
    int32_t* rows_s = reinterpret_cast<int32_t*>(fold_ml + kWarps * 2 * kMaxGroup);  // TMA row per page
    uint64_t* bars = reinterpret_cast<uint64_t*>(rows_s + kMaxPagesPerCta);
    __shared__ int bad_page;

    if (tid == 0) {
        bad_page = 0;
        for (int i = 0; i < kStages; ++i) bi::mbar_init(&bars[i], 1);
        bi::fence_mbar_init();
        bi::tma_prefetch_desc(&tmap_k);
        bi::tma_prefetch_desc(&tmap_v);
    }
    __syncthreads();
    for (int i = tid; i < npg_group; i += kThreads) {
        const int pg = a.block_table[static_cast<int64_t>(s) * a.max_pages_per_seq + pg0 + i];
        if (pg < 0 || pg >= a.num_pages) {
            bad_page = 1;
        } else {
            rows_s[i] = (pg * a.Hkv + g) * kPage;
        }
    }
    __syncthreads();
    if (bad_page) {
        if (tid == 0) bi::report_error(a.err, bi::kErrBadInput | bi::kWhereAttnSplit);
        return;
    }

    auto pages_in = [&](int c) { return min(ppc, npg_total - c * ppc); };
    auto stage_ptr = [&](int st) { return smem + st * kStageBytes; };

    // This warp's pages, in order: for each chunk of the group, pages warp,
    // warp + 4, warp + 8, ... of that chunk.  The loader runs two pages ahead
    // of the compute loop through a 2-stage ring; every lane tracks the
    // loader position, lane 0 issues the copies.
    int lc = c0, lp = warp, lj = 0;
    while (lc < c1 && lp >= pages_in(lc)) { ++lc; lp = warp; }
    auto issue_next = [&]() {
        if (lc >= c1) return;
        if (lane == 0) {
            const int st = warp * kStagesPerWarp + (lj & 1);
            uint8_t* kd = stage_ptr(st);
            uint8_t* vd = kd + kMatBytes;
            const int row = rows_s[(lc - c0) * ppc + lp];
            bi::mbar_arrive_expect_tx(&bars[st], kStageBytes);
            bi::tma_load_2d(kd, &tmap_k, &bars[st], 0, row);
            bi::tma_load_2d(kd + kHalfBytes, &tmap_k, &bars[st], 64, row);
            bi::tma_load_2d(vd, &tmap_v, &bars[st], 0, row);
            bi::tma_load_2d(vd + kHalfBytes, &tmap_v, &bars[st], 64, row);
        }
        ++lj;
        lp += kWarps;
        while (lc < c1 && lp >= pages_in(lc)) { ++lc; lp = warp; }
    };
    issue_next();
    issue_next();

    // Q^T as the mma B operand: lane holds head (lane/4) of the group and
    // dims 16ks + 2(lane%4) + {0,1} (b0) and +8 (b1).
    const int qh = lane >> 2;
    uint32_t qb0[8], qb1[8];
    {
        const bool valid = qh < a.group;
        const __nv_bfloat16* qp =
            a.q + (static_cast<int64_t>(s) * a.Hq + g * a.group + (valid ? qh : 0)) * kD + 2 * (lane & 3);
#pragma unroll
        for (int ks = 0; ks < 8; ++ks) {
            qb0[ks] = valid ? *reinterpret_cast<const uint32_t*>(qp + 16 * ks) : 0u;
            qb1[ks] = valid ? *reinterpret_cast<const uint32_t*>(qp + 16 * ks + 8) : 0u;
        }
    }

    // ldmatrix lane roles
    const int lm_j = lane >> 3;  // which 8x8 matrix this lane addresses
    const int lm_r = lane & 7;   // row within it
    const int h0 = 2 * (lane & 3);
    const int d = tid;           // output dim this thread owns in the folds
    float Mr[kMaxGroup], Lr[kMaxGroup], Ar[kMaxGroup];  // running fold over chunks (whole)
    bool timed_out = false;
    int j = 0;  // this warp's page counter (matches the loader's)

    for (int c = c0; c < c1; ++c) {
        float m_run[2] = {-INFINITY, -INFINITY};
        float l_run[2] = {0.f, 0.f};
        float acc[8][4];
#pragma unroll
        for (int mt = 0; mt < 8; ++mt) acc[mt][0] = acc[mt][1] = acc[mt][2] = acc[mt][3] = 0.f;

        const int np = pages_in(c);
        for (int p = warp; p < np; p += kWarps, ++j) {
            const int st = warp * kStagesPerWarp + (j & 1);
            if (timed_out) continue;
            if (!bi::mbar_wait(&bars[st], (j >> 1) & 1)) {
                timed_out = true;
                continue;
            }
            const uint32_t ks_base = bi::smem_u32(stage_ptr(st));
            const uint32_t vs_base = ks_base + kMatBytes;
            const int valid = min(kPage, L - (c * ppc + p) * kPage);
            if (valid < kPage) {
                // zero V rows past the sequence end (16-byte units)
                uint8_t* vd = stage_ptr(st) + kMatBytes;
                for (int idx = lane; idx < (kPage - valid) * 16; idx += 32) {
                    const int r = valid + (idx >> 4), ch = idx & 15;
                    *reinterpret_cast<uint4*>(vd + swz(r, ch)) = make_uint4(0, 0, 0, 0);
                }
                __syncwarp();
            }

            // S^T = K . Q^T  (tokens on M, heads on N), dims in ascending 16-blocks
            float sc[4] = {0.f, 0.f, 0.f, 0.f};
#pragma unroll
            for (int ks = 0; ks < 8; ++ks) {
                uint32_t a0, a1, a2, a3;
                const int r = lm_r + 8 * (lm_j & 1);
                const int ch = 2 * ks + (lm_j >> 1);
                bi::ldmatrix_x4(ks_base + swz(r, ch), a0, a1, a2, a3);
                bi::mma_bf16_16816(sc, a0, a1, a2, a3, qb0[ks], qb1[ks]);
            }
            // sc[0], sc[1]: token lane/4, heads 2(lane%4)+{0,1}; sc[2], sc[3]: token +8
            const int tokA = lane >> 2, tokB = tokA + 8;
            const float x0 = tokA < valid ? sc[0] * a.scale_log2 : -INFINITY;
            const float x1 = tokA < valid ? sc[1] * a.scale_log2 : -INFINITY;
            const float x2 = tokB < valid ? sc[2] * a.scale_log2 : -INFINITY;
            const float x3 = tokB < valid ? sc[3] * a.scale_log2 : -INFINITY;
            float mx0 = fmaxf(x0, x2), mx1 = fmaxf(x1, x3);
#pragma unroll
            for (int off = 4; off <= 16; off <<= 1) {
                mx0 = fmaxf(mx0, __shfl_xor_sync(0xffffffffu, mx0, off));
                mx1 = fmaxf(mx1, __shfl_xor_sync(0xffffffffu, mx1, off));
            }
            const float mn0 = fmaxf(m_run[0], mx0), mn1 = fmaxf(m_run[1], mx1);
            const float al0 = exp2f(m_run[0] - mn0), al1 = exp2f(m_run[1] - mn1);
            const uint32_t pA = bi::pack_bf16x2(exp2f(x0 - mn0), exp2f(x1 - mn1));
            const uint32_t pB = bi::pack_bf16x2(exp2f(x2 - mn0), exp2f(x3 - mn1));
            // the row sums use the same bf16-rounded weights that multiply V
            float ps0 = __uint_as_float(pA << 16) + __uint_as_float(pB << 16);
            float ps1 = __uint_as_float(pA & 0xffff0000u) + __uint_as_float(pB & 0xffff0000u);
#pragma unroll
            for (int off = 4; off <= 16; off <<= 1) {
                ps0 += __shfl_xor_sync(0xffffffffu, ps0, off);
                ps1 += __shfl_xor_sync(0xffffffffu, ps1, off);
            }
            l_run[0] = __fmaf_rn(l_run[0], al0, ps0);
            l_run[1] = __fmaf_rn(l_run[1], al1, ps1);
            m_run[0] = mn0;
            m_run[1] = mn1;
#pragma unroll
            for (int mt = 0; mt < 8; ++mt) {
                acc[mt][0] *= al0;
                acc[mt][1] *= al1;
                acc[mt][2] *= al0;
                acc[mt][3] *= al1;
            }
            // P^T fragments (tokens on K, heads on N) by an in-register transpose
            const uint32_t pb0 = bi::movmatrix_trans(pA);
            const uint32_t pb1 = bi::movmatrix_trans(pB);
            // O^T += V^T . P^T, dims in ascending 16-blocks
#pragma unroll
            for (int mt = 0; mt < 8; ++mt) {
                uint32_t a0, a1, a2, a3;
                const int r = lm_r + 8 * (lm_j >> 1);
                const int ch = 2 * mt + (lm_j & 1);
                bi::ldmatrix_x4_trans(vs_base + swz(r, ch), a0, a1, a2, a3);
                bi::mma_bf16_16816(acc[mt], a0, a1, a2, a3, pb0, pb1);
            }
            // hand the stage back to TMA for this warp's page two ahead
            bi::fence_proxy_async_smem();
            __syncwarp();
            issue_next();
        }

        // ---- fold the four warp states of chunk c, in warp order 0..3 ----
        //   M = max_w m_w;  f_w = 2^(m_w - M);
        //   l = fma(l_3, f_3, fma(l_2, f_2, fma(l_1, f_1, fma(l_0, f_0, 0))))
        //   O = the same fma chain over the warps' O, which the warps apply
        //       to one shared [heads][128] buffer one after another.
        if (lane < 4) {
            fold_ml[warp * 2 * kMaxGroup + h0] = m_run[0];
            fold_ml[warp * 2 * kMaxGroup + h0 + 1] = m_run[1];
            fold_ml[warp * 2 * kMaxGroup + kMaxGroup + h0] = l_run[0];
            fold_ml[warp * 2 * kMaxGroup + kMaxGroup + h0 + 1] = l_run[1];
        }
        __syncthreads();
        {
            float Mh0 = fold_ml[h0], Mh1 = fold_ml[h0 + 1];
#pragma unroll
            for (int w = 1; w < kWarps; ++w) {
                Mh0 = fmaxf(Mh0, fold_ml[w * 2 * kMaxGroup + h0]);
                Mh1 = fmaxf(Mh1, fold_ml[w * 2 * kMaxGroup + h0 + 1]);
            }
            const float f0 = exp2f(m_run[0] - Mh0), f1 = exp2f(m_run[1] - Mh1);
#pragma unroll 1
            for (int w = 0; w < kWarps; ++w) {
                if (warp == w) {
#pragma unroll
                    for (int mt = 0; mt < 8; ++mt) {
                        const int dd = 16 * mt + (lane >> 2);
                        float* o0 = fold_o + h0 * kD + dd;
                        float* o1 = fold_o + (h0 + 1) * kD + dd;
                        const float p00 = w ? o0[0] : 0.f, p10 = w ? o1[0] : 0.f;
                        const float p01 = w ? o0[8] : 0.f, p11 = w ? o1[8] : 0.f;
                        o0[0] = __fmaf_rn(acc[mt][0], f0, p00);
                        o1[0] = __fmaf_rn(acc[mt][1], f1, p10);
                        o0[8] = __fmaf_rn(acc[mt][2], f0, p01);
                        o1[8] = __fmaf_rn(acc[mt][3], f1, p11);
                    }
                }
                __syncthreads();
            }
        }
#pragma unroll
        for (int h = 0; h < kMaxGroup; ++h) {
            if (h >= a.group) break;
            float M = fold_ml[h];
#pragma unroll
            for (int w = 1; w < kWarps; ++w) M = fmaxf(M, fold_ml[w * 2 * kMaxGroup + h]);
            float Ls = 0.f;
#pragma unroll
            for (int w = 0; w < kWarps; ++w) {
                const float* ml = fold_ml + w * 2 * kMaxGroup;
                Ls = __fmaf_rn(ml[kMaxGroup + h], exp2f(ml[h] - M), Ls);
            }
            const float A = fold_o[h * kD + d];
            if (whole) {
                // the merge kernel's fold, chunk by chunk in ascending order
                if (c == c0) {
                    Mr[h] = M;
                    Lr[h] = Ls;
                    Ar[h] = A;
                } else {
                    const float Mn = fmaxf(Mr[h], M);
                    const float fo = exp2f(Mr[h] - Mn), fc = exp2f(M - Mn);
                    Lr[h] = __fmaf_rn(Ls, fc, __fmul_rn(Lr[h], fo));
                    Ar[h] = __fmaf_rn(A, fc, __fmul_rn(Ar[h], fo));
                    Mr[h] = Mn;
                }
            } else {
                const int64_t row = static_cast<int64_t>(s) * a.Hq + g * a.group + h;
                const int64_t pidx = row * a.max_chunks + c;
                a.ws_acc[pidx * kD + d] = A;
                if (d == 0) {
                    a.ws_ml[pidx * 2] = M;
                    a.ws_ml[pidx * 2 + 1] = Ls;
                }
            }
        }
        __syncthreads();  // fold area free for the next chunk
    }

    if (timed_out && lane == 0) bi::report_error(a.err, bi::kErrTimeout | bi::kWhereAttnSplit);
    if (whole) {
#pragma unroll
        for (int h = 0; h < kMaxGroup; ++h) {
            if (h >= a.group) break;
            const int64_t row = static_cast<int64_t>(s) * a.Hq + g * a.group + h;
            a.out[row * kD + d] = __float2bfloat16_rn(__fdiv_rn(Ar[h], Lr[h]));
        }
    }
}

// Fold the chunk partials of one (sequence, query head) in ascending chunk
// order:  M' = max(M, m_c);  l' = l 2^(M-M') + l_c 2^(m_c-M');
//         O' = O 2^(M-M') + O_c 2^(m_c-M');   out = bf16(O / l).
__global__ void __launch_bounds__(kD)
    attn_merge_kernel(const int32_t* __restrict__ seq_lens, const float* __restrict__ ws_acc,
                      const float* __restrict__ ws_ml, __nv_bfloat16* __restrict__ out, int Hq,
                      int max_chunks, int max_seq_len, int num_splits, int chunks_per_cta) {
    const int hq = blockIdx.x;
    const int s = blockIdx.y;
    const int d = threadIdx.x;
    const int L = seq_lens[s];
    if (L < 1 || L > max_seq_len) return;  // reported by the split kernel
    int ppc, nch;
    chunk_geometry(L, num_splits, ppc, nch);
    if (nch <= chunks_per_cta) return;  // one CTA walked and folded every chunk
    const int64_t base = (static_cast<int64_t>(s) * Hq + hq) * max_chunks;
    float M = ws_ml[base * 2];
    float Ls = ws_ml[base * 2 + 1];
    float A = ws_acc[base * kD + d];
    for (int c = 1; c < nch; ++c) {
        const float mc = ws_ml[(base + c) * 2];
        const float lc = ws_ml[(base + c) * 2 + 1];
        const float ac = ws_acc[(base + c) * kD + d];
        const float Mn = fmaxf(M, mc);
        const float fo = exp2f(M - Mn), fc = exp2f(mc - Mn);
        Ls = __fmaf_rn(lc, fc, __fmul_rn(Ls, fo));
        A = __fmaf_rn(ac, fc, __fmul_rn(A, fo));
        M = Mn;
    }
    out[(static_cast<int64_t>(s) * Hq + hq) * kD + d] = __float2bfloat16_rn(__fdiv_rn(A, Ls));
}

int ceil_div(int64_t a, int64_t b) { return static_cast<int>((a + b - 1) / b); }

bool g_attr_set[64] = {};

}  // namespace

extern "C" size_t bi_decode_attention_workspace_size(int32_t B, int32_t Hq, int32_t D,
                                                     int32_t max_seq_len) {
    if (B < 0 || Hq <= 0 || D <= 0 || max_seq_len < 1) return 0;
    const int64_t chunks = ceil_div(max_seq_len, kChunk);
    if (chunks < 2) return 0;
    return static_cast<size_t>(B) * Hq * chunks * (static_cast<size_t>(D) + 2) * sizeof(float);
}

extern "C" int32_t bi_decode_num_chunks(int32_t seq_len) {
    return seq_len < 1 ? 0 : ceil_div(seq_len, kChunk);
}

extern "C" int32_t bi_decode_chunk_len(int32_t seq_len, int32_t c) {
    const int32_t n = bi_decode_num_chunks(seq_len);
    if (c < 0 || c >= n) return 0;
    return c < n - 1 ? kChunk : seq_len - (n - 1) * kChunk;
}

namespace {

// Validate and launch split + merge.  num_splits == 0 is the batch-invariant
// fixed split size; num_splits > 0 the fixed-split-count comparison variant,
// whose workspace then holds num_splits partials per (sequence, query head).
bi_status launch_attention(const void* q, const void* k_cache, const void* v_cache,
                           const int32_t* block_table, int32_t max_pages_per_seq,
                           const int32_t* seq_lens, int32_t B, int32_t Hq, int32_t Hkv, int32_t D,
                           int32_t page_size, int32_t num_pages, int32_t max_seq_len, float scale,
                           void* out, void* workspace, size_t workspace_bytes, int32_t num_splits,
                           cudaStream_t stream) {
    if (B < 0 || Hq <= 0 || Hkv <= 0 || max_pages_per_seq < 1 || num_pages < 1 ||
        max_seq_len < 1 || num_splits < 0)
        return BI_ERR_INVALID_ARG;
    if (!(scale > 0.f) || !std::isfinite(scale)) return BI_ERR_INVALID_ARG;
    if (D != kD || page_size != kPage) return BI_ERR_UNSUPPORTED_SHAPE;
    if (Hq % Hkv != 0 || Hq / Hkv > kMaxGroup) return BI_ERR_UNSUPPORTED_SHAPE;
    if (B > 65535) return BI_ERR_UNSUPPORTED_SHAPE;
    if (static_cast<int64_t>(num_pages) * Hkv * kPage >= (int64_t{1} << 31))
        return BI_ERR_UNSUPPORTED_SHAPE;
    if (static_cast<int64_t>(max_seq_len) > static_cast<int64_t>(max_pages_per_seq) * kPage)
        return BI_ERR_INVALID_ARG;
    if (num_splits > 0 && ceil_div(ceil_div(max_seq_len, kPage), num_splits) > kMaxPagesPerCta)
        return BI_ERR_UNSUPPORTED_SHAPE;
    if (B == 0) return BI_OK;
    if (!q || !k_cache || !v_cache || !block_table || !seq_lens || !out) return BI_ERR_INVALID_ARG;
    if (!bi::aligned16(q) || !bi::aligned16(k_cache) || !bi::aligned16(v_cache) ||
        !bi::aligned16(out) || (reinterpret_cast<uintptr_t>(block_table) & 3) ||
        (reinterpret_cast<uintptr_t>(seq_lens) & 3))
        return BI_ERR_MISALIGNED;
    const int max_chunks = num_splits > 0 ? num_splits : ceil_div(max_seq_len, kChunk);
    const size_t need = max_chunks >= 2 ? static_cast<size_t>(B) * Hq * max_chunks *
                                              (static_cast<size_t>(D) + 2) * sizeof(float)
                                        : 0;
    if (need > 0) {
        if (!workspace || workspace_bytes < need) return BI_ERR_WORKSPACE_TOO_SMALL;
        if (!bi::aligned16(workspace)) return BI_ERR_MISALIGNED;
    }

    CUtensorMap tk, tv;
    const uint64_t rows = static_cast<uint64_t>(num_pages) * Hkv * kPage;
    if (bi::encode_tensor_map_2d(&tk, k_cache, kD, rows, kD * 2, 64, kPage) != CUDA_SUCCESS ||
        bi::encode_tensor_map_2d(&tv, v_cache, kD, rows, kD * 2, 64, kPage) != CUDA_SUCCESS)
        return BI_ERR_CUDA;

    int dev = 0;
    if (cudaGetDevice(&dev) != cudaSuccess) return BI_ERR_CUDA;
    if (dev >= 0 && dev < 64 && !g_attr_set[dev]) {
        if (cudaFuncSetAttribute(attn_split_kernel, cudaFuncAttributeMaxDynamicSharedMemorySize,
                                 kSmemBytes) != cudaSuccess)
            return BI_ERR_CUDA;
        g_attr_set[dev] = true;
    }

    SplitArgs args;
    args.q = static_cast<const __nv_bfloat16*>(q);
    args.block_table = block_table;
    args.seq_lens = seq_lens;
    args.out = static_cast<__nv_bfloat16*>(out);
    args.ws_acc = need ? static_cast<float*>(workspace) : nullptr;
    args.ws_ml = need ? static_cast<float*>(workspace) +
                            static_cast<size_t>(B) * Hq * max_chunks * kD
                      : nullptr;
    args.err = bi::device_error_word();
    args.max_pages_per_seq = max_pages_per_seq;
    args.Hq = Hq;
    args.Hkv = Hkv;
    args.group = Hq / Hkv;
    args.num_pages = num_pages;
    args.max_seq_len = max_seq_len;
    args.max_chunks = max_chunks;
    args.num_splits = num_splits;
    args.scale_log2 = static_cast<float>(static_cast<double>(scale) * 1.4426950408889634);

    // Schedule (never the arithmetic): how many consecutive chunks one CTA
    // walks.  Enough CTAs for about four waves of the resident slots; a
    // sequence whose chunks all fall to one CTA is folded there, the rest by
    // the merge kernel -- both apply the same fold in the same chunk order.
    int cpc = 1;
    if (num_splits == 0) {
        const int64_t slots = static_cast<int64_t>(bi::sm_count()) * 3;  // 3 CTAs per SM
        const int64_t units = static_cast<int64_t>(B) * Hkv * max_chunks;
        cpc = static_cast<int>(std::min<int64_t>(kMaxChunksPerCta,
                                                 std::max<int64_t>(1, units / (4 * slots))));
    }
    args.chunks_per_cta = cpc;
    const int groups = ceil_div(max_chunks, cpc);

    attn_split_kernel<<<dim3(groups, Hkv, B), kThreads, kSmemBytes, stream>>>(tk, tv, args);
    if (cudaGetLastError() != cudaSuccess) return BI_ERR_CUDA;
    if (max_chunks > cpc) {
        attn_merge_kernel<<<dim3(Hq, B), kD, 0, stream>>>(seq_lens, args.ws_acc, args.ws_ml,
                                                          args.out, Hq, max_chunks, max_seq_len,
                                                          num_splits, cpc);
        if (cudaGetLastError() != cudaSuccess) return BI_ERR_CUDA;
    }
    return BI_OK;
}

}  // namespace

extern "C" bi_status bi_decode_attention(const void* q, const void* k_cache, const void* v_cache,
                                         const int32_t* block_table, int32_t max_pages_per_seq,
                                         const int32_t* seq_lens, int32_t B, int32_t Hq,
                                         int32_t Hkv, int32_t D, int32_t page_size,
                                         int32_t num_pages, int32_t max_seq_len, float scale,
                                         void* out, void* workspace, size_t workspace_bytes,
                                         cudaStream_t stream) {
    return launch_attention(q, k_cache, v_cache, block_table, max_pages_per_seq, seq_lens, B, Hq,
                            Hkv, D, page_size, num_pages, max_seq_len, scale, out, workspace,
                            workspace_bytes, 0, stream);
}

extern "C" bi_status bi_decode_attention_fixed_splits(
    const void* q, const void* k_cache, const void* v_cache, const int32_t* block_table,
    int32_t max_pages_per_seq, const int32_t* seq_lens, int32_t B, int32_t Hq, int32_t Hkv,
    int32_t D, int32_t page_size, int32_t num_pages, int32_t max_seq_len, float scale,
    int32_t num_splits, void* out, void* workspace, size_t workspace_bytes, cudaStream_t stream) {
    if (num_splits < 1) return BI_ERR_INVALID_ARG;
    return launch_attention(q, k_cache, v_cache, block_table, max_pages_per_seq, seq_lens, B, Hq,
                            Hkv, D, page_size, num_pages, max_seq_len, scale, out, workspace,
                            workspace_bytes, num_splits, stream);
}

// ---------------------------------------------------------------------------
// bi_decode_attention_noalloc: the same computation for callers that cannot
// allocate device memory at call time.  The chunk partials live in a fixed
// array that is part of the library's own device image instead of a
// caller-provided workspace.
namespace {

// Capacity in chunk partials (one per sequence x query head x 256-token
// chunk), each kD + 2 floats: 65536 x 130 x 4 bytes = 32.5 MiB per device.
constexpr int64_t kNoAllocPartials = 65536;
constexpr size_t kNoAllocBytes = static_cast<size_t>(kNoAllocPartials) * (kD + 2) * sizeof(float);

static __device__ __align__(256) float g_noalloc_scratch[kNoAllocPartials * (kD + 2)];

std::mutex g_noalloc_mu;
void* g_noalloc_ptr[64] = {};

// Device address of g_noalloc_scratch on the current device.  The host-side
// name of the array is only a stand-in; the address a kernel can use comes
// from cudaGetSymbolAddress, resolved once per device with that device
// current and cached.
void* noalloc_scratch_address(int dev) {
    std::lock_guard<std::mutex> lk(g_noalloc_mu);
    if (!g_noalloc_ptr[dev]) {
        void* p = nullptr;
        if (cudaGetSymbolAddress(&p, g_noalloc_scratch) != cudaSuccess || !p) return nullptr;
        g_noalloc_ptr[dev] = p;
    }
    return g_noalloc_ptr[dev];
}

}  // namespace

extern "C" bi_status bi_decode_attention_noalloc(const void* q, const void* k_cache,
                                                 const void* v_cache, const int32_t* block_table,
                                                 int32_t max_pages_per_seq,
                                                 const int32_t* seq_lens, int32_t B, int32_t Hq,
                                                 int32_t Hkv, int32_t D, int32_t page_size,
                                                 int32_t num_pages, int32_t max_seq_len,
                                                 float scale, void* out, cudaStream_t stream) {
    if (B < 0 || Hq <= 0 || max_seq_len < 1) return BI_ERR_INVALID_ARG;
    const int64_t partials = static_cast<int64_t>(B) * Hq * ceil_div(max_seq_len, kChunk);
    const size_t need = bi_decode_attention_workspace_size(B, Hq, D, max_seq_len);
    if (need > kNoAllocBytes || partials > kNoAllocPartials) return BI_ERR_WORKSPACE_TOO_SMALL;
    void* ws = nullptr;
    if (need > 0) {
        int dev = -1;
        if (cudaGetDevice(&dev) != cudaSuccess || dev < 0 || dev >= 64) return BI_ERR_CUDA;
        ws = noalloc_scratch_address(dev);
        if (!ws) return BI_ERR_CUDA;
    }
    return bi_decode_attention(q, k_cache, v_cache, block_table, max_pages_per_seq, seq_lens, B,
                               Hq, Hkv, D, page_size, num_pages, max_seq_len, scale, out, ws,
                               need > 0 ? kNoAllocBytes : 0, stream);
}
