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
// Kernel 1 (split): one CTA (4 warps) per (sequence s, kv-head g, group of
// consecutive chunks).  Chunk c is tokens [256c, min(256c + 256, L)), i.e. up
// to 16 pages of 16 tokens.  Warp w takes chunks c0 + w, c0 + w + 4, ... of
// the group and, for the Hq/Hkv query heads sharing kv-head g, runs one online
// softmax over each chunk's pages 0, 1, 2, ... in order (attn_common.cuh
// gives the per-page arithmetic).  Pages arrive by TMA (one 3-D tiled load
// per page block of K and of V, 128-byte swizzle) into a 2-stage ring per
// warp.  A chunk's final state is its
// partial (m, l, O).  If the CTA's group holds every chunk of the sequence,
// the partials are folded in ascending chunk order inside the CTA (warp by
// warp after each round of four chunks) and bf16(O / l) is written.
// Otherwise the CTA writes its chunks' partials to the workspace and counts
// itself in on an integer arrival counter of its (sequence, kv-head); the CTA
// that arrives last reads every chunk's partial back and folds them in
// ascending chunk order -- the same fp32 operations in the same order -- then
// writes bf16(O / l) and returns the counter to zero.  Which CTA arrives last
// decides only who folds, never what is folded or in which order.  No float
// atomics: the counter is a plain integer add.
// Kernel 1' (pair), instead of kernel 1 for launches of a few sequences: the
// same chunks and per-page operations with two warps per chunk (one forms
// the scores, one runs the softmax update and the output products), every
// chunk's partial folded by the last CTA to arrive.
// Kernel 2 (merge), only for launches with more (sequence, kv-head) pairs
// than the workspace has counters: the same fold as a separate kernel.
// How many chunks a CTA walks is chosen per launch to fill the GPU; it moves
// work between CTAs but never changes any operation or its order, so it
// cannot change a bit of the result.
//
// Tokens past the sequence end inside its last page are masked to -inf and
// their V rows are zeroed in shared memory before use, so whatever the cache
// holds there (a later token, or uninitialised bits) never reaches the result.
#include <cuda_bf16.h>

#include <algorithm>
#include <atomic>
#include <cmath>
#include <mutex>

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
constexpr int kWarps = 4;
constexpr int kThreads = kWarps * 32;
constexpr int kMaxPagesPerCta = 512;                                // pages one CTA walks
constexpr int kMaxChunksPerCta = kMaxPagesPerCta / kPagesPerChunk;  // 32
constexpr int kFoldFloats = kMaxGroup * kD + 2 * kMaxGroup;          // running fold (O, M, L)
// Pages in flight per warp (its private TMA ring): 72.8 KB per CTA, 3 CTAs
// per SM.  A six-deep ring (one CTA per SM) was measured as no faster at one
// sequence and slower from eight sequences up: a warp's chunk is paced by its
// per-page arithmetic, not by HBM latency.
constexpr int kSPW = 2;
constexpr int kStages = kWarps * kSPW;
constexpr int kSmemBytes = kStages * kStageBytes + kFoldFloats * 4 + 4 * kMaxPagesPerCta +
                           8 * kStages + 1024 /*align*/;
// Arrival counters at the start of the workspace: one uint32 per (sequence,
// kv-head), low 16 bits = CTAs arrived, high bits set by a CTA that found a bad
// page index.  Every call leaves them zero.
constexpr int64_t kMaxCounters = BI_DECODE_COUNTER_BYTES / 4;
constexpr uint32_t kArrive = 1u;
constexpr uint32_t kArriveBad = 0x10001u;

struct SplitArgs {
    const __nv_bfloat16* q;
    const int32_t* block_table;
    const int32_t* seq_lens;
    __nv_bfloat16* out;
    float* ws_acc;  // [B][Hq][max_chunks][D]
    float* ws_ml;   // [B][Hq][max_chunks][2]
    uint32_t* counters;  // [B][Hkv] arrival counters; nullptr: the merge kernel folds
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

// The fold of one (sequence, kv-head) by the CTA that arrived last: for each
// of its G query heads h and dims d (thread d), the chunk partials are folded
// in ascending chunk order,
//     M' = max(M, m_c);  fo = 2^(M - M');  fc = 2^(m_c - M');
//     l' = fma(l_c, fc, l * fo);  O' = fma(O_c, fc, O * fo),
// starting from chunk 0's (m, l, O), and bf16(O / l) is written -- exactly the
// merge kernel's operations, on the same values.  Only the schedule differs:
//   - the running maxima M are a prefix maximum, exact in any evaluation
//     order, so a warp computes them for 32 chunks at once by a shuffle scan,
//     and with them every chunk's factors fo, fc;
//   - the recurrences of l and O then run in every thread from shared
//     memory, loads issued a few chunks ahead (each thread computes its
//     heads' l itself, the same operations on the same values).
// The partials are staged in shared memory (the TMA ring, free by now) a
// batch of chunks at a time: the (m, l) pairs first, then the unnormalised
// outputs by cp.async while the factors are computed.  ws reads go through L2
// only (ld.cg, cp.async.cg): the data was written by other CTAs.
template <int G>
__device__ __forceinline__ void fold_sequence(const SplitArgs& a, int s, int g, int nch,
                                              uint8_t* stage, float* small, int tid) {
    constexpr int kcb = (kStages * kStageBytes) / (G * kD * 4);  // chunks per batch, G*kcb <= 128
    // thread -> (head, G consecutive dims) when G divides 128 (vector loads,
    // one head per warp at G = 4); otherwise thread d -> dim d of every head
    constexpr bool kVec = kThreads % G == 0 && kD == kThreads;  // G = 1, 2, 4, 8
    constexpr int TPH = kVec ? kThreads / G : kThreads;  // threads per head
    constexpr int NH = kVec ? 1 : G;                     // heads per thread
    constexpr int ND = kVec ? G : 1;                     // dims per thread
    constexpr int U = kVec ? 4 : (16 / G > 0 ? 16 / G : 1);  // chunks loaded ahead
    float* acc_s = reinterpret_cast<float*>(stage);  // [kcb][G][kD]
    float* ml_s = small;                             // [kcb][G][2]  (m_c, l_c)
    float4* fl = reinterpret_cast<float4*>(small + 256);  // [kcb][G]  (fo, fc, l_c, -)
    float* mcarry = small + 768;                     // [G] running max before the batch
    const int lane = tid & 31, warp = tid >> 5;
    const int64_t row0 = static_cast<int64_t>(s) * a.Hq + g * G;
    const int h0 = kVec ? tid / TPH : 0;               // this thread's (first) head
    const int d0 = kVec ? (tid % TPH) * ND : tid;      // this thread's first dim
    float A[NH][ND], Lr[NH];
#pragma unroll
    for (int j = 0; j < NH; ++j) {
        Lr[j] = 0.f;
#pragma unroll
        for (int e = 0; e < ND; ++e) A[j][e] = 0.f;
    }
    for (int cb = 0; cb < nch; cb += kcb) {
        const int nb = min(kcb, nch - cb);
        float2 ml = make_float2(0.f, 0.f);  // one (m, l) pair per thread (nb * G <= 128)
        const int mi = tid / G, mh = tid - mi * G;
        if (mi < nb)
            ml = __ldcg(reinterpret_cast<const float2*>(a.ws_ml + ((row0 + mh) * a.max_chunks + cb + mi) * 2));
        for (int idx = tid; idx < nb * G * (kD / 4); idx += kThreads) {
            const int v = idx % (kD / 4);
            const int hg = idx / (kD / 4);  // i * G + h
            const int i = hg / G, h = hg - i * G;
            bi::cp_async_16(acc_s + hg * kD + 4 * v,
                            a.ws_acc + ((row0 + h) * a.max_chunks + cb + i) * kD + 4 * v);
        }
        if (mi < nb) *reinterpret_cast<float2*>(ml_s + 2 * tid) = ml;
        __syncthreads();  // (m, l) staged; the outputs may still be in flight
        for (int h = warp; h < G; h += kWarps) {
            float carry = cb == 0 ? -INFINITY : mcarry[h];
            for (int j0 = 0; j0 < nb; j0 += 32) {
                const int i = j0 + lane;
                const int k = i * G + h;
                const float mc = i < nb ? ml_s[2 * k] : -INFINITY;
                float v = mc;  // inclusive prefix maximum over the lanes
#pragma unroll
                for (int off = 1; off < 32; off <<= 1) {
                    const float o = __shfl_up_sync(0xffffffffu, v, off);
                    if (lane >= off) v = fmaxf(v, o);
                }
                // running max after chunk cb + i (chunk 0 starts the run)
                const float Mn = cb + j0 == 0 ? v : fmaxf(carry, v);
                float Mo = __shfl_up_sync(0xffffffffu, Mn, 1);
                if (lane == 0) Mo = carry;
                if (i < nb) {
                    const bool first = cb + i == 0;  // chunk 0: no factors
                    fl[k] = make_float4(first ? 0.f : bi_attn::exp2_ftz(Mo - Mn),
                                        first ? 0.f : bi_attn::exp2_ftz(mc - Mn), ml_s[2 * k + 1], 0.f);
                }
                carry = __shfl_sync(0xffffffffu, Mn, 31);
            }
            __syncwarp();
            if (lane == 0) mcarry[h] = carry;
        }
        bi::cp_async_wait_all();
        __syncthreads();  // factors and outputs staged
        for (int i0 = 0; i0 < nb; i0 += U) {
            float x[U][NH][ND];
            float4 f[U][NH];
#pragma unroll
            for (int u = 0; u < U; ++u)
#pragma unroll
                for (int j = 0; j < NH; ++j) {
                    const int k = (i0 + u) * G + h0 + j;
                    if (i0 + u < nb) {
                        f[u][j] = fl[k];
                        const float* xs = acc_s + k * kD + d0;
                        if constexpr (ND % 4 == 0) {
#pragma unroll
                            for (int e = 0; e < ND; e += 4) {
                                const float4 t = *reinterpret_cast<const float4*>(xs + e);
                                x[u][j][e] = t.x;
                                x[u][j][e + 1] = t.y;
                                x[u][j][e + 2] = t.z;
                                x[u][j][e + 3] = t.w;
                            }
                        } else if constexpr (ND == 2) {
                            const float2 t = *reinterpret_cast<const float2*>(xs);
                            x[u][j][0] = t.x;
                            x[u][j][1] = t.y;
                        } else {
                            x[u][j][0] = xs[0];
                        }
                    }
                }
#pragma unroll
            for (int u = 0; u < U; ++u)
#pragma unroll
                for (int j = 0; j < NH; ++j) {
                    if (i0 + u >= nb) continue;
                    if (cb + i0 + u == 0) {
                        Lr[j] = f[u][j].z;
#pragma unroll
                        for (int e = 0; e < ND; ++e) A[j][e] = x[u][j][e];
                    } else {
                        const float fo = f[u][j].x, fc = f[u][j].y;
                        Lr[j] = bi_attn::fold_value(Lr[j], fo, f[u][j].z, fc);
#pragma unroll
                        for (int e = 0; e < ND; ++e) A[j][e] = bi_attn::fold_value(A[j][e], fo, x[u][j][e], fc);
                    }
                }
        }
        __syncthreads();  // staging is reused by the next batch
    }
#pragma unroll
    for (int j = 0; j < NH; ++j) {
        __nv_bfloat16* o = a.out + (row0 + h0 + j) * kD + d0;
        const float il = bi_attn::inv_weight(Lr[j]);
        if constexpr (ND % 2 == 0) {
#pragma unroll
            for (int e = 0; e < ND; e += 2)
                *reinterpret_cast<__nv_bfloat162*>(o + e) = __halves2bfloat162(
                    __float2bfloat16_rn(bi_attn::normalise(A[j][e], il)),
                    __float2bfloat16_rn(bi_attn::normalise(A[j][e + 1], il)));
        } else {
            o[0] = __float2bfloat16_rn(bi_attn::normalise(A[j][0], il));
        }
    }
}

__global__ void __launch_bounds__(kThreads)
    attn_split_kernel(const __grid_constant__ CUtensorMap tmap_k,
                      const __grid_constant__ CUtensorMap tmap_v, const SplitArgs a) {
    bi::launch_dependents();
    bi::grid_dependency_wait();  // nothing global is touched before the previous kernel ends
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
    // several CTAs share the sequence and the last one to arrive folds it
    const bool shared_fold = !whole && a.counters != nullptr;
    const uint32_t ngroups = static_cast<uint32_t>((nch + a.chunks_per_cta - 1) / a.chunks_per_cta);
    uint32_t* const ctr = shared_fold ? a.counters + static_cast<int64_t>(s) * a.Hkv + g : nullptr;
    const int npg_total = (L + kPage - 1) / kPage;
    const int pg0 = c0 * ppc;
    const int npg_group = min(c1 * ppc, npg_total) - pg0;

    extern __shared__ uint8_t smem_raw[];
    uint8_t* smem = reinterpret_cast<uint8_t*>(
        (reinterpret_cast<uintptr_t>(smem_raw) + 1023) & ~static_cast<uintptr_t>(1023));
    float* fold_o = reinterpret_cast<float*>(smem + kStages * kStageBytes);  // [8 heads][128]
    float* fold_m = fold_o + kMaxGroup * kD;                                // [8]
    float* fold_l = fold_m + kMaxGroup;                                     // [8]
    int32_t* rows_s = reinterpret_cast<int32_t*>(fold_l + kMaxGroup);      // TMA row per page
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
        if (tid == 0) {
            bi::report_error(a.err, bi::kErrBadInput | bi::kWhereAttnSplit);
            if (shared_fold) {
                // count in, marking the sequence bad (its output stays
                // unwritten); the last arrival still returns the counter to 0
                const uint32_t now = bi::atomic_add_acq_rel_gpu(ctr, kArriveBad) + kArriveBad;
                if ((now & 0xffffu) == ngroups) atomicExch(ctr, 0u);
            }
        }
        return;
    }

    auto pages_in = [&](int c) { return min(ppc, npg_total - c * ppc); };
    auto stage_ptr = [&](int st) { return smem + st * kStageBytes; };

    // This warp's pages, in order: chunk c0 + warp, its pages 0, 1, ...; then
    // chunk c0 + warp + 4, ...  The loader runs kSPW pages ahead of the
    // compute loop through this warp's kSPW-stage ring; every lane tracks the
    // loader position, lane 0 issues the copies.
    int lc = c0 + warp, lp = 0, lj = 0;
    auto issue_next = [&]() {
        if (lc >= c1) return;
        if (lane == 0) {
            const int st = warp * kSPW + lj % kSPW;
            uint8_t* kd = stage_ptr(st);
            uint8_t* vd = kd + kMatBytes;
            const int row = rows_s[(lc - c0) * ppc + lp];
            bi::mbar_arrive_expect_tx(&bars[st], kStageBytes);
            bi::tma_load_3d(kd, &tmap_k, &bars[st], 0, row, 0);
            bi::tma_load_3d(vd, &tmap_v, &bars[st], 0, row, 0);
        }
        ++lj;
        if (++lp >= pages_in(lc)) {
            lc += kWarps;
            lp = 0;
        }
    };
#pragma unroll
    for (int i = 0; i < kSPW; ++i) issue_next();

    // column n of the mma tile = query head g*group + n (n < group)
    uint32_t qb0[8], qb1[8];
    {
        const int n = lane >> 2;
        bi_attn::load_q_frags(
            n < a.group ? a.q + (static_cast<int64_t>(s) * a.Hq + g * a.group + n) * kD : nullptr,
            lane, qb0, qb1);
    }
    const int h0 = 2 * (lane & 3);
    bool timed_out = false;
    int j = 0;       // this warp's page counter (matches the loader's)
    int j_fail = 0;  // first page whose wait timed out
    const int rounds = (c1 - c0 + kWarps - 1) / kWarps;

    for (int r = 0; r < rounds; ++r) {
        const int c = c0 + r * kWarps + warp;  // this warp's chunk in round r
        bi_attn::ColState st;
        bi_attn::colstate_init(st);
        if (c < c1) {
            const int np = pages_in(c);
            for (int p = 0; p < np; ++p, ++j) {
                const int stg = warp * kSPW + j % kSPW;
                if (timed_out) continue;
                if (!bi::mbar_wait(&bars[stg], (j / kSPW) & 1)) {
                    timed_out = true;
                    j_fail = j;
                    continue;
                }
                const int valid = min(kPage, L - (c * ppc + p) * kPage);
                if (valid < kPage) {
                    bi_attn::zero_v_tail(stage_ptr(stg) + kMatBytes, valid, lane);
                    __syncwarp();
                }
                const uint32_t kb = bi::smem_u32(stage_ptr(stg));
                bi_attn::attend_page(st, kb, kb + kMatBytes, qb0, qb1, valid, valid, a.scale_log2,
                                     lane);
                // hand the stage back to TMA for this warp's page kSPW ahead; the
                // zeroed V tail (generic-proxy writes) must be ordered before the
                // next copy (an async-proxy write) into the same stage
                if (valid < kPage) bi::fence_proxy_async_smem();
                __syncwarp();
                issue_next();
            }
            if (!whole) {
                // chunk partial -> workspace
#pragma unroll
                for (int e = 0; e < 2; ++e) {
                    const int h = h0 + e;
                    if (h >= a.group) continue;
                    const int64_t pidx =
                        (static_cast<int64_t>(s) * a.Hq + g * a.group + h) * a.max_chunks + c;
#pragma unroll
                    for (int mt = 0; mt < 8; ++mt) {
                        const int d = 16 * mt + (lane >> 2);
                        a.ws_acc[pidx * kD + d] = st.acc[mt][e];
                        a.ws_acc[pidx * kD + d + 8] = st.acc[mt][2 + e];
                    }
                    if (lane < 4) {
                        a.ws_ml[pidx * 2] = st.m[e];
                        a.ws_ml[pidx * 2 + 1] = st.l[e];
                    }
                }
            }
        }
        if (whole) {
            // fold this round's chunks into the running state, in chunk order
            for (int w = 0; w < kWarps; ++w) {
                if (warp == w && c < c1) {
#pragma unroll
                    for (int e = 0; e < 2; ++e) {
                        const int h = h0 + e;
                        if (c == 0) {
#pragma unroll
                            for (int mt = 0; mt < 8; ++mt) {
                                const int d = 16 * mt + (lane >> 2);
                                fold_o[h * kD + d] = st.acc[mt][e];
                                fold_o[h * kD + d + 8] = st.acc[mt][2 + e];
                            }
                        } else {
                            float Mn, fo, fc;
                            bi_attn::fold_scalars(fold_m[h], st.m[e], Mn, fo, fc);
#pragma unroll
                            for (int mt = 0; mt < 8; ++mt) {
                                const int d = 16 * mt + (lane >> 2);
                                float* o = fold_o + h * kD + d;
                                o[0] = bi_attn::fold_value(o[0], fo, st.acc[mt][e], fc);
                                o[8] = bi_attn::fold_value(o[8], fo, st.acc[mt][2 + e], fc);
                            }
                        }
                    }
                    __syncwarp();  // every lane has read M before lanes 0..3 replace it
                    if (lane < 4) {
#pragma unroll
                        for (int e = 0; e < 2; ++e) {
                            const int h = h0 + e;
                            if (c == 0) {
                                fold_m[h] = st.m[e];
                                fold_l[h] = st.l[e];
                            } else {
                                float Mn, fo, fc;
                                bi_attn::fold_scalars(fold_m[h], st.m[e], Mn, fo, fc);
                                fold_l[h] = bi_attn::fold_value(fold_l[h], fo, st.l[e], fc);
                                fold_m[h] = Mn;
                            }
                        }
                    }
                }
                __syncthreads();
            }
        }
    }

    if (timed_out && lane == 0) {
        bi::report_error(a.err, bi::kErrTimeout | bi::kWhereAttnSplit);
        // pages j_fail .. lj-1 were issued and never seen to land (at most kSPW):
        // give each one more bounded wait before this warp's stages are released
        for (int i = j_fail; i < lj; ++i)
            bi::mbar_wait_for(&bars[warp * kSPW + i % kSPW], (i / kSPW) & 1, bi::kDrainNs);
    }
    if (whole) {
        const int d = tid;
        for (int h = 0; h < a.group; ++h) {
            const int64_t row = static_cast<int64_t>(s) * a.Hq + g * a.group + h;
            a.out[row * kD + d] = __float2bfloat16_rn(
                bi_attn::normalise(fold_o[h * kD + d], bi_attn::inv_weight(fold_l[h])));
        }
        return;
    }
    if (!shared_fold) return;  // the merge kernel folds

    // ---- arrival: the last CTA of this (sequence, kv-head) folds it ------
    __shared__ int fold_here;
    __syncthreads();  // every warp's partial stores precede the arrival
    if (tid == 0) {
        // release: this CTA's partials are visible before its arrival counts;
        // acquire: the last arrival sees every other CTA's partials
        const uint32_t now = bi::atomic_add_acq_rel_gpu(ctr, kArrive) + kArrive;
        const bool last = (now & 0xffffu) == ngroups;
        if (last) {
            atomicExch(ctr, 0u);  // ready for the next call
            if (now >> 16) bi::report_error(a.err, bi::kErrBadInput | bi::kWhereAttnSplit);
        }
        fold_here = last && (now >> 16) == 0;
    }
    __syncthreads();
    if (!fold_here) return;
    switch (a.group) {
        case 1: fold_sequence<1>(a, s, g, nch, smem, fold_o, tid); break;
        case 2: fold_sequence<2>(a, s, g, nch, smem, fold_o, tid); break;
        case 3: fold_sequence<3>(a, s, g, nch, smem, fold_o, tid); break;
        case 4: fold_sequence<4>(a, s, g, nch, smem, fold_o, tid); break;
        case 5: fold_sequence<5>(a, s, g, nch, smem, fold_o, tid); break;
        case 6: fold_sequence<6>(a, s, g, nch, smem, fold_o, tid); break;
        case 7: fold_sequence<7>(a, s, g, nch, smem, fold_o, tid); break;
        default: fold_sequence<8>(a, s, g, nch, smem, fold_o, tid); break;
    }
}

// Small-batch form of the split kernel: the same chunks, pages and per-page
// operations, in the same order, with each chunk's page steps shared by a
// pair of warps.  The score warp computes each page's scores
// (bi_attn::page_scores) and hands them over through a shared-memory ring;
// the update warp runs the online-softmax update and the output products
// (softmax_step, pv_step) page after page.  A page's scores do not depend on
// the previous page, so they come off the chain of dependent steps that
// paces a single warp; the chunk's result is the same partial, bit for bit.
// CTA = (sequence, kv-head, group of chunks); pair k of its two pairs takes
// chunks c0 + k, c0 + k + 2, ...  Every chunk's partial goes to the workspace
// and the last CTA of the (sequence, kv-head) to arrive folds them, as in the
// split kernel.  Used when a launch's chunks fill less than a wave of the GPU
// (a few sequences), where one warp per chunk leaves most of it idle.
constexpr int kPairs = kWarps / 2;
constexpr int kPairStages = kStages / kPairs;  // K+V pages in flight per pair: 4
constexpr int kScoreSlots = 4;                 // pages' scores between the two warps
constexpr int kPairSmemBytes = kStages * kStageBytes + kFoldFloats * 4 + 4 * kMaxPagesPerCta +
                               kPairs * kScoreSlots * 32 * 16 + 8 * kPairs * 4 * kPairStages + 1024;

__global__ void __launch_bounds__(kThreads)
    attn_pair_kernel(const __grid_constant__ CUtensorMap tmap_k,
                     const __grid_constant__ CUtensorMap tmap_v, const SplitArgs a) {
    bi::launch_dependents();
    bi::grid_dependency_wait();  // nothing global is touched before the previous kernel ends
    const int cg = blockIdx.x;  // chunk group
    const int g = blockIdx.y;
    const int s = blockIdx.z;
    const int tid = threadIdx.x;
    const int warp = tid >> 5;
    const int lane = tid & 31;
    const int pair = warp >> 1;
    const bool scorer = (warp & 1) == 0;

    const int L = a.seq_lens[s];
    if (L < 1 || L > a.max_seq_len) {
        if (tid == 0 && cg == 0 && g == 0) bi::report_error(a.err, bi::kErrBadInput | bi::kWhereAttnSplit);
        return;
    }
    int ppc, nch;
    chunk_geometry(L, 0, ppc, nch);
    const int c0 = cg * a.chunks_per_cta;
    if (c0 >= nch) return;
    const int c1 = min(nch, c0 + a.chunks_per_cta);
    const uint32_t ngroups = static_cast<uint32_t>((nch + a.chunks_per_cta - 1) / a.chunks_per_cta);
    uint32_t* const ctr = a.counters + static_cast<int64_t>(s) * a.Hkv + g;
    const int npg_total = (L + kPage - 1) / kPage;
    const int pg0 = c0 * ppc;
    const int npg_group = min(c1 * ppc, npg_total) - pg0;

    extern __shared__ uint8_t smem_raw[];
    uint8_t* smem = reinterpret_cast<uint8_t*>(
        (reinterpret_cast<uintptr_t>(smem_raw) + 1023) & ~static_cast<uintptr_t>(1023));
    float* fold_o = reinterpret_cast<float*>(smem + kStages * kStageBytes);
    int32_t* rows_s = reinterpret_cast<int32_t*>(fold_o + kFoldFloats);  // TMA row per page
    float4* ring = reinterpret_cast<float4*>(rows_s + kMaxPagesPerCta);    // [pair][slot][lane]
    uint64_t* bars = reinterpret_cast<uint64_t*>(ring + kPairs * kScoreSlots * 32);
    uint64_t* full = bars + pair * 4 * kPairStages;   // [kPairStages] page landed
    uint64_t* empty = full + kPairStages;             // [kPairStages] page's products done
    uint64_t* sfull = empty + kPairStages;            // [kScoreSlots] scores written
    uint64_t* sempty = sfull + kScoreSlots;           // [kScoreSlots] scores read
    float4* my_ring = ring + pair * kScoreSlots * 32;
    __shared__ int bad_page;

    if (tid == 0) {
        bad_page = 0;
        for (int i = 0; i < kPairs * 4 * kPairStages; ++i) bi::mbar_init(&bars[i], 1);
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
        if (tid == 0) {
            bi::report_error(a.err, bi::kErrBadInput | bi::kWhereAttnSplit);
            const uint32_t now = bi::atomic_add_acq_rel_gpu(ctr, kArriveBad) + kArriveBad;
            if ((now & 0xffffu) == ngroups) atomicExch(ctr, 0u);
        }
        return;
    }

    auto pages_in = [&](int c) { return min(ppc, npg_total - c * ppc); };
    auto stage_ptr = [&](int j) { return smem + (pair * kPairStages + j % kPairStages) * kStageBytes; };
    bool timed_out = false;

    if (scorer) {
        // ---- loads (lane 0) and page scores ----
        int lc = c0 + pair, lp = 0, lj = 0;
        auto issue_next = [&]() {
            if (lc >= c1) return;
            if (lane == 0) {
                uint8_t* kd = stage_ptr(lj);
                const int row = rows_s[(lc - c0) * ppc + lp];
                uint64_t* bar = &full[lj % kPairStages];
                bi::mbar_arrive_expect_tx(bar, kStageBytes);
                bi::tma_load_3d(kd, &tmap_k, bar, 0, row, 0);
                bi::tma_load_3d(kd + kMatBytes, &tmap_v, bar, 0, row, 0);
            }
            ++lj;
            if (++lp >= pages_in(lc)) {
                lc += kPairs;
                lp = 0;
            }
        };
#pragma unroll
        for (int i = 0; i < kPairStages; ++i) issue_next();
        uint32_t qb0[8], qb1[8];
        {
            const int n = lane >> 2;
            bi_attn::load_q_frags(
                n < a.group ? a.q + (static_cast<int64_t>(s) * a.Hq + g * a.group + n) * kD : nullptr,
                lane, qb0, qb1);
        }
        int j = 0;
        int seen = 0;  // pages whose copies this warp saw land
        for (int c = c0 + pair; c < c1 && !timed_out; c += kPairs) {
            const int np = pages_in(c);
            for (int p = 0; p < np; ++p, ++j) {
                if (!__all_sync(0xffffffffu, bi::mbar_wait(&full[j % kPairStages], (j / kPairStages) & 1))) {
                    timed_out = true;
                    break;
                }
                seen = j + 1;
                float sc[4];
                bi_attn::page_scores(sc, bi::smem_u32(stage_ptr(j)), qb0, qb1, lane);
                const int slot = j % kScoreSlots;
                if (!__all_sync(0xffffffffu, bi::mbar_wait(&sempty[slot], ((j / kScoreSlots) & 1) ^ 1))) {
                    timed_out = true;
                    break;
                }
                my_ring[slot * 32 + lane] = make_float4(sc[0], sc[1], sc[2], sc[3]);
                __syncwarp();
                if (lane == 0) bi::mbar_arrive(&sfull[slot]);
                if (j >= 1) {
                    // page j - 1's stage is free once its products are done:
                    // the copy for page j - 1 + kPairStages goes into it (after
                    // this page's scores are handed over, so the score warp
                    // stays ahead of the update warp)
                    if (!__all_sync(0xffffffffu, bi::mbar_wait(&empty[(j - 1) % kPairStages],
                                                              ((j - 1) / kPairStages) & 1))) {
                        timed_out = true;
                        break;
                    }
                    issue_next();
                }
            }
        }
        if (timed_out && lane == 0) {
            bi::report_error(a.err, bi::kErrTimeout | bi::kWhereAttnSplit);
            // copies issued and never seen to land: one more bounded wait each
            for (int i = seen; i < lj; ++i)
                bi::mbar_wait_for(&full[i % kPairStages], (i / kPairStages) & 1, bi::kDrainNs);
        }
    } else {
        // ---- online-softmax update and output products, page after page ----
        const int h0 = 2 * (lane & 3);
        int j = 0;
        for (int c = c0 + pair; c < c1 && !timed_out; c += kPairs) {
            bi_attn::ColState st;
            bi_attn::colstate_init(st);
            const int np = pages_in(c);
            for (int p = 0; p < np; ++p, ++j) {
                const int slot = j % kScoreSlots;
                if (!__all_sync(0xffffffffu, bi::mbar_wait(&sfull[slot], (j / kScoreSlots) & 1))) {
                    timed_out = true;
                    break;
                }
                const float4 v4 = my_ring[slot * 32 + lane];
                const float sc[4] = {v4.x, v4.y, v4.z, v4.w};
                __syncwarp();
                if (lane == 0) bi::mbar_arrive(&sempty[slot]);
                // the page's V, landed (the score warp saw the same phase)
                if (!__all_sync(0xffffffffu, bi::mbar_wait(&full[j % kPairStages], (j / kPairStages) & 1))) {
                    timed_out = true;
                    break;
                }
                uint8_t* vd = stage_ptr(j) + kMatBytes;
                const int valid = min(kPage, L - (c * ppc + p) * kPage);
                if (valid < kPage) {
                    bi_attn::zero_v_tail(vd, valid, lane);
                    __syncwarp();
                }
                bi_attn::PFrags pf;
                bi_attn::softmax_step(st, sc, valid, valid, a.scale_log2, lane, pf);
                bi_attn::pv_step(st, pf, bi::smem_u32(vd), lane);
                // the zeroed V tail (generic-proxy writes) is ordered before the
                // next copy (an async-proxy write) into the same stage
                if (valid < kPage) bi::fence_proxy_async_smem();
                __syncwarp();
                if (lane == 0) bi::mbar_arrive(&empty[j % kPairStages]);
            }
            if (timed_out) break;
            // chunk partial -> workspace
#pragma unroll
            for (int e = 0; e < 2; ++e) {
                const int h = h0 + e;
                if (h >= a.group) continue;
                const int64_t pidx = (static_cast<int64_t>(s) * a.Hq + g * a.group + h) * a.max_chunks + c;
#pragma unroll
                for (int mt = 0; mt < 8; ++mt) {
                    const int d = 16 * mt + (lane >> 2);
                    a.ws_acc[pidx * kD + d] = st.acc[mt][e];
                    a.ws_acc[pidx * kD + d + 8] = st.acc[mt][2 + e];
                }
                if (lane < 4) {
                    a.ws_ml[pidx * 2] = st.m[e];
                    a.ws_ml[pidx * 2 + 1] = st.l[e];
                }
            }
        }
        if (timed_out && lane == 0) bi::report_error(a.err, bi::kErrTimeout | bi::kWhereAttnSplit);
    }

    // ---- arrival: the last CTA of this (sequence, kv-head) folds it ------
    __shared__ int fold_here;
    __syncthreads();  // every warp's partial stores precede the arrival
    if (tid == 0) {
        const uint32_t now = bi::atomic_add_acq_rel_gpu(ctr, kArrive) + kArrive;
        const bool last = (now & 0xffffu) == ngroups;
        if (last) {
            atomicExch(ctr, 0u);  // ready for the next call
            if (now >> 16) bi::report_error(a.err, bi::kErrBadInput | bi::kWhereAttnSplit);
        }
        fold_here = last && (now >> 16) == 0;
    }
    __syncthreads();
    if (!fold_here) return;
    switch (a.group) {
        case 1: fold_sequence<1>(a, s, g, nch, smem, fold_o, tid); break;
        case 2: fold_sequence<2>(a, s, g, nch, smem, fold_o, tid); break;
        case 3: fold_sequence<3>(a, s, g, nch, smem, fold_o, tid); break;
        case 4: fold_sequence<4>(a, s, g, nch, smem, fold_o, tid); break;
        case 5: fold_sequence<5>(a, s, g, nch, smem, fold_o, tid); break;
        case 6: fold_sequence<6>(a, s, g, nch, smem, fold_o, tid); break;
        case 7: fold_sequence<7>(a, s, g, nch, smem, fold_o, tid); break;
        default: fold_sequence<8>(a, s, g, nch, smem, fold_o, tid); break;
    }
}

// Fold the chunk partials of one (sequence, query head) in ascending chunk
// order:  M' = max(M, m_c);  l' = l 2^(M-M') + l_c 2^(m_c-M');
//         O' = O 2^(M-M') + O_c 2^(m_c-M');   out = bf16(O / l).
// kBatch: chunks whose partials are loaded before any of them is folded (a
// schedule choice; the fold stays strictly sequential in c).
template <int kBatch>
__global__ void __launch_bounds__(kD)
    attn_merge_kernel(const int32_t* __restrict__ seq_lens, const float* __restrict__ ws_acc,
                      const float* __restrict__ ws_ml, __nv_bfloat16* __restrict__ out, int Hq,
                      int max_chunks, int max_seq_len, int num_splits, int chunks_per_cta) {
    bi::launch_dependents();
    bi::grid_dependency_wait();  // nothing global is touched before the previous kernel ends
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
    for (int cb = 1; cb < nch; cb += kBatch) {
        float mc[kBatch], lc[kBatch], ac[kBatch];
#pragma unroll
        for (int i = 0; i < kBatch; ++i) {
            if (cb + i < nch) {
                const int64_t pc = base + cb + i;
                mc[i] = ws_ml[pc * 2];
                lc[i] = ws_ml[pc * 2 + 1];
                ac[i] = ws_acc[pc * kD + d];
            }
        }
#pragma unroll
        for (int i = 0; i < kBatch; ++i) {
            if (cb + i >= nch) break;
            float Mn, fo, fc;
            bi_attn::fold_scalars(M, mc[i], Mn, fo, fc);
            Ls = bi_attn::fold_value(Ls, fo, lc[i], fc);
            A = bi_attn::fold_value(A, fo, ac[i], fc);
            M = Mn;
        }
    }
    out[(static_cast<int64_t>(s) * Hq + hq) * kD + d] =
        __float2bfloat16_rn(bi_attn::normalise(A, bi_attn::inv_weight(Ls)));
}

int ceil_div(int64_t a, int64_t b) { return static_cast<int>((a + b - 1) / b); }

// (sequence, query head) rows up to which the merge batches 32 chunks' loads:
// at B = 1 that was 2-3 us faster than 8; at 64 sequences and more it was 2 %
// slower (more registers, fewer resident CTAs).
constexpr int64_t kMergeWideRows = 512;

// set once per device; any thread may race to set it, the attribute is idempotent
std::atomic<bool> g_attr_set[64] = {};

}  // namespace

extern "C" size_t bi_decode_attention_workspace_size(int32_t B, int32_t Hq, int32_t D,
                                                     int32_t max_seq_len) {
    if (B < 0 || Hq <= 0 || D <= 0 || max_seq_len < 1) return 0;
    const int64_t chunks = ceil_div(max_seq_len, kChunk);
    if (chunks < 2) return 0;
    return BI_DECODE_COUNTER_BYTES +
           static_cast<size_t>(B) * Hq * chunks * (static_cast<size_t>(D) + 2) * sizeof(float);
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

// Schedule (never the arithmetic): how many consecutive chunks one CTA walks.
// Measured on GB300 (cold L2, lengths uniform up to the bound, 3 CTAs per SM):
//   - 4 (one chunk per warp) is fastest from one sequence up to 2^16
//     (sequence, kv-head, chunk) units in the launch: B = 1 .. 128 at 8192
//     tokens (B = 128: 313 us against 318-336 us for 6 .. 32);
//   - from 2^16 units on, 32: the CTA holds whole sequences and folds them
//     without partials (B = 256: 599 against 605 us);
//   - when groups of 4 would fill between one and two waves of the resident
//     slots (about half the bound's CTAs have work when lengths spread up to
//     the bound), groups of 8 fit in one wave: B = 16, 57 against 62 us.
int chunks_per_cta(int64_t B, int64_t Hkv, int64_t max_chunks, int sms) {
    const int64_t slots = static_cast<int64_t>(sms) * 3;
    if (B * Hkv * max_chunks >= (int64_t{1} << 16)) return kMaxChunksPerCta;
    const int64_t ctas4 = B * Hkv * ((max_chunks + kWarps - 1) / kWarps);
    if (ctas4 > 2 * slots && ctas4 <= 4 * slots) return 2 * kWarps;
    return kWarps;
}

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
    const size_t need = max_chunks >= 2 ? BI_DECODE_COUNTER_BYTES +
                                              static_cast<size_t>(B) * Hq * max_chunks *
                                                  (static_cast<size_t>(D) + 2) * sizeof(float)
                                        : 0;
    if (need > 0) {
        if (!workspace || workspace_bytes < need) return BI_ERR_WORKSPACE_TOO_SMALL;
        if (!bi::aligned16(workspace)) return BI_ERR_MISALIGNED;
    }

    CUtensorMap tk, tv;
    const uint64_t rows = static_cast<uint64_t>(num_pages) * Hkv * kPage;
    if (bi::encode_page_map(&tk, k_cache, rows) != CUDA_SUCCESS ||
        bi::encode_page_map(&tv, v_cache, rows) != CUDA_SUCCESS)
        return BI_ERR_CUDA;

    int dev = 0;
    if (cudaGetDevice(&dev) != cudaSuccess || dev < 0 || dev >= 64) return BI_ERR_CUDA;
    if (!g_attr_set[dev]) {
        if (cudaFuncSetAttribute(attn_split_kernel, cudaFuncAttributeMaxDynamicSharedMemorySize,
                                 kSmemBytes) != cudaSuccess ||
            cudaFuncSetAttribute(attn_pair_kernel, cudaFuncAttributeMaxDynamicSharedMemorySize,
                                 kPairSmemBytes) != cudaSuccess)
            return BI_ERR_CUDA;
        g_attr_set[dev] = true;
    }

    SplitArgs args;
    args.q = static_cast<const __nv_bfloat16*>(q);
    args.block_table = block_table;
    args.seq_lens = seq_lens;
    args.out = static_cast<__nv_bfloat16*>(out);
    // workspace: [counters, BI_DECODE_COUNTER_BYTES][acc partials][(m, l) partials]
    uint8_t* ws = static_cast<uint8_t*>(workspace);
    const bool counted = need && static_cast<int64_t>(B) * Hkv <= kMaxCounters;
    args.counters = counted ? reinterpret_cast<uint32_t*>(ws) : nullptr;
    args.ws_acc = need ? reinterpret_cast<float*>(ws + BI_DECODE_COUNTER_BYTES) : nullptr;
    args.ws_ml = need ? args.ws_acc + static_cast<size_t>(B) * Hq * max_chunks * kD : nullptr;
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

    // A sequence whose chunks all fall to one CTA is folded there, the rest by
    // the last of its CTAs to arrive (or by the merge kernel when there are
    // more (sequence, kv-head) pairs than counters) -- every one of them
    // applies the same fold in the same chunk order.
    int cpc = 1;
    if (num_splits == 0) {
        cpc = chunks_per_cta(B, Hkv, max_chunks, bi::sm_count());
    } else {
        // comparison variant: up to one split per warp, within the page list
        const int ppc_max = ceil_div(ceil_div(max_seq_len, kPage), num_splits);
        cpc = std::max(1, std::min(std::min(num_splits, kWarps), kMaxPagesPerCta / ppc_max));
    }
    // a few sequences: their chunks, one per warp pair, need no more than two
    // CTAs per SM, so each chunk's page steps are shared by two warps
    // (attn_pair_kernel; same operations, same order, same bits).  Measured
    // cold against the split kernel: faster at 1-2 sequences of up to 8192
    // tokens, even or slower from 3 on.
    const bool paired = num_splits == 0 && counted &&
                        static_cast<int64_t>(B) * Hkv * ceil_div(max_chunks, kPairs) <=
                            2 * static_cast<int64_t>(bi::sm_count());
    if (paired) cpc = kPairs;
    args.chunks_per_cta = cpc;
    const int groups = ceil_div(max_chunks, cpc);
    if (paired) {
        return bi::launch_pdl(attn_pair_kernel, dim3(groups, Hkv, B), dim3(kThreads), kPairSmemBytes,
                              stream, tk, tv, args) == cudaSuccess
                   ? BI_OK
                   : BI_ERR_CUDA;
    }
    if (bi::launch_pdl(attn_split_kernel, dim3(groups, Hkv, B), dim3(kThreads), kSmemBytes, stream,
                       tk, tv, args) != cudaSuccess)
        return BI_ERR_CUDA;
    if (max_chunks > cpc && !counted) {
        // few rows: each thread's chain of loads is the bound, so load up to
        // 32 chunks at once; many rows: 8, for more resident CTAs
        const cudaError_t e =
            static_cast<int64_t>(B) * Hq <= kMergeWideRows
                ? bi::launch_pdl(attn_merge_kernel<32>, dim3(Hq, B), dim3(kD), 0, stream, seq_lens,
                                 static_cast<const float*>(args.ws_acc),
                                 static_cast<const float*>(args.ws_ml), args.out, Hq, max_chunks,
                                 max_seq_len, num_splits, cpc)
                : bi::launch_pdl(attn_merge_kernel<8>, dim3(Hq, B), dim3(kD), 0, stream, seq_lens,
                                 static_cast<const float*>(args.ws_acc),
                                 static_cast<const float*>(args.ws_ml), args.out, Hq, max_chunks,
                                 max_seq_len, num_splits, cpc);
        if (e != cudaSuccess) return BI_ERR_CUDA;
    }
    return BI_OK;
}

}  // namespace

extern "C" int32_t bi_decode_attention_launches(int32_t B, int32_t Hkv, int32_t max_seq_len) {
    if (B < 1 || Hkv < 1 || max_seq_len < 1) return 0;
    const int sms = bi::sm_count();
    if (sms <= 0) return 0;
    const int max_chunks = ceil_div(max_seq_len, kChunk);
    const bool counted = static_cast<int64_t>(B) * Hkv <= kMaxCounters;
    return max_chunks > chunks_per_cta(B, Hkv, max_chunks, sms) && !counted ? 2 : 1;
}

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
// chunk), each kD + 2 floats: 65536 x 130 x 4 bytes = 32.5 MiB per device,
// after the arrival counters (zero when the library is loaded, and every call
// leaves them zero).
constexpr int64_t kNoAllocPartials = 65536;
constexpr size_t kNoAllocBytes =
    BI_DECODE_COUNTER_BYTES + static_cast<size_t>(kNoAllocPartials) * (kD + 2) * sizeof(float);

static __device__ __align__(256) float g_noalloc_scratch[kNoAllocBytes / sizeof(float)];

std::mutex g_noalloc_mu;
void* g_noalloc_ptr[64] = {};

// Device address of g_noalloc_scratch on the current device.  The host-side
// name of the array is only a stand-in; the address a kernel can use comes
// from cudaGetSymbolAddress, resolved once per device with that device
// current and cached.  The first call on a device must not come while the
// stream is being captured (the lookup may load the module): refused then.
void* noalloc_scratch_address(int dev, cudaStream_t stream) {
    std::lock_guard<std::mutex> lk(g_noalloc_mu);
    if (!g_noalloc_ptr[dev]) {
        cudaStreamCaptureStatus cap = cudaStreamCaptureStatusNone;
        if (cudaStreamIsCapturing(stream, &cap) != cudaSuccess || cap != cudaStreamCaptureStatusNone)
            return nullptr;
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
    // a call whose sequences all fit in one chunk writes no partials at all
    const size_t need = bi_decode_attention_workspace_size(B, Hq, D, max_seq_len);
    if (need > 0) {
        const int64_t partials = static_cast<int64_t>(B) * Hq * ceil_div(max_seq_len, kChunk);
        if (need > kNoAllocBytes || partials > kNoAllocPartials) return BI_ERR_WORKSPACE_TOO_SMALL;
    }
    void* ws = nullptr;
    if (need > 0) {
        int dev = -1;
        if (cudaGetDevice(&dev) != cudaSuccess || dev < 0 || dev >= 64) return BI_ERR_CUDA;
        ws = noalloc_scratch_address(dev, stream);
        if (!ws) return BI_ERR_CUDA;
    }
    return bi_decode_attention(q, k_cache, v_cache, block_table, max_pages_per_seq, seq_lens, B,
                               Hq, Hkv, D, page_size, num_pages, max_seq_len, scale, out, ws,
                               need > 0 ? kNoAllocBytes : 0, stream);
}
