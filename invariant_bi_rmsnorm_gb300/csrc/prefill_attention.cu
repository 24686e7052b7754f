// bi_prefill_attention: attention for many query rows of the same sequence at
// once (prompt prefill, chunked prefill), with causal visibility, and per row
// exactly the arithmetic bi_decode_attention uses -- here on tcgen05 tensor
// cores with TMEM accumulators.
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
// The same products on other instructions.  Decode forms each page's scores
// with mma.sync (S^T = K . Q^T, eight 16-deep steps over the dims, ascending,
// into one fp32 accumulator) and each page's output update with mma.sync
// (O^T = O^T * alpha + V^T . P_hi^T, then + V^T . P_lo^T).  Here, per tile of
// 128 (query row, head) columns:
//     S = Q . K_block^T       8 tcgen05.mma (M 128, N 64, K 16) per block of
//                             four pages, dims ascending
//     O = O * alpha           by the softmax threads, in TMEM
//     O += P_hi . V_page      tcgen05.mma (M 128, K 16), P from shared memory
//     O += P_lo . V_page
// Each output element gets the same 16-deep steps in the same order, only
// with the operand roles swapped; on GB300 the tcgen05 and mma.sync steps
// give identical fp32 bits (measured on random and scaled operands; the tests
// compare every prefilled row with decode, bit for bit).  The softmax of a
// column is one thread's (softmax_page_col: decode's operations for that
// column, in decode's order).
//
// CTA = (sequence, kv-head, tile of 128 (query row, head) columns), two CTAs
// per SM (TMEM: 256 columns each).  Warp 0 loads the Q tile, then K in blocks
// of four pages and V page by page; warp 1 issues the output products and
// warp 6 the score products, each from one thread; warps 2-5 are the softmax
// threads, one column each (warp w reads TMEM lanes 32 (w % 4) ..).
// A page's weights are handed to the tensor core as soon as they are
// written; the softmax threads wait for the previous page's products only to
// rescale O (rare: the reference maximum moves only past a slack), to fold a
// finished chunk, or to finish the tile.  A page a row
// cannot see leaves that row's state exactly unchanged (alpha = 1, weights
// 0).  Rows longer than one chunk keep their running output in a caller
// workspace between chunks.
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

constexpr int kTiles = 1;        // query tiles per CTA
constexpr int kCols = 128;       // (row, head) columns per tile = TMEM lanes = MMA M
constexpr int kSoftWarps = 4;    // softmax warps per tile, one column per thread
constexpr int kScoreWarp = 2 + kTiles * kSoftWarps;  // after the softmax warps
constexpr int kThreads = (kScoreWarp + 1) * 32;
constexpr int kGroupPages = 4;   // pages per score block: S is one N = 64 product
constexpr int kKSlots = 2;       // K ring, in score blocks
constexpr int kKSlotBytes = 2 * kGroupPages * kHalfBytes;  // [dim half][64 tokens][128 B]: 16 KB
constexpr int kSBuf = 2;         // score blocks per tile in TMEM
constexpr int kQHalf = kCols * 128;          // one 64-dim half of a Q tile: 16 KB
constexpr int kQBytes = 2 * kQHalf;          // 32 KB
constexpr int kPBytes = kCols * kPage * 2;   // one bf16 [128][16] weight operand: 4 KB
// Weight operands by page.  A page is handed to the tensor core as soon as
// its weights are written: its products add onto O behind the previous
// page's in the tensor pipe, so the softmax threads wait for the previous
// page's products only when they must touch O themselves (a rescale, which
// the reference-maximum slack makes rare, a chunk fold, the tile's end).
// The buffers bound how far ahead of the tensor core they run.
constexpr int kPBufs = 3;
// V ring, in pages, one slot per weight buffer: page p's V slot and weight
// buffer are free again once page p's products are done (pempty), so one
// barrier per slot serves both rings and the output products need one commit.
constexpr int kVSlots = kPBufs;
constexpr int kOffK = kTiles * kQBytes;
constexpr int kOffV = kOffK + kKSlots * kKSlotBytes;
constexpr int kOffP = kOffV + kVSlots * kMatBytes;
constexpr int kOffBar = kOffP + kPBufs * 2 * kPBytes;
constexpr int kNumBars = 2 * kKSlots + kVSlots + 3 + 2 * kSBuf + 2 * kPBufs;
constexpr int kSmemBytes = kOffBar + kNumBars * 8 + 16 + 1024 /*align*/;
static_assert(kSmemBytes <= 227 * 1024, "shared memory");
// TMEM columns: O of tile t at t * 128; score block b of tile t at kColS +
// (t * kSBuf + b) * 64 (page j of the block in its columns 16 j ..).
constexpr uint32_t kTmemCols = 256;  // two CTAs per SM
constexpr uint32_t kColS = kTiles * kD;
constexpr uint32_t kSCols = kGroupPages * kPage;
static_assert(kColS + kTiles * kSBuf * kSCols <= kTmemCols, "TMEM columns");
// Instruction descriptors, kind::f16: D fp32 (bits 4-5 = 1), A and B bf16
// (bits 7-9, 10-12 = 1), A K-major (bit 15 = 0), B K-major (bit 16 = 0) for S
// and MN-major (bit 16 = 1) for V, N >> 3 at bits 17-22, M >> 4 at 24-28.
constexpr uint32_t kIdescS = (1u << 4) | (1u << 7) | (1u << 10) | ((kSCols >> 3) << 17) |
                             ((128u >> 4) << 24);
constexpr uint32_t kIdescPV = (1u << 4) | (1u << 7) | (1u << 10) | (1u << 16) |
                              ((128u >> 3) << 17) | ((128u >> 4) << 24);

struct PrefillArgs {
    const int32_t* block_table;
    const int32_t* seq_lens;
    const int32_t* q_indptr;
    __nv_bfloat16* out;
    float* ws;  // [T][Hq][D] running fold of rows with more than one chunk
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

// A bounded wait every lane of the warp takes, with one verdict for all of
// them: a warp never splits over a timeout before its next collective TMEM
// access.  (Polling from lane 0 alone, the other lanes parked in a shuffle,
// was measured slower: 231 against 190 us for an 8048-token prefill.)
__device__ __forceinline__ bool warp_wait(uint64_t* bar, uint32_t parity) {
    return __all_sync(0xffffffffu, bi::mbar_wait(bar, parity));
}

// K-major tile of 128-byte rows (8-row groups 1024 bytes apart).
__device__ __forceinline__ uint64_t kmajor_desc(uint32_t saddr) {
    return bi::sw128_desc_lbo_sbo(saddr, 16, 1024);
}

// A V page block [16 tokens][128 dims] as the MN-major B operand of the PV
// product: dims 64-127 one half block (kHalfBytes) on, tokens 8-15 1024 bytes on.
__device__ __forceinline__ uint64_t v_desc(uint32_t saddr) {
    return bi::sw128_desc_lbo_sbo(saddr, kHalfBytes, 1024);
}

// The weights of a page as the K-major A operand [128 columns][16 tokens],
// no swizzle: core matrices of 8 columns x 8 tokens (128 bytes), tokens 8-15
// 128 bytes on, the next 8 columns 256 bytes on.
__device__ __forceinline__ uint64_t p_desc(uint32_t saddr) {
    return bi::plain_desc_lbo_sbo(saddr, 128, 256);
}

__global__ void __launch_bounds__(kThreads, 2)
    prefill_attn_kernel(const __grid_constant__ CUtensorMap tmap_q,
                        const __grid_constant__ CUtensorMap tmap_k,
                        const __grid_constant__ CUtensorMap tmap_v, const PrefillArgs a) {
    const int tid = threadIdx.x;
    const int warp = tid >> 5;
    const int lane = tid & 31;
    bi::launch_dependents();
    bi::grid_dependency_wait();  // nothing global is touched before the previous kernel ends

    // ---- geometry: grid = (sequence, kv-head, tile), the tile index slowest
    // and reversed, so the last (longest) tiles of every sequence start first ----
    const int G = a.group;
    const int rpt = a.rows_per_tile;
    const int pair = gridDim.z - 1 - blockIdx.z;
    const int g = blockIdx.y;
    const int s = blockIdx.x;
    const int q0 = a.q_indptr[s];
    const int nq = a.q_indptr[s + 1] - q0;
    const int Ls = a.seq_lens[s];
    const bool bad = q0 < 0 || nq < 0 || q0 + nq > a.T || nq > a.max_q_len ||
                     (nq > 0 && (Ls < nq || Ls > a.max_seq_len));
    if (bad) {
        if (tid == 0 && pair == 0 && g == 0)
            bi::report_error(a.err, bi::kErrBadInput | bi::kWhereAttnSplit);
        return;
    }
    // query row r (0-based among the sequence's nq rows) sees the first
    // Lbase + r tokens
    const int Lbase = Ls - nq + 1;
    const int r0 = pair * kTiles * rpt;
    if (r0 >= nq) return;  // no rows here: leave before any set-up
    int nrt[kTiles], npg_t[kTiles];
    int ntiles = 0, npg = 0, Lmax = 0;
#pragma unroll
    for (int t = 0; t < kTiles; ++t) {
        nrt[t] = max(0, min(rpt, nq - (r0 + t * rpt)));
        npg_t[t] = 0;
        if (nrt[t] > 0) {
            const int Lt = Lbase + r0 + t * rpt + nrt[t] - 1;
            npg_t[t] = (Lt + kPage - 1) / kPage;
            ntiles = t + 1;
            npg = max(npg, npg_t[t]);
            Lmax = max(Lmax, Lt);
        }
    }
    const int ngroups = (npg + kGroupPages - 1) / kGroupPages;

    extern __shared__ uint8_t smem_raw[];
    uint8_t* smem = reinterpret_cast<uint8_t*>(
        (reinterpret_cast<uintptr_t>(smem_raw) + 1023) & ~static_cast<uintptr_t>(1023));
    uint64_t* kfull = reinterpret_cast<uint64_t*>(smem + kOffBar);  // [kKSlots] K block landed
    uint64_t* kempty = kfull + kKSlots;                              // [kKSlots] K slot free
    uint64_t* vfull = kempty + kKSlots;                              // [kVSlots] V page landed
    uint64_t* qfull = vfull + kVSlots;                               // Q tiles landed
    uint64_t* drain = qfull + 1;                                     // output MMAs after a timeout
    uint64_t* drain_s = drain + 1;                                   // score MMAs after a timeout
    uint64_t* sfull = drain_s + 1;               // [kTiles][kSBuf] score block ready
    uint64_t* sfree = sfull + kTiles * kSBuf;    // [kTiles][kSBuf] score block read
    uint64_t* pfull = sfree + kTiles * kSBuf;    // [kPBufs] a page's weights written (O ready)
    uint64_t* pempty = pfull + kPBufs;           // [kPBufs] that page's products done
    uint32_t* tmem_slot = reinterpret_cast<uint32_t*>(pempty + kPBufs);
    if (tid == 0) {
        for (int i = 0; i < kKSlots; ++i) {
            bi::mbar_init(&kfull[i], 1);
            bi::mbar_init(&kempty[i], 1);
        }
        for (int i = 0; i < kVSlots; ++i) {
            bi::mbar_init(&vfull[i], 1);
        }
        bi::mbar_init(qfull, 1);
        bi::mbar_init(drain, 1);
        bi::mbar_init(drain_s, 1);
        for (int i = 0; i < kTiles * kSBuf; ++i) {
            bi::mbar_init(&sfull[i], 1);
            bi::mbar_init(&sfree[i], kSoftWarps);
        }
        for (int i = 0; i < kPBufs; ++i) {
            bi::mbar_init(&pfull[i], kSoftWarps);
            bi::mbar_init(&pempty[i], 1);
        }
        bi::fence_mbar_init();
        bi::tma_prefetch_desc(&tmap_q);
        bi::tma_prefetch_desc(&tmap_k);
        bi::tma_prefetch_desc(&tmap_v);
        // the Q tile does not depend on the page table: its loads go out now
        const uint32_t qbytes = static_cast<uint32_t>(ntiles * 2 * 64 * G * rpt * 2);
        bi::mbar_arrive_expect_tx(qfull, qbytes);
        for (int t = 0; t < ntiles; ++t)
            for (int h2 = 0; h2 < 2; ++h2)
                bi::tma_load_3d(smem + t * kQBytes + h2 * kQHalf, &tmap_q, qfull, 64 * h2, g * G,
                                q0 + r0 + t * rpt);
    }
    if (warp == 1) {
        bi::tmem_alloc(tmem_slot, kTmemCols);
        bi::tmem_relinquish();
    }
    const int32_t* bt = a.block_table + static_cast<int64_t>(s) * a.max_pages_per_seq;
    bi::tc_fence_before();
    __syncthreads();
    bi::tc_fence_after();
    const uint32_t tm = *tmem_slot;
    // The page table is not checked before the loads go out: a page outside
    // the cache maps past the tensor's end, where a TMA load reads zeros, and
    // the softmax threads judge the pages before they write anything.
    auto page_row = [&](int pg) -> int32_t {
        if (pg < 0 || pg >= a.num_pages) return a.num_pages * a.Hkv * kPage;
        return (pg * a.Hkv + g) * kPage;
    };

    if (warp == 0) {
        // ---------------- producers: lane 0 the Q tiles and the K blocks,
        // lane 16 the V pages (independent loops, each on its own ring) ------
        if (lane == 0) {
            int b = 0;
            for (; b < ngroups; ++b) {
                const int slot = b % kKSlots;
                if (!bi::mbar_wait(&kempty[slot], ((b / kKSlots) & 1) ^ 1)) {
                    bi::report_error(a.err, bi::kErrTimeout | bi::kWhereAttnSplit);
                    break;
                }
                const int np = min(kGroupPages, npg - b * kGroupPages);
                uint8_t* kd = smem + kOffK + slot * kKSlotBytes;
                bi::mbar_arrive_expect_tx(&kfull[slot], static_cast<uint32_t>(np * 2 * kHalfBytes));
                for (int j = 0; j < np; ++j) {
                    const int32_t row = page_row(bt[b * kGroupPages + j]);
                    bi::tma_load_2d(kd + j * kHalfBytes, &tmap_k, &kfull[slot], 0, row);
                    bi::tma_load_2d(kd + kGroupPages * kHalfBytes + j * kHalfBytes, &tmap_k,
                                    &kfull[slot], 64, row);
                }
            }
            // the CTA's shared memory outlives no copy: wait (bounded) for the
            // last copies issued into each slot
            for (int i = max(0, b - kKSlots); i < b; ++i)
                bi::mbar_wait_for(&kfull[i % kKSlots], (i / kKSlots) & 1, bi::kDrainNs);
            bi::mbar_wait_for(qfull, 0, bi::kDrainNs);
        } else if (lane == 16) {
            int p = 0;
            for (; p < npg; ++p) {
                const int slot = p % kVSlots;
                // the slot's previous page (p - kVSlots) has had its products
                if (!bi::mbar_wait(&pempty[slot], ((p / kVSlots) & 1) ^ 1)) {
                    bi::report_error(a.err, bi::kErrTimeout | bi::kWhereAttnSplit);
                    break;
                }
                const int32_t row = page_row(bt[p]);
                bi::mbar_arrive_expect_tx(&vfull[slot], kMatBytes);
                bi::tma_load_3d(smem + kOffV + slot * kMatBytes, &tmap_v, &vfull[slot], 0, row, 0);
            }
            for (int i = max(0, p - kVSlots); i < p; ++i)
                bi::mbar_wait_for(&vfull[i % kVSlots], (i / kVSlots) & 1, bi::kDrainNs);
        }
    } else if (warp == 1) {
        // ---------------- output products (lane 0 issues; the warp waits
        // together).  The descriptors are built before the waits: the start
        // address field is addr >> 4, so a shared-memory offset is added as
        // offset >> 4, and no address arithmetic sits between a hand-over and
        // its products.
        const uint64_t vd0 = v_desc(bi::smem_u32(smem + kOffV));
        const uint64_t pd0 = p_desc(bi::smem_u32(smem + kOffP));
        bool ok = true;
        bool issued = false;
        for (int p = 0; ok && p < npg; ++p) {
            const int vslot = p % kVSlots;
            const uint64_t vdp = vd0 + static_cast<uint64_t>((vslot * kMatBytes) >> 4);
            const uint64_t pdp = pd0 + static_cast<uint64_t>(((p % kPBufs) * 2 * kPBytes) >> 4);
            if (!warp_wait(&vfull[vslot], (p / kVSlots) & 1)) {
                ok = false;
                break;
            }
            const int vmax = Lmax - p * kPage;
            if (vmax < kPage) {
                // tokens past the longest row: zero their V rows (whatever
                // the cache holds there must not meet a zero weight as NaN)
                bi_attn::zero_v_tail(smem + kOffV + vslot * kMatBytes, vmax, lane);
                bi::fence_proxy_async_smem();
                __syncwarp();
            }
            const int pb = p % kPBufs;
            if (!warp_wait(&pfull[pb], (p / kPBufs) & 1)) {
                ok = false;
                break;
            }
            bi::tc_fence_after();
            if (lane == 0) {
                // O += P_hi . V, then O += P_lo . V (N = 128: all of O's dims)
                bi::tc_mma_f16(tm, pdp, vdp, kIdescPV, 1u);
                bi::tc_mma_f16(tm, pdp + static_cast<uint64_t>(kPBytes >> 4), vdp, kIdescPV, 1u);
                bi::tc_commit(&pempty[pb]);  // the page's products (and all before) done
            }
            issued = true;
            __syncwarp();
        }
        if (!ok) {
            if (lane == 0) {
                bi::report_error(a.err, bi::kErrTimeout | bi::kWhereAttnSplit);
                if (issued) {
                    // products still in flight read shared memory and write
                    // TMEM: a bounded wait for them before both are released
                    bi::tc_commit(drain);
                    bi::mbar_wait_for(drain, 0, bi::kDrainNs);
                }
            }
            __syncwarp();
        }
    } else if (warp == kScoreWarp) {
        // ---------------- score products (lane 0 issues), on their own
        // thread so that no output product queues behind them: block b of
        // four pages into TMEM buffer b % kSBuf once its K block has landed
        // and the softmax threads have read the buffer's previous block.
        static_assert(kTiles == 1, "one tile per CTA");
        const uint64_t qd = kmajor_desc(bi::smem_u32(smem));
        const uint64_t kd0 = kmajor_desc(bi::smem_u32(smem + kOffK));
        bool ok = warp_wait(qfull, 0);
        bool issued = false;
        for (int b = 0; ok && b < ngroups; ++b) {
            const int slot = b % kKSlots;
            const uint64_t kd = kd0 + static_cast<uint64_t>((slot * kKSlotBytes) >> 4);
            const uint32_t d = tm + kColS + static_cast<uint32_t>(b % kSBuf) * kSCols;
            ok = warp_wait(&kfull[slot], (b / kKSlots) & 1) &&
                 warp_wait(&sfree[b % kSBuf], ((b / kSBuf) & 1) ^ 1);
            if (!ok) break;
            bi::tc_fence_after();
            if (lane == 0) {
                // k-step ks covers dims 16 ks .. 16 ks + 15: 32 bytes into
                // the rows of 64-dim half ks / 4 of Q and of the K block
#pragma unroll
                for (int ks = 0; ks < kD / 16; ++ks)
                    bi::tc_mma_f16(d, qd + static_cast<uint64_t>(((ks >> 2) * kQHalf + 32 * (ks & 3)) >> 4),
                                   kd + static_cast<uint64_t>(((ks >> 2) * kGroupPages * kHalfBytes + 32 * (ks & 3)) >> 4),
                                   kIdescS, ks > 0 ? 1u : 0u);
                bi::tc_commit(&sfull[b % kSBuf]);
                bi::tc_commit(&kempty[slot]);  // the K block is free once these finish
            }
            issued = true;
            __syncwarp();
        }
        if (!ok) {
            if (lane == 0) {
                bi::report_error(a.err, bi::kErrTimeout | bi::kWhereAttnSplit);
                if (issued) {
                    bi::tc_commit(drain_s);
                    bi::mbar_wait_for(drain_s, 0, bi::kDrainNs);
                }
            }
            __syncwarp();
        }
    } else if (warp >= 2) {
        // ---------------- softmax: thread = one (row, head) column -----------
        const int t = (warp - 2) / kSoftWarps;
        if (t < ntiles) {
            const int quarter = warp & 3;
            const int c = quarter * 32 + lane;
            const uint32_t lrow = tm + (static_cast<uint32_t>(quarter * 32) << 16);
            const uint32_t col_o = lrow + static_cast<uint32_t>(t * kD);
            const int rr = c / G;
            const bool live = c < rpt * G && rr < nrt[t];
            const int Lc = live ? Lbase + r0 + t * rpt + rr : 0;
            const int64_t row = static_cast<int64_t>(q0 + r0 + t * rpt + rr) * a.Hq + g * G + c % G;
            // This column's running output in the workspace.  The tile owns
            // the workspace span of its rows' tokens ([T][Hq][D] floats in
            // size); the kv-head's share of it is laid out dims-by-4 major,
            // column minor, so the 32 columns of a warp move 512 contiguous
            // bytes per access.
            const int ncols = nrt[t] * G;
            const int wstride = 4 * ncols;
            float* wcol = a.ws == nullptr ? nullptr
                                          : a.ws + static_cast<int64_t>(q0 + r0 + t * rpt) * a.Hq * kD +
                                                static_cast<int64_t>(g) * ncols * kD + 4 * c;
            // this column's weights in the page's P operands (high parts,
            // remainders), buffer p % kPBufs
            uint8_t* p_col = smem + kOffP + (c >> 3) * 256 + (c & 7) * 16;
            float m = -INFINITY, l = 0.f;    // online softmax of the current chunk
            float Mr = -INFINITY, Lr = 0.f;  // fold over the finished chunks
            bool ok = true;
            // A page outside the cache: the tile is computed on the zeros its
            // loads read there and is not written.  The page numbers are read
            // now and judged at the first write, so the loads' latency hides
            // behind the tile's pages.
            const int pg0 = lane < npg ? bt[lane] : 0;
            int bad_more = 0;
            for (int i = lane + 32; i < npg; i += 32) bad_more |= bt[i] < 0 || bt[i] >= a.num_pages;
            int judged = 0;
            bool writes = true;
            auto judge = [&]() {
                if (judged) return;
                judged = 1;
                writes = !__any_sync(0xffffffffu, pg0 < 0 || pg0 >= a.num_pages || bad_more);
                if (!writes && warp == 2 && lane == 0)
                    bi::report_error(a.err, bi::kErrBadInput | bi::kWhereAttnSplit);
            };

            // Fold chunk k (state mk, lk and its O in TMEM) into the column's
            // running state, as decode folds a chunk partial, and write the
            // output if k is the column's last chunk.  Rows of one chunk keep
            // everything in TMEM; the running O of longer rows lives in the
            // workspace between chunks.  Columns that do not see chunk k are
            // left unchanged.
            auto fold_chunk = [&](int k, float mk, float lk) {
                judge();
                const bool sees = Lc > k * kChunk;
                const bool last = sees && Lc <= (k + 1) * kChunk;
                float fo = 1.f, fc = 1.f;
                if (sees) {
                    if (k == 0) {
                        Mr = mk;
                        Lr = lk;
                    } else {
                        float Mn;
                        bi_attn::fold_scalars(Mr, mk, Mn, fo, fc);
                        Lr = bi_attn::fold_value(Lr, fo, lk, fc);
                        Mr = Mn;
                    }
                }
                const float il = bi_attn::inv_weight(Lr);
#pragma unroll 1
                for (int q4 = 0; q4 < kD / 32; ++q4) {
                    uint32_t o[32];
                    __syncwarp();
                    bi::tmem_ld_32x32b_x32(col_o + 32 * q4, o);
                    bi::tmem_ld_wait();
                    if (!sees || !writes) continue;
                    float A[32];
#pragma unroll
                    for (int i = 0; i < 32; i += 4) {
                        if (k == 0) {
                            A[i] = __uint_as_float(o[i]);
                            A[i + 1] = __uint_as_float(o[i + 1]);
                            A[i + 2] = __uint_as_float(o[i + 2]);
                            A[i + 3] = __uint_as_float(o[i + 3]);
                        } else {
                            const float4 w = *reinterpret_cast<const float4*>(wcol + (8 * q4 + i / 4) * wstride);
                            A[i] = bi_attn::fold_value(w.x, fo, __uint_as_float(o[i]), fc);
                            A[i + 1] = bi_attn::fold_value(w.y, fo, __uint_as_float(o[i + 1]), fc);
                            A[i + 2] = bi_attn::fold_value(w.z, fo, __uint_as_float(o[i + 2]), fc);
                            A[i + 3] = bi_attn::fold_value(w.w, fo, __uint_as_float(o[i + 3]), fc);
                        }
                    }
                    if (last) {
                        __nv_bfloat16* orow = a.out + row * kD + 32 * q4;
#pragma unroll
                        for (int i = 0; i < 32; i += 8) {
                            uint4 v;
                            v.x = bi::pack_bf16x2(bi_attn::normalise(A[i], il), bi_attn::normalise(A[i + 1], il));
                            v.y = bi::pack_bf16x2(bi_attn::normalise(A[i + 2], il), bi_attn::normalise(A[i + 3], il));
                            v.z = bi::pack_bf16x2(bi_attn::normalise(A[i + 4], il), bi_attn::normalise(A[i + 5], il));
                            v.w = bi::pack_bf16x2(bi_attn::normalise(A[i + 6], il), bi_attn::normalise(A[i + 7], il));
                            *reinterpret_cast<uint4*>(orow + i) = v;
                        }
                    } else {
#pragma unroll
                        for (int i = 0; i < 32; i += 4)
                            *reinterpret_cast<float4*>(wcol + (8 * q4 + i / 4) * wstride) =
                                make_float4(A[i], A[i + 1], A[i + 2], A[i + 3]);
                    }
                }
                __syncwarp();
            };

            // One page p whose 16 raw scores are in sv.  The weights go to
            // buffer p % kPBufs once the page that used it last has had its
            // products; the page is handed over at once unless O must be
            // touched first: rescaled (some alpha of the warp not 1), or
            // folded and zeroed at a chunk start.  Either waits for the
            // previous page's products, which by then are the last on O.
            auto wait_products = [&](int q) {  // page q's products (and all before) done
                return warp_wait(&pempty[q % kPBufs], (q / kPBufs) & 1);
            };
            auto hand_over = [&](int pb) {
                bi::tmem_st_wait();
                bi::tc_fence_before();
                __syncwarp();
                if (lane == 0) bi::mbar_arrive(&pfull[pb]);
            };
            auto page = [&](int p, const float (&sv)[16]) -> bool {
                const bool first = (p % kPagesPerChunk) == 0;
                const float m_prev = m, l_prev = l;
                if (first) {
                    m = -INFINITY;
                    l = 0.f;
                }
                uint32_t hi[8], lo[8];
                const int valid = max(0, min(kPage, Lc - p * kPage));
                const float al = bi_attn::softmax_page_col(m, l, sv, valid, a.scale_log2, hi, lo);
                const int pb = p % kPBufs;
                if (!warp_wait(&pempty[pb], ((p / kPBufs) & 1) ^ 1)) return false;  // buffer free
                // weights of tokens 0-7 and 8-15: two core matrices of the operand
                uint8_t* ph = p_col + pb * 2 * kPBytes;
                *reinterpret_cast<uint4*>(ph) = make_uint4(hi[0], hi[1], hi[2], hi[3]);
                *reinterpret_cast<uint4*>(ph + 128) = make_uint4(hi[4], hi[5], hi[6], hi[7]);
                *reinterpret_cast<uint4*>(ph + kPBytes) = make_uint4(lo[0], lo[1], lo[2], lo[3]);
                *reinterpret_cast<uint4*>(ph + kPBytes + 128) = make_uint4(lo[4], lo[5], lo[6], lo[7]);
                bi::fence_proxy_async_smem();  // the weights are read by the tensor core
                if (first) {
                    if (p > 0) {
                        // the chunk that ended: its O is complete once the
                        // previous page's products are done
                        if (!wait_products(p - 1)) return false;
                        bi::tc_fence_after();
                        fold_chunk(p / kPagesPerChunk - 1, m_prev, l_prev);
                    }
                    uint32_t z[32];
#pragma unroll
                    for (int i = 0; i < 32; ++i) z[i] = 0u;
#pragma unroll
                    for (int q4 = 0; q4 < kD / 32; ++q4) bi::tmem_st_32x32b_x32(col_o + 32 * q4, z);
                } else if (__any_sync(0xffffffffu, al != 1.f)) {
                    // alpha == 1 leaves O's bits unchanged, so only a moved
                    // reference maximum needs O rescaled (after the previous
                    // page's products)
                    if (!wait_products(p - 1)) return false;
                    bi::tc_fence_after();
#pragma unroll 1
                    for (int q4 = 0; q4 < kD / 32; ++q4) {
                        uint32_t o0[32];
                        const uint32_t cb = col_o + static_cast<uint32_t>(32 * q4);
                        bi::tmem_ld_32x32b_x32(cb, o0);
                        bi::tmem_ld_wait();
#pragma unroll
                        for (int i = 0; i < 32; ++i) o0[i] = __float_as_uint(__fmul_rn(__uint_as_float(o0[i]), al));
                        bi::tmem_st_32x32b_x32(cb, o0);
                    }
                }
                hand_over(pb);
                return true;
            };

            const int np = npg_t[t];
            const int nb = (np + kGroupPages - 1) / kGroupPages;
            for (int b = 0; ok && b < nb; ++b) {
                const int sb = b % kSBuf;
                if (!warp_wait(&sfull[t * kSBuf + sb], (b / kSBuf) & 1)) {
                    ok = false;
                    break;
                }
                bi::tc_fence_after();
                const int npb = min(kGroupPages, np - b * kGroupPages);
                const uint32_t scol = lrow + kColS + static_cast<uint32_t>(t * kSBuf + sb) * kSCols;
                for (int h = 0; ok && h * 2 < npb; ++h) {
                    uint32_t sr[32];
                    bi::tmem_ld_32x32b_x32(scol + 32 * h, sr);
                    bi::tmem_ld_wait();
                    if (h == 1 || npb <= 2) {  // the block's last read
                        bi::tc_fence_before();
                        __syncwarp();
                        if (lane == 0) bi::mbar_arrive(&sfree[t * kSBuf + sb]);
                    }
                    for (int jj = 0; ok && jj < 2 && 2 * h + jj < npb; ++jj) {
                        float sv[16];
#pragma unroll
                        for (int i = 0; i < 16; ++i) sv[i] = __uint_as_float(sr[16 * jj + i]);
                        ok = page(b * kGroupPages + 2 * h + jj, sv);
                    }
                }
            }
            const bool last_ok = ok && wait_products(np - 1);
            if (last_ok) {
                bi::tc_fence_after();
                fold_chunk((np - 1) / kPagesPerChunk, m, l);
            } else if (lane == 0) {
                bi::report_error(a.err, bi::kErrTimeout | bi::kWhereAttnSplit);
            }
        }
    }

    bi::tc_fence_before();
    __syncthreads();
    if (warp == 1) {
        bi::tc_fence_after();
        bi::tmem_dealloc(tm, kTmemCols);
    }
}

// ---------------------------------------------------------------------------
// Self-test of the premise above: one page's products on both instruction
// paths, with this file's descriptors and MMA forms and decode's mma.sync
// steps (attn_common.cuh), fp32 results returned for a bit-for-bit comparison.
//   S = Q . K^T        tcgen05 (as prefill_attn_kernel)  vs  page_scores
//   O = O0 + P . V     tcgen05, P from shared memory      vs  one mma.sync per
//                                                             16-dim tile
// Q [128 columns][128], K and V one page [16][128], P [128 columns][16] (bf16),
// O0 [128][128] fp32.  One CTA of 128 threads.
constexpr int kStSmemQ = 0;              // 32 KB, as a Q tile
constexpr int kStSmemK = kQBytes;        // 4 KB, as a K page block
constexpr int kStSmemV = kStSmemK + kMatBytes;
constexpr int kStSmemP = kStSmemV + kMatBytes;
constexpr int kStSmemBar = kStSmemP + kPBytes;
constexpr int kStSmemBytes = kStSmemBar + 64 + 1024;

struct SelftestArgs {
    const __nv_bfloat16 *q, *k, *v, *p;
    const float* o0;
    float *s_tc, *s_mma, *o_tc, *o_mma;
    uint32_t* err;
};

__global__ void __launch_bounds__(128, 1) tc_selftest_kernel(const SelftestArgs a) {
    extern __shared__ uint8_t smem_raw[];
    uint8_t* smem = reinterpret_cast<uint8_t*>(
        (reinterpret_cast<uintptr_t>(smem_raw) + 1023) & ~static_cast<uintptr_t>(1023));
    uint8_t* qs = smem + kStSmemQ;
    uint8_t* ks = smem + kStSmemK;
    uint8_t* vs = smem + kStSmemV;
    uint8_t* ps = smem + kStSmemP;
    uint64_t* bar = reinterpret_cast<uint64_t*>(smem + kStSmemBar);
    uint32_t* tmem_slot = reinterpret_cast<uint32_t*>(bar + 1);
    const int tid = threadIdx.x, warp = tid >> 5, lane = tid & 31;
    // operands into the kernel's shared-memory layouts (128-byte swizzle for
    // Q, K, V; core matrices for P)
    for (int i = tid; i < kCols * kD; i += 128) {
        const int c = i / kD, d = i % kD;
        *reinterpret_cast<__nv_bfloat16*>(qs + (d / 64) * kQHalf + c * 128 +
                                          ((((d % 64) / 8) ^ (c % 8)) * 16) + (d % 8) * 2) = a.q[i];
    }
    for (int i = tid; i < kPage * kD; i += 128) {
        const int t = i / kD, d = i % kD;
        const uint32_t off = bi_attn::swz(t, d / 8) + (d % 8) * 2;
        *reinterpret_cast<__nv_bfloat16*>(ks + off) = a.k[i];
        *reinterpret_cast<__nv_bfloat16*>(vs + off) = a.v[i];
    }
    for (int i = tid; i < kCols * kPage; i += 128) {
        const int c = i / kPage, t = i % kPage;
        *reinterpret_cast<__nv_bfloat16*>(ps + (c / 8) * 256 + (t / 8) * 128 + (c % 8) * 16 +
                                          (t % 8) * 2) = a.p[i];
    }
    if (tid == 0) {
        bi::mbar_init(bar, 1);
        bi::fence_mbar_init();
    }
    if (warp == 0) {
        bi::tmem_alloc(tmem_slot, 256);
        bi::tmem_relinquish();
    }
    bi::fence_proxy_async_smem();
    bi::tc_fence_before();
    __syncthreads();
    bi::tc_fence_after();
    const uint32_t tm = *tmem_slot;

    // mma.sync: S^T and O^T for 8 columns per group, 4 groups per warp
    for (int j = warp * 4; j < warp * 4 + 4; ++j) {
        uint32_t qb0[8], qb1[8];
        bi_attn::load_q_frags(a.q + (8 * j + lane / 4) * kD, lane, qb0, qb1);
        float sc[4];
        bi_attn::page_scores(sc, bi::smem_u32(ks), qb0, qb1, lane);
        for (int e = 0; e < 2; ++e) {
            const int col = 8 * j + 2 * (lane % 4) + e;
            a.s_mma[col * kPage + lane / 4] = sc[e];
            a.s_mma[col * kPage + lane / 4 + 8] = sc[2 + e];
        }
        float acc[8][4];
        for (int mt = 0; mt < 8; ++mt)
            for (int e = 0; e < 2; ++e) {
                const int col = 8 * j + 2 * (lane % 4) + e;
                acc[mt][e] = a.o0[col * kD + 16 * mt + lane / 4];
                acc[mt][2 + e] = a.o0[col * kD + 16 * mt + lane / 4 + 8];
            }
        const __nv_bfloat16* pr = a.p + (8 * j + lane / 4) * kPage + 2 * (lane % 4);
        const uint32_t b0 = *reinterpret_cast<const uint32_t*>(pr);
        const uint32_t b1 = *reinterpret_cast<const uint32_t*>(pr + 8);
        const int lm_j = lane >> 3, lm_r = lane & 7;
        for (int mt = 0; mt < 8; ++mt) {
            uint32_t a0, a1, a2, a3;
            bi::ldmatrix_x4_trans(bi::smem_u32(vs) + bi_attn::swz(lm_r + 8 * (lm_j >> 1), 2 * mt + (lm_j & 1)),
                                  a0, a1, a2, a3);
            bi::mma_bf16_16816(acc[mt], a0, a1, a2, a3, b0, b1);
        }
        for (int mt = 0; mt < 8; ++mt)
            for (int e = 0; e < 2; ++e) {
                const int col = 8 * j + 2 * (lane % 4) + e;
                a.o_mma[col * kD + 16 * mt + lane / 4] = acc[mt][e];
                a.o_mma[col * kD + 16 * mt + lane / 4 + 8] = acc[mt][2 + e];
            }
    }

    // tcgen05: O0 into TMEM columns [0, 128), S into [128, 144)
    const int c = 32 * warp + lane;
    const uint32_t lrow = tm + (static_cast<uint32_t>(32 * warp) << 16);
    for (int q4 = 0; q4 < kD / 32; ++q4) {
        uint32_t r[32];
        for (int i = 0; i < 32; ++i) r[i] = __float_as_uint(a.o0[c * kD + 32 * q4 + i]);
        bi::tmem_st_32x32b_x32(lrow + 32 * q4, r);
    }
    bi::tmem_st_wait();
    bi::tc_fence_before();
    __syncthreads();
    bi::tc_fence_after();
    if (tid == 0) {
        const uint64_t qd = kmajor_desc(bi::smem_u32(qs));
        const uint64_t kd = kmajor_desc(bi::smem_u32(ks));
        constexpr uint32_t idesc16 = (1u << 4) | (1u << 7) | (1u << 10) | ((16u >> 3) << 17) |
                                     ((128u >> 4) << 24);
        for (int k = 0; k < kD / 16; ++k)
            bi::tc_mma_f16(tm + 128, qd + static_cast<uint64_t>(((k >> 2) * kQHalf + 32 * (k & 3)) >> 4),
                           kd + static_cast<uint64_t>(((k >> 2) * kHalfBytes + 32 * (k & 3)) >> 4),
                           idesc16, k > 0 ? 1u : 0u);
        bi::tc_mma_f16(tm, p_desc(bi::smem_u32(ps)), v_desc(bi::smem_u32(vs)), kIdescPV, 1u);
        bi::tc_commit(bar);
    }
    __syncwarp();
    if (!bi::mbar_wait(bar, 0)) {
        if (lane == 0) bi::report_error(a.err, bi::kErrTimeout | bi::kWhereAttnSplit);
    } else {
        bi::tc_fence_after();
        uint32_t sr[16];
        bi::tmem_ld_32x32b_x16(lrow + 128, sr);
        bi::tmem_ld_wait();
        for (int i = 0; i < kPage; ++i) a.s_tc[c * kPage + i] = __uint_as_float(sr[i]);
        for (int q4 = 0; q4 < kD / 32; ++q4) {
            uint32_t r[32];
            bi::tmem_ld_32x32b_x32(lrow + 32 * q4, r);
            bi::tmem_ld_wait();
            for (int i = 0; i < 32; ++i) a.o_tc[c * kD + 32 * q4 + i] = __uint_as_float(r[i]);
        }
    }
    bi::tc_fence_before();
    __syncthreads();
    if (warp == 0) {
        bi::tc_fence_after();
        bi::tmem_dealloc(tm, 256);
    }
}

// set once per device; any thread may race to set it, the attribute is idempotent
std::atomic<bool> g_attr_set[64] = {};
std::atomic<bool> g_st_attr_set[64] = {};

}  // namespace

extern "C" size_t bi_prefill_attention_workspace_size(int32_t T, int32_t Hq, int32_t D,
                                                      int32_t max_seq_len) {
    if (T < 0 || Hq <= 0 || D <= 0 || max_seq_len <= kChunk) return 0;
    return static_cast<size_t>(T) * Hq * D * sizeof(float);
}

extern "C" bi_status bi_prefill_attention(const void* q, const void* k_cache, const void* v_cache,
                                          const int32_t* block_table, int32_t max_pages_per_seq,
                                          const int32_t* seq_lens, const int32_t* q_indptr,
                                          int32_t S, int32_t T, int32_t Hq, int32_t Hkv, int32_t D,
                                          int32_t page_size, int32_t num_pages,
                                          int32_t max_q_len, int32_t max_seq_len, float scale,
                                          void* out, void* workspace, size_t workspace_bytes,
                                          cudaStream_t stream) {
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
    const size_t need = bi_prefill_attention_workspace_size(T, Hq, D, max_seq_len);
    if (need > 0) {
        if (!workspace || workspace_bytes < need) return BI_ERR_WORKSPACE_TOO_SMALL;
        if (!bi::aligned16(workspace)) return BI_ERR_MISALIGNED;
    }

    const int group = Hq / Hkv;
    const int rows_per_tile = kCols / group;
    CUtensorMap tq, tk, tv;
    const uint64_t rows = static_cast<uint64_t>(num_pages) * Hkv * kPage;
    if (bi::encode_q_map(&tq, q, static_cast<uint64_t>(T), static_cast<uint64_t>(Hq),
                         static_cast<uint32_t>(group), static_cast<uint32_t>(rows_per_tile)) !=
            CUDA_SUCCESS ||
        bi::encode_tensor_map_2d(&tk, k_cache, kD, rows, kD * 2, 64, kPage) != CUDA_SUCCESS ||
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
    args.block_table = block_table;
    args.seq_lens = seq_lens;
    args.q_indptr = q_indptr;
    args.out = static_cast<__nv_bfloat16*>(out);
    args.ws = need > 0 ? static_cast<float*>(workspace) : nullptr;
    args.err = bi::device_error_word();
    args.max_pages_per_seq = max_pages_per_seq;
    args.Hq = Hq;
    args.Hkv = Hkv;
    args.group = group;
    args.rows_per_tile = rows_per_tile;
    args.num_pages = num_pages;
    args.max_seq_len = max_seq_len;
    args.max_q_len = max_q_len;
    args.T = T;
    args.scale_log2 = static_cast<float>(static_cast<double>(scale) * 1.4426950408889634);
    const int tiles = (max_q_len + kTiles * rows_per_tile - 1) / (kTiles * rows_per_tile);
    if (tiles > 65535) return BI_ERR_UNSUPPORTED_SHAPE;
    return bi::launch_pdl(prefill_attn_kernel, dim3(S, Hkv, tiles), dim3(kThreads), kSmemBytes,
                          stream, tq, tk, tv, args) == cudaSuccess
               ? BI_OK
               : BI_ERR_CUDA;
}

extern "C" bi_status bi_selftest_tcgen05_vs_mma_sync(const void* q, const void* k, const void* v,
                                                     const void* p, const float* o0, float* s_tc,
                                                     float* s_mma, float* o_tc, float* o_mma,
                                                     cudaStream_t stream) {
    if (!q || !k || !v || !p || !o0 || !s_tc || !s_mma || !o_tc || !o_mma) return BI_ERR_INVALID_ARG;
    if (!bi::aligned16(q) || !bi::aligned16(k) || !bi::aligned16(v) || !bi::aligned16(p) ||
        !bi::aligned16(o0))
        return BI_ERR_MISALIGNED;
    int dev = 0;
    if (cudaGetDevice(&dev) != cudaSuccess || dev < 0 || dev >= 64) return BI_ERR_CUDA;
    if (!g_st_attr_set[dev]) {
        if (cudaFuncSetAttribute(tc_selftest_kernel, cudaFuncAttributeMaxDynamicSharedMemorySize,
                                 kStSmemBytes) != cudaSuccess)
            return BI_ERR_CUDA;
        g_st_attr_set[dev] = true;
    }
    SelftestArgs args;
    args.q = static_cast<const __nv_bfloat16*>(q);
    args.k = static_cast<const __nv_bfloat16*>(k);
    args.v = static_cast<const __nv_bfloat16*>(v);
    args.p = static_cast<const __nv_bfloat16*>(p);
    args.o0 = o0;
    args.s_tc = s_tc;
    args.s_mma = s_mma;
    args.o_tc = o_tc;
    args.o_mma = o_mma;
    args.err = bi::device_error_word();
    tc_selftest_kernel<<<1, 128, kStSmemBytes, stream>>>(args);
    return cudaGetLastError() == cudaSuccess ? BI_OK : BI_ERR_CUDA;
}
