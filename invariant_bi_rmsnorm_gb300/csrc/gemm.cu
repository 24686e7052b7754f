// bi_gemm: y[M,N] = x[M,K] . W[N,K]^T on tcgen05 tensor cores, one kernel
// configuration for every shape.
//
// "Defeating Nondeterminism in LLM Inference: The Core Role of Batch
// Invariance", section "2. Batch-Invariant Matrix Multiplication": a
// data-parallel matmul gives each output tile to one core and reduces its
// whole K range there; splitting K when M*N is small, or switching tensor-core
// instruction or tile shape with the batch size, changes the reduction order.
// So this kernel has exactly one tile shape (256 x 256, computed by a pair of
// CTAs on two SMs), one MMA instruction shape (tcgen05.mma.cta_group::2
// kind::f16, M=256, N=256, K=16) and one K order (64-wide blocks ascending,
// each as 4 ascending 16-deep MMAs into one fp32 TMEM accumulator), whatever
// M, N and K are.  No split-K, no stream-K.
//
// Structure (persistent, one CTA pair per two SMs, warp-specialised):
//   warp 0      TMA producer in each CTA: its 128 rows of x and its 128 rows
//               of W (64-wide K slabs, 128-byte swizzle) into a 7-stage ring;
//               both CTAs' copies complete on the leader CTA's barrier;
//   warp 1      allocates 512 TMEM columns in both CTAs (two accumulators);
//               in the leader CTA one thread issues the pair MMAs, which read
//               both CTAs' shared memory, so each SM streams half of the W tile;
//   warps 2..5  epilogue in each CTA: tcgen05.ld of its own 128 rows of the
//               accumulator (warp w reads TMEM lanes 32*(w%4) ..), fp32 -> bf16
//               round-to-nearest-even, store.
// The fused SwiGLU variant (bi_gemm_swiglu) runs the same main loop over a
// gate|up weight whose rows are interleaved in groups of 8 (8 gate rows, then
// the 8 matching up rows); its epilogue rounds each gate and up value to bf16
// exactly as the plain GEMM would store them, then writes
// bf16(silu(gate) * up) -- the bits bi_gemm followed by bi_silu_mul give.
// Rows past M and columns past N read as zeros (TMA out-of-bounds fill) and
// are never stored; adding zero products leaves the other sums unchanged.
#include <cuda_bf16.h>

#include <algorithm>
#include <atomic>

#include "bi_internal.h"
#include "bi_ptx.cuh"

namespace {

// Shared-memory matrix descriptor for a K-major tile stored as 128-byte rows
// with the 128-byte swizzle: start address >> 4 (bits 0-13), leading byte
// offset (unused for this layout, bits 16-29), stride byte offset = 1024 bytes
// between 8-row groups (bits 32-45), the fixed 0b001 at bits 46-48, swizzle
// mode 2 = 128-byte (bits 61-63).
__device__ __forceinline__ uint64_t sw128_desc(uint32_t saddr) {
    return static_cast<uint64_t>((saddr & 0x3FFFFu) >> 4) | (uint64_t{1} << 16) |
           (uint64_t{1024 >> 4} << 32) | (uint64_t{1} << 46) | (uint64_t{2} << 61);
}

// Tile order (a schedule choice; every tile's arithmetic is the same in any
// order): groups of `group_m` M-tiles, and within a group all N-tiles with the
// M-tile fastest.  With group_m = all M-tiles this is plain m-fastest order;
// a smaller group keeps a large activation operand's slice resident in L2
// while the N-tiles sweep past it.
__device__ __forceinline__ void tile_coords(int tile, int num_m, int num_n, int group_m, int& mb,
                                            int& nb) {
    const int per_group = group_m * num_n;
    const int g = tile / per_group;
    const int r = tile - g * per_group;
    const int gm = min(group_m, num_m - g * group_m);
    mb = g * group_m + r % gm;
    nb = r / gm;
}

namespace pair {
constexpr int BMP = 256;  // pair tile rows
constexpr int BMC = 128;  // rows per CTA
constexpr int BN = 256;
constexpr int BNC = BN / 2;  // W rows per CTA
constexpr int BK = 64;
constexpr int kStages = 7;
constexpr int kABytes = BMC * BK * 2;  // 16 KiB
constexpr int kBBytes = BNC * BK * 2;  // 16 KiB
constexpr int kStageBytes = kABytes + kBBytes;
constexpr int kThreads = 192;
constexpr uint32_t kTmemCols = 512;
constexpr uint32_t kAccStride = 256;
constexpr int kSmemBytes = kStages * kStageBytes + 1024 + 256;
static_assert(kStageBytes % 1024 == 0 && kABytes % 1024 == 0, "swizzle alignment");
static_assert(BN % 16 == 0 && BN <= 256 && BN <= static_cast<int>(kAccStride), "tcgen05 shape");
// Instruction descriptor, kind::f16: D fp32 (bits 4-5 = 1), A bf16 (bits 7-9
// = 1), B bf16 (bits 10-12 = 1), both K-major (bits 15, 16 = 0), N >> 3 at
// bits 17-22, M >> 4 at bits 24-28 (M = 256: the pair's rows).
constexpr uint32_t kIdesc = (1u << 4) | (1u << 7) | (1u << 10) |
                            (static_cast<uint32_t>(BN >> 3) << 17) |
                            (static_cast<uint32_t>(BMP >> 4) << 24);
}  // namespace pair

__device__ __forceinline__ float round_bf16(uint32_t acc_bits) {
    return __bfloat162float(__float2bfloat16_rn(__uint_as_float(acc_bits)));
}

template <bool kSwiGLU>
__global__ void __cluster_dims__(2, 1, 1) __launch_bounds__(pair::kThreads, 1)
    gemm_tcgen05_pair_kernel(const __grid_constant__ CUtensorMap tmap_x,
                             const __grid_constant__ CUtensorMap tmap_w,
                             __nv_bfloat16* __restrict__ y, int M, int N, int K, int64_t ld_y,
                             int group_m, uint32_t* err) {
    constexpr int BMP = pair::BMP, BMC = pair::BMC, BN = pair::BN, BNC = pair::BNC, BK = pair::BK;
    constexpr int kStages = pair::kStages, kABytes = pair::kABytes, kStageBytes = pair::kStageBytes;
    constexpr uint32_t kTmemCols = pair::kTmemCols, kAccStride = pair::kAccStride;
    constexpr uint32_t kIdesc = pair::kIdesc;
    extern __shared__ uint8_t smem_raw[];
    uint8_t* smem = reinterpret_cast<uint8_t*>(
        (reinterpret_cast<uintptr_t>(smem_raw) + 1023) & ~static_cast<uintptr_t>(1023));
    uint64_t* full = reinterpret_cast<uint64_t*>(smem + kStages * kStageBytes);
    uint64_t* empty = full + kStages;
    uint64_t* tfull = empty + kStages;
    uint64_t* tempty = tfull + 2;
    uint64_t* drain = tempty + 2;  // MMA completion after a timeout
    uint32_t* tmem_slot = reinterpret_cast<uint32_t*>(drain + 1);
    __shared__ int s_timeout;    // a role of this CTA gave up on a wait
    __shared__ int s_issued;     // k-block loads the producer issued
    __shared__ int s_consumed;   // k-block loads the MMA thread saw land

    const uint32_t rank = bi::cluster_ctarank();
    const bool leader = rank == 0;
    const int warp = threadIdx.x >> 5;
    const int lane = threadIdx.x & 31;
    const int num_m = (M + BMP - 1) / BMP;
    const int num_n = (N + BN - 1) / BN;
    const int num_tiles = num_m * num_n;
    const int num_kb = (K + BK - 1) / BK;
    const int pair_id = blockIdx.x >> 1;
    const int npairs = gridDim.x >> 1;

    if (threadIdx.x == 0) {
        for (int i = 0; i < kStages; ++i) {
            bi::mbar_init(&full[i], 1);   // the leader's arrive (+ both CTAs' bytes)
            bi::mbar_init(&empty[i], 1);  // one pair-MMA commit
        }
        for (int i = 0; i < 2; ++i) {
            bi::mbar_init(&tfull[i], 1);
            bi::mbar_init(&tempty[i], 8);  // 4 epilogue warps in each CTA (leader's copy used)
        }
        bi::mbar_init(drain, 1);
        bi::fence_mbar_init();
        s_timeout = 0;
        s_issued = 0;
        s_consumed = 0;
        bi::tma_prefetch_desc(&tmap_x);
        bi::tma_prefetch_desc(&tmap_w);
    }
    if (warp == 1) {
        bi::tmem_alloc_pair(tmem_slot, kTmemCols);
        bi::tmem_relinquish_pair();
    }
    bi::tc_fence_before();
    bi::cluster_sync();  // both CTAs' barriers exist before either signals the other
    bi::tc_fence_after();
    const uint32_t tmem_base = *tmem_slot;
    // set-up done: let the next kernel's CTAs take SMs as this grid's free up,
    // and wait for the previous kernel before any operand or output access
    bi::launch_dependents();
    bi::grid_dependency_wait();

    if (warp == 0) {
        if (lane == 0) {
            int stage = 0;
            uint32_t phase = 0;
            int issued = 0;
            for (int tile = pair_id; tile < num_tiles; tile += npairs) {
                int mb, nb;
                tile_coords(tile, num_m, num_n, group_m, mb, nb);
                for (int kb = 0; kb < num_kb; ++kb) {
                    if (!bi::mbar_wait(&empty[stage], phase ^ 1)) {
                        bi::report_error(err, bi::kErrTimeout | bi::kWhereGemmProducer);
                        s_timeout = 1;
                        goto producer_done;
                    }
                    uint8_t* sa = smem + stage * kStageBytes;
                    const uint32_t full_leader = bi::mapa_shared(bi::smem_u32(&full[stage]), 0);
                    if (leader) bi::mbar_arrive_expect_tx(&full[stage], 2 * kStageBytes);
                    bi::tma_load_2d_pair(sa, &tmap_x, full_leader, kb * BK,
                                         mb * BMP + static_cast<int>(rank) * BMC);
                    bi::tma_load_2d_pair(sa + kABytes, &tmap_w, full_leader, kb * BK,
                                         nb * BN + static_cast<int>(rank) * BNC);
                    ++issued;
                    if (++stage == kStages) {
                        stage = 0;
                        phase ^= 1;
                    }
                }
            }
        producer_done:
            s_issued = issued;
        }
    } else if (warp == 1) {
        if (lane == 0 && leader) {
            int stage = 0;
            uint32_t phase = 0;
            int acc = 0;
            uint32_t acc_phase = 0;
            int consumed = 0;
            bool issued_any = false;
            for (int tile = pair_id; tile < num_tiles; tile += npairs) {
                if (!bi::mbar_wait(&tempty[acc], acc_phase ^ 1)) {
                    bi::report_error(err, bi::kErrTimeout | bi::kWhereGemmMma);
                    s_timeout = 1;
                    break;
                }
                bi::tc_fence_after();
                const uint32_t d_tmem = tmem_base + static_cast<uint32_t>(acc) * kAccStride;
                bool ok = true;
                for (int kb = 0; kb < num_kb; ++kb) {
                    if (!bi::mbar_wait(&full[stage], phase)) {
                        bi::report_error(err, bi::kErrTimeout | bi::kWhereGemmMma);
                        s_timeout = 1;
                        ok = false;
                        break;
                    }
                    ++consumed;
                    issued_any = true;
                    bi::tc_fence_after();
                    const uint32_t sa = bi::smem_u32(smem + stage * kStageBytes);
                    const uint32_t sb = sa + kABytes;
#pragma unroll
                    for (int k = 0; k < BK / 16; ++k) {
                        bi::tc_mma_f16_pair(d_tmem, sw128_desc(sa + 32 * k),
                                            sw128_desc(sb + 32 * k), kIdesc,
                                            (kb | k) != 0 ? 1u : 0u);
                    }
                    bi::tc_commit_pair_multicast(&empty[stage], 0x3);  // stage free in both CTAs
                    if (++stage == kStages) {
                        stage = 0;
                        phase ^= 1;
                    }
                }
                if (!ok) break;
                bi::tc_commit_pair_multicast(&tfull[acc], 0x3);  // both halves of D ready
                if (++acc == 2) {
                    acc = 0;
                    acc_phase ^= 1;
                }
            }
            s_consumed = consumed;
            if (s_timeout && issued_any) {
                // the MMAs issued so far may still be reading shared memory and
                // writing TMEM: a bounded wait for them before both are freed
                bi::tc_commit_pair_multicast(drain, 0x1);
                bi::mbar_wait_for(drain, 0, bi::kDrainNs);
            }
        }
    } else {
        // epilogue warps 2..5 -> TMEM lane quarter warp % 4 of this CTA's 128 rows
        const int quarter = warp & 3;
        int acc = 0;
        uint32_t acc_phase = 0;
        for (int tile = pair_id; tile < num_tiles; tile += npairs) {
            int mb, nb;
            tile_coords(tile, num_m, num_n, group_m, mb, nb);
            if (!bi::mbar_wait(&tfull[acc], acc_phase)) {
                if (lane == 0) {
                    bi::report_error(err, bi::kErrTimeout | bi::kWhereGemmEpilogue);
                    s_timeout = 1;
                }
                break;
            }
            bi::tc_fence_after();
            const int row = mb * BMP + static_cast<int>(rank) * BMC + quarter * 32 + lane;
            __nv_bfloat16* yrow = y + static_cast<int64_t>(row) * ld_y;
            const uint32_t taddr = tmem_base + (static_cast<uint32_t>(quarter * 32) << 16) +
                                   static_cast<uint32_t>(acc) * kAccStride;
#pragma unroll 1
            for (int ch = 0; ch < BN / 32; ++ch) {
                const int col0 = nb * BN + ch * 32;
                if (col0 >= N) break;  // warp-uniform
                uint32_t r[32];
                bi::tmem_ld_32x32b_x32(taddr + ch * 32, r);
                bi::tmem_ld_wait();
                if (row < M && !kSwiGLU) {
#pragma unroll
                    for (int v = 0; v < 4; ++v) {
                        if (col0 + 8 * v + 8 > N) break;
                        uint4 o;
                        o.x = bi::pack_bf16x2(__uint_as_float(r[8 * v + 0]), __uint_as_float(r[8 * v + 1]));
                        o.y = bi::pack_bf16x2(__uint_as_float(r[8 * v + 2]), __uint_as_float(r[8 * v + 3]));
                        o.z = bi::pack_bf16x2(__uint_as_float(r[8 * v + 4]), __uint_as_float(r[8 * v + 5]));
                        o.w = bi::pack_bf16x2(__uint_as_float(r[8 * v + 6]), __uint_as_float(r[8 * v + 7]));
                        *reinterpret_cast<uint4*>(yrow + col0 + 8 * v) = o;
                    }
                } else if (row < M) {
                    // two groups of 16 accumulator columns: 8 gate, then 8 up
#pragma unroll
                    for (int v = 0; v < 2; ++v) {
                        if (col0 + 16 * v + 16 > N) break;
                        uint32_t o[4];
#pragma unroll
                        for (int e = 0; e < 4; ++e) {
                            const float h0 = bi::swiglu(round_bf16(r[16 * v + 2 * e]),
                                                        round_bf16(r[16 * v + 8 + 2 * e]));
                            const float h1 = bi::swiglu(round_bf16(r[16 * v + 2 * e + 1]),
                                                        round_bf16(r[16 * v + 8 + 2 * e + 1]));
                            o[e] = bi::pack_bf16x2(h0, h1);
                        }
                        *reinterpret_cast<uint4*>(yrow + (col0 + 16 * v) / 2) =
                            make_uint4(o[0], o[1], o[2], o[3]);
                    }
                }
            }
            bi::tc_fence_before();
            __syncwarp();
            if (lane == 0) bi::mbar_arrive_cluster(bi::mapa_shared(bi::smem_u32(&tempty[acc]), 0));
            if (++acc == 2) {
                acc = 0;
                acc_phase ^= 1;
            }
        }
    }

    __syncthreads();
    if (s_timeout && leader && threadIdx.x == 0) {
        // Loads issued but never seen to land (at most one ring's worth): a
        // bounded wait for each before the pair's shared memory is released.
        // The leader's barriers count both CTAs' bytes, and both producers
        // walk the same stage sequence, so this covers the peer's copies.
        for (int i = s_consumed; i < s_issued; ++i)
            bi::mbar_wait_for(&full[i % kStages], (i / kStages) & 1, bi::kDrainNs);
    }
    bi::tc_fence_before();
    bi::cluster_sync();  // both CTAs past their last TMEM access and remote arrive
    if (warp == 1) {
        bi::tc_fence_after();
        bi::tmem_dealloc_pair(tmem_base, kTmemCols);
    }
}

// set once per device; any thread may race to set it, the attribute is idempotent
std::atomic<bool> g_attr_set[2][64] = {};

// Validate and launch.  N is the weight's row count (the accumulator width);
// the output has N columns, or N/2 for the fused SwiGLU variant.
template <bool kSwiGLU>
bi_status launch_gemm(const void* x, const void* W, void* y, int32_t M, int32_t N, int32_t K,
                      int64_t ld_x, int64_t ld_w, int64_t ld_y, cudaStream_t stream) {
    const int64_t out_cols = kSwiGLU ? N / 2 : N;
    if (M < 0 || N < 8 || K < 8) return M < 0 ? BI_ERR_INVALID_ARG : BI_ERR_UNSUPPORTED_SHAPE;
    if (M > 0x7fffffff - pair::BMP) return BI_ERR_UNSUPPORTED_SHAPE;  // row indices stay in int
    if ((N & (kSwiGLU ? 15 : 7)) || (K & 7)) return BI_ERR_UNSUPPORTED_SHAPE;
    if (ld_x < K || ld_w < K || ld_y < out_cols) return BI_ERR_INVALID_ARG;
    if ((ld_x & 7) || (ld_w & 7) || (ld_y & 7)) return BI_ERR_MISALIGNED;
    if (M == 0) return BI_OK;
    if (!x || !W || !y) return BI_ERR_INVALID_ARG;
    if (!bi::aligned16(x) || !bi::aligned16(W) || !bi::aligned16(y)) return BI_ERR_MISALIGNED;

    // TMA boxes: each CTA loads 128 rows of x and 128 rows of W per 64-wide K slab
    CUtensorMap tx, tw;
    if (bi::encode_tensor_map_2d(&tx, x, static_cast<uint64_t>(K), static_cast<uint64_t>(M),
                                 static_cast<uint64_t>(ld_x) * 2, pair::BK, pair::BMC) != CUDA_SUCCESS ||
        bi::encode_tensor_map_2d(&tw, W, static_cast<uint64_t>(K), static_cast<uint64_t>(N),
                                 static_cast<uint64_t>(ld_w) * 2, pair::BK, pair::BNC) != CUDA_SUCCESS)
        return BI_ERR_CUDA;

    int dev = 0;
    if (cudaGetDevice(&dev) != cudaSuccess || dev < 0 || dev >= 64) return BI_ERR_CUDA;
    if (!g_attr_set[kSwiGLU][dev]) {
        if (cudaFuncSetAttribute(gemm_tcgen05_pair_kernel<kSwiGLU>,
                                 cudaFuncAttributeMaxDynamicSharedMemorySize,
                                 pair::kSmemBytes) != cudaSuccess)
            return BI_ERR_CUDA;
        g_attr_set[kSwiGLU][dev] = true;
    }
    const int sms = bi::sm_count();
    if (sms < 2) return BI_ERR_CUDA;
    const int num_m = (M + pair::BMP - 1) / pair::BMP;
    const int64_t tiles = static_cast<int64_t>(num_m) * ((N + pair::BN - 1) / pair::BN);
    if (tiles > 0x7fffffffLL) return BI_ERR_UNSUPPORTED_SHAPE;
    const int pairs = static_cast<int>(tiles < sms / 2 ? tiles : sms / 2);
    // Tile order: keep at most ~48 MB of the activation operand per group of
    // M-tiles, so a large x stays L2-resident while the N-tiles sweep past it
    // (48 MB measured best: equal to 64-96 MB at M = 4096, 2.5-3.5 % faster at
    // M = 8192 for qkv, o and gate|up).
    const int64_t slab = static_cast<int64_t>(pair::BMP) * K * 2;
    const int64_t budget = int64_t{48} << 20;
    int group_m = num_m;
    if (slab * num_m > budget) group_m = static_cast<int>(std::max<int64_t>(1, budget / slab));
    // programmatic serialization: this grid's set-up may overlap the previous
    // kernel's tail (the kernel waits for it before touching memory)
    if (bi::launch_pdl(gemm_tcgen05_pair_kernel<kSwiGLU>, dim3(2 * pairs), dim3(pair::kThreads),
                       pair::kSmemBytes, stream, tx, tw, static_cast<__nv_bfloat16*>(y), M, N, K,
                       ld_y, group_m, bi::device_error_word()) != cudaSuccess)
        return BI_ERR_CUDA;
    return cudaGetLastError() == cudaSuccess ? BI_OK : BI_ERR_CUDA;
}

}  // namespace

extern "C" bi_status bi_gemm(const void* x, const void* W, void* y, int32_t M, int32_t N,
                             int32_t K, int64_t ld_x, int64_t ld_w, int64_t ld_y,
                             cudaStream_t stream) {
    return launch_gemm<false>(x, W, y, M, N, K, ld_x, ld_w, ld_y, stream);
}

extern "C" bi_status bi_gemm_swiglu(const void* x, const void* W_gu, void* h, int32_t M,
                                    int32_t F, int32_t K, int64_t ld_x, int64_t ld_w,
                                    int64_t ld_h, cudaStream_t stream) {
    if (F < 8 || F > (0x7fffffff >> 1)) return BI_ERR_UNSUPPORTED_SHAPE;
    return launch_gemm<true>(x, W_gu, h, M, 2 * F, K, ld_x, ld_w, ld_h, stream);
}
