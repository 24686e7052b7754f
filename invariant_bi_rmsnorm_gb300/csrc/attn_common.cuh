// The per-page step of fixed-split-size attention, shared by the decode and
// prefill kernels so that a query row gets the same bits from either.
//
// Arithmetic of one query row (one column) over one 256-token chunk: an online
// softmax over the chunk's pages 0, 1, 2, ... in order.  For a page of 16
// tokens (rows of K and V) and 8 columns (query head x query row pairs):
//     S^T[16 x 8] = K_page[16 x 128] . Q^T[128 x 8]       8 mma.sync, dims ascending
//     x = S * scale * log2(e)        (tokens past a column's length -> -inf)
//     m' = max_t x if it exceeds m by more than kRescaleSlack, else m;
//     alpha = 2^(m - m') (exactly 1 when m' = m);  p = 2^(x - m')  (fp32)
//     l' = l * alpha + sum_t p       (fixed xor-butterfly order over tokens)
//     p = p_hi + p_lo with p_hi = bf16(p), p_lo = bf16(p - p_hi)
//     O^T[128 x 8] = (O^T * alpha + V^T . P_hi^T) + V^T . P_lo^T   16 mma.sync
// Splitting p keeps the weights to about 16 significant bits in the PV
// product (one bf16 operand alone would keep 8), at the price of a second
// mma per 16 dims -- cheap in a kernel bound by HBM.
// Each output element of an mma depends only on its own column, so a column's
// result does not depend on what shares the tile with it.
//
// Shared-memory layout of one page block (K or V), as written by one TMA box
// of 64 dims x 16 rows x 2 halves with the 128-byte swizzle: dims
// [64*(ch/8), +64) at offset (ch/8)*2048, 128-byte rows, the 16-byte unit
// index XORed with (row % 8).
#pragma once
#include <cuda_bf16.h>

#include <cmath>

#include "bi_ptx.cuh"

namespace bi_attn {

constexpr int kD = 128;
constexpr int kPage = BI_PAGE_SIZE;             // 16 tokens
constexpr int kChunk = BI_DECODE_CHUNK;         // 256 tokens
constexpr int kPagesPerChunk = kChunk / kPage;  // 16
constexpr int kHalfBytes = kPage * 64 * 2;      // 16 rows x 64 dims: one TMA box
constexpr int kMatBytes = 2 * kHalfBytes;       // one (page, kv-head) K or V block
constexpr int kStageBytes = 2 * kMatBytes;      // K + V
constexpr int kMaxGroup = 8;                    // query heads per kv-head

__device__ __forceinline__ uint32_t swz(int r, int ch) {
    return static_cast<uint32_t>((ch >> 3) * kHalfBytes + r * 128 + (((ch & 7) ^ (r & 7)) << 4));
}

// Online-softmax state of one warp for 8 columns.  Lane l holds columns
// 2(l%4) and 2(l%4)+1: m, l for both, and O[d][col] for d = 16mt + l/4 (+8).
struct ColState {
    float m[2];
    float l[2];
    float acc[8][4];
};

__device__ __forceinline__ void colstate_init(ColState& st) {
    st.m[0] = st.m[1] = -INFINITY;
    st.l[0] = st.l[1] = 0.f;
#pragma unroll
    for (int mt = 0; mt < 8; ++mt) st.acc[mt][0] = st.acc[mt][1] = st.acc[mt][2] = st.acc[mt][3] = 0.f;
}

// Q^T fragments (mma B operand) for the 8 columns: lane l supplies column l/4
// whose 128-dim query starts at `col_q` (nullptr: a padding column, zeros).
__device__ __forceinline__ void load_q_frags(const __nv_bfloat16* col_q, int lane, uint32_t (&qb0)[8],
                                             uint32_t (&qb1)[8]) {
    const __nv_bfloat16* qp = col_q ? col_q + 2 * (lane & 3) : nullptr;
#pragma unroll
    for (int ks = 0; ks < 8; ++ks) {
        qb0[ks] = qp ? *reinterpret_cast<const uint32_t*>(qp + 16 * ks) : 0u;
        qb1[ks] = qp ? *reinterpret_cast<const uint32_t*>(qp + 16 * ks + 8) : 0u;
    }
}

// P^T fragments of one page for one 8-column group: the bf16 high parts and
// the bf16 remainders (mma B operands, tokens on K, columns on N).
struct PFrags {
    uint32_t hi0, hi1, lo0, lo1;
};

// The page's raw scores S^T = K_page . Q^T for this lane's 4 entries: sc[0],
// sc[1] are token l/4 for columns 2(l%4) and 2(l%4)+1, sc[2], sc[3] token
// l/4 + 8.  Eight MMAs over the dims in ascending 16-blocks into one
// accumulator.
__device__ __forceinline__ void page_scores(float (&sc)[4], uint32_t ks_base,
                                            const uint32_t (&qb0)[8], const uint32_t (&qb1)[8],
                                            int lane) {
    const int lm_j = lane >> 3;  // which 8x8 matrix this lane addresses
    const int lm_r = lane & 7;   // row within it
#pragma unroll
    for (int i = 0; i < 4; ++i) sc[i] = 0.f;
#pragma unroll
    for (int ks = 0; ks < 8; ++ks) {
        uint32_t a0, a1, a2, a3;
        bi::ldmatrix_x4(ks_base + swz(lm_r + 8 * (lm_j & 1), 2 * ks + (lm_j >> 1)), a0, a1, a2, a3);
        bi::mma_bf16_16816(sc, a0, a1, a2, a3, qb0[ks], qb1[ks]);
    }
}

// The reference maximum m of a column moves only when a page's maximum
// exceeds it by more than this many log2 units (a factor of 256): below
// that, the page's weights stay at most 2^8 and the running sum and output
// keep their scale -- alpha is exactly 1, so the output needs no rescaling.
// The result is the same softmax (the final O / l does not depend on the
// reference); only the rounding sequence is fixed differently.
constexpr float kRescaleSlack = 8.f;

// 2^x as one ex2.approx.ftz.f32 (bi::ex2_approx) on the per-page dependency
// chain, where exp2f() takes several instructions.  Decode, prefill and the
// chunk folds all take their exponentials from here.
__device__ __forceinline__ float exp2_ftz(float x) { return bi::ex2_approx(x); }

// Online-softmax update of one column group from its raw scores: masking,
// running max, the rescale of l and O, p = 2^(x - m), l += sum p, and p split
// into bf16 high part + bf16 remainder, transposed into mma B fragments.
// Every operation is an explicit rounding intrinsic, so the compiler cannot
// fuse a different pair of them in one caller than in another.
__device__ __forceinline__ void softmax_step(ColState& st, const float (&sc)[4], int valid0,
                                             int valid1, float scale_log2, int lane, PFrags& pf) {
    const int tokA = lane >> 2, tokB = tokA + 8;
    const float x0 = tokA < valid0 ? __fmul_rn(sc[0], scale_log2) : -INFINITY;
    const float x1 = tokA < valid1 ? __fmul_rn(sc[1], scale_log2) : -INFINITY;
    const float x2 = tokB < valid0 ? __fmul_rn(sc[2], scale_log2) : -INFINITY;
    const float x3 = tokB < valid1 ? __fmul_rn(sc[3], scale_log2) : -INFINITY;
    float mx0 = fmaxf(x0, x2), mx1 = fmaxf(x1, x3);
#pragma unroll
    for (int off = 4; off <= 16; off <<= 1) {
        mx0 = fmaxf(mx0, __shfl_xor_sync(0xffffffffu, mx0, off));
        mx1 = fmaxf(mx1, __shfl_xor_sync(0xffffffffu, mx1, off));
    }
    // the reference moves only past the slack; a column with no visible token
    // so far keeps m = -inf (-inf + slack is -inf): no rescale, p = 0
    const float mn0 = mx0 > __fadd_rn(st.m[0], kRescaleSlack) ? mx0 : st.m[0];
    const float mn1 = mx1 > __fadd_rn(st.m[1], kRescaleSlack) ? mx1 : st.m[1];
    const float al0 = mn0 == st.m[0] ? 1.f : exp2_ftz(__fsub_rn(st.m[0], mn0));
    const float al1 = mn1 == st.m[1] ? 1.f : exp2_ftz(__fsub_rn(st.m[1], mn1));
    const float p0 = x0 == -INFINITY ? 0.f : exp2_ftz(__fsub_rn(x0, mn0));
    const float p1 = x1 == -INFINITY ? 0.f : exp2_ftz(__fsub_rn(x1, mn1));
    const float p2 = x2 == -INFINITY ? 0.f : exp2_ftz(__fsub_rn(x2, mn0));
    const float p3 = x3 == -INFINITY ? 0.f : exp2_ftz(__fsub_rn(x3, mn1));
    const uint32_t pA = bi::pack_bf16x2(p0, p1);  // high parts
    const uint32_t pB = bi::pack_bf16x2(p2, p3);
    const uint32_t rA = bi::pack_bf16x2(__fsub_rn(p0, __uint_as_float(pA << 16)),
                                        __fsub_rn(p1, __uint_as_float(pA & 0xffff0000u)));
    const uint32_t rB = bi::pack_bf16x2(__fsub_rn(p2, __uint_as_float(pB << 16)),
                                        __fsub_rn(p3, __uint_as_float(pB & 0xffff0000u)));
    float ps0 = __fadd_rn(p0, p2);
    float ps1 = __fadd_rn(p1, p3);
#pragma unroll
    for (int off = 4; off <= 16; off <<= 1) {
        ps0 = __fadd_rn(ps0, __shfl_xor_sync(0xffffffffu, ps0, off));
        ps1 = __fadd_rn(ps1, __shfl_xor_sync(0xffffffffu, ps1, off));
    }
    st.l[0] = __fmaf_rn(st.l[0], al0, ps0);
    st.l[1] = __fmaf_rn(st.l[1], al1, ps1);
    st.m[0] = mn0;
    st.m[1] = mn1;
#pragma unroll
    for (int mt = 0; mt < 8; ++mt) {
        st.acc[mt][0] = __fmul_rn(st.acc[mt][0], al0);
        st.acc[mt][1] = __fmul_rn(st.acc[mt][1], al1);
        st.acc[mt][2] = __fmul_rn(st.acc[mt][2], al0);
        st.acc[mt][3] = __fmul_rn(st.acc[mt][3], al1);
    }
    // P^T fragments (tokens on K, columns on N) by an in-register transpose
    pf.hi0 = bi::movmatrix_trans(pA);
    pf.hi1 = bi::movmatrix_trans(pB);
    pf.lo0 = bi::movmatrix_trans(rA);
    pf.lo1 = bi::movmatrix_trans(rB);
}

// softmax_step for one column whose 16 raw scores of the page one thread
// holds whole (s[t] = score of token t): the same operations on the same
// values, so the column's state and weights get the same bits.  The page max
// is exact in any order; the sum of the 16 weights follows softmax_step's
// butterfly exactly: pairs (t, t + 8), then token groups j with j ^ 1, with
// j ^ 2, with j ^ 4 (each fp32 addition commutative).  Returns alpha, the
// factor the column's O is rescaled by; hi[i] / lo[i] receive the bf16 high
// parts and remainders of tokens 2i, 2i + 1 (token 2i in the low half).
__device__ __forceinline__ float softmax_page_col(float& m, float& l, const float (&s)[16],
                                                  int valid, float scale_log2, uint32_t (&hi)[8],
                                                  uint32_t (&lo)[8]) {
    float x[16];
#pragma unroll
    for (int t = 0; t < 16; ++t) x[t] = t < valid ? __fmul_rn(s[t], scale_log2) : -INFINITY;
    float mx = x[0];
#pragma unroll
    for (int t = 1; t < 16; ++t) mx = fmaxf(mx, x[t]);
    const float mn = mx > __fadd_rn(m, kRescaleSlack) ? mx : m;
    const float al = mn == m ? 1.f : exp2_ftz(__fsub_rn(m, mn));
    float p[16];
#pragma unroll
    for (int t = 0; t < 16; ++t) p[t] = x[t] == -INFINITY ? 0.f : exp2_ftz(__fsub_rn(x[t], mn));
#pragma unroll
    for (int i = 0; i < 8; ++i) {
        hi[i] = bi::pack_bf16x2(p[2 * i], p[2 * i + 1]);
        lo[i] = bi::pack_bf16x2(__fsub_rn(p[2 * i], __uint_as_float(hi[i] << 16)),
                                __fsub_rn(p[2 * i + 1], __uint_as_float(hi[i] & 0xffff0000u)));
    }
    float a[8];
#pragma unroll
    for (int j = 0; j < 8; ++j) a[j] = __fadd_rn(p[j], p[j + 8]);
    const float b0 = __fadd_rn(a[0], a[1]), b2 = __fadd_rn(a[2], a[3]);
    const float b4 = __fadd_rn(a[4], a[5]), b6 = __fadd_rn(a[6], a[7]);
    const float ps = __fadd_rn(__fadd_rn(b0, b2), __fadd_rn(b4, b6));
    l = __fmaf_rn(l, al, ps);
    m = mn;
    return al;
}

// O^T += V^T . P_hi^T, then += V^T . P_lo^T, per 16-dim tile in ascending
// order.
__device__ __forceinline__ void pv_step(ColState& st, const PFrags& pf, uint32_t vs_base,
                                        int lane) {
    const int lm_j = lane >> 3;
    const int lm_r = lane & 7;
#pragma unroll
    for (int mt = 0; mt < 8; ++mt) {
        uint32_t a0, a1, a2, a3;
        bi::ldmatrix_x4_trans(vs_base + swz(lm_r + 8 * (lm_j >> 1), 2 * mt + (lm_j & 1)), a0, a1, a2, a3);
        bi::mma_bf16_16816(st.acc[mt], a0, a1, a2, a3, pf.hi0, pf.hi1);
        bi::mma_bf16_16816(st.acc[mt], a0, a1, a2, a3, pf.lo0, pf.lo1);
    }
}

// One page for one 8-column group.  valid0 / valid1: how many of the page's
// 16 tokens columns 2(l%4) and 2(l%4)+1 may see (0 .. 16).  A column that sees
// none of them keeps its state unchanged.
__device__ __forceinline__ void attend_page(ColState& st, uint32_t ks_base, uint32_t vs_base,
                                            const uint32_t (&qb0)[8], const uint32_t (&qb1)[8],
                                            int valid0, int valid1, float scale_log2, int lane) {
    float sc[4];
    page_scores(sc, ks_base, qb0, qb1, lane);
    PFrags pf;
    softmax_step(st, sc, valid0, valid1, scale_log2, lane, pf);
    pv_step(st, pf, vs_base, lane);
}

// Zero V rows [valid, 16) of a page block in shared memory (one warp).
__device__ __forceinline__ void zero_v_tail(uint8_t* vd, int valid, int lane) {
    for (int idx = lane; idx < (kPage - valid) * 16; idx += 32) {
        const int r = valid + (idx >> 4), ch = idx & 15;
        *reinterpret_cast<uint4*>(vd + swz(r, ch)) = make_uint4(0, 0, 0, 0);
    }
}

// Fold step shared by every chunk fold (in-CTA and the merge kernel):
//   M' = max(M, m_c);  fo = 2^(M - M');  fc = 2^(m_c - M');
//   l' = fma(l_c, fc, l * fo);  O' = fma(O_c, fc, O * fo).
__device__ __forceinline__ void fold_scalars(float M, float mc, float& Mn, float& fo, float& fc) {
    Mn = fmaxf(M, mc);
    fo = exp2_ftz(M - Mn);
    fc = exp2_ftz(mc - Mn);
}

__device__ __forceinline__ float fold_value(float acc, float fo, float part, float fc) {
    return __fmaf_rn(part, fc, __fmul_rn(acc, fo));
}

// A column's output is its folded weighted sum of values times the
// reciprocal of its folded weight sum: one correctly rounded reciprocal per
// column and one rounded product per element (a division per element costs
// several times more).  Every path normalises through these two, so decode,
// its fold kernel and prefill round alike.
__device__ __forceinline__ float inv_weight(float l) { return __frcp_rn(l); }
__device__ __forceinline__ float normalise(float acc, float inv_l) { return __fmul_rn(acc, inv_l); }

}  // namespace bi_attn
