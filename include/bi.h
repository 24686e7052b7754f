/*
 * bi.h -- batch-invariant forward kernels for LLM inference on GB300 (sm_103a).
 *
 * C ABI of libbi.so.  Every entry point takes plain device pointers, sizes and
 * a CUDA stream; none allocates memory, keeps per-call state, or synchronises
 * the stream (except bi_get_device_error).  All launches are asynchronous on
 * `stream`.  Arguments are validated on the host before anything is launched:
 * an invalid call returns an error status and launches nothing.  Kernels are
 * launched with programmatic stream serialization: a kernel may be scheduled,
 * and do its set-up, while the previous kernel on the stream finishes, but it
 * waits for that kernel to complete before it reads or writes global memory,
 * so stream order holds as for any launch.
 *
 * The property every kernel here guarantees ("batch invariance", after
 * "Defeating Nondeterminism in LLM Inference: The Core Role of Batch
 * Invariance", section "Batch Invariance: The True Culprit"): the bits of one
 * request's output depend only on that request's own inputs -- never on the
 * batch size, the request's row position in the batch, the other requests in
 * the batch, or (for attention) how many more tokens the KV cache holds
 * beyond the request's own length.  Each output's floating-point reduction
 * order is a fixed function of the problem's static sizes (hidden, K, D) and,
 * for attention, of the request's own KV length.
 *
 * Data types: all activations, weights, caches and outputs are bf16
 * (IEEE binary32 truncated to its top 16 bits); arithmetic is fp32; every
 * output is rounded once, to nearest-even, to bf16.
 */
#ifndef BI_H_
#define BI_H_

#include <stddef.h>
#include <stdint.h>

#include <cuda_runtime_api.h>

#ifdef __cplusplus
extern "C" {
#endif

#define BI_ABI_VERSION 2

/* Tokens per KV-cache page and per attention split.  Both are fixed: the
 * split size is part of the arithmetic (see bi_decode_attention). */
#define BI_PAGE_SIZE 16
#define BI_DECODE_CHUNK 256
/* Bytes of arrival counters at the start of a decode-attention workspace. */
#define BI_DECODE_COUNTER_BYTES 262144

typedef enum {
    BI_OK = 0,
    BI_ERR_INVALID_ARG = 1,        /* null pointer, negative size, bad eps ... */
    BI_ERR_UNSUPPORTED_SHAPE = 2,  /* a size the library does not handle */
    BI_ERR_MISALIGNED = 3,         /* pointer or leading dimension not 16-byte aligned */
    BI_ERR_WORKSPACE_TOO_SMALL = 4,
    BI_ERR_CUDA = 5,               /* a CUDA runtime call or launch failed */
    BI_ERR_DEVICE_TIMEOUT = 6,     /* a kernel gave up waiting on a barrier */
    BI_ERR_DEVICE_BAD_INPUT = 7    /* a kernel found an invalid device-resident
                                      input (seq_lens / block_table entry) */
} bi_status;

/* BI_ABI_VERSION of the loaded library. */
int bi_abi_version(void);

/* Static, human-readable name of a status code. */
const char* bi_status_string(bi_status s);

/* Synchronise `stream`, then read and clear the current device's error word.
 * Kernels that detect a problem on the device (a barrier wait that ran past
 * its limit, a sequence length or page index out of range) record the first
 * such event there and stop work on the affected output instead of faulting.
 * Returns BI_OK, BI_ERR_DEVICE_TIMEOUT, BI_ERR_DEVICE_BAD_INPUT or BI_ERR_CUDA. */
bi_status bi_get_device_error(cudaStream_t stream);

/* Self-test of the device-side timeout path: launch one CTA whose bounded
 * barrier wait is made to run out -- it waits for `limit_us` microseconds
 * (1 .. 2,000,000) on an mbarrier nothing arrives on, then records
 * BI_ERR_DEVICE_TIMEOUT in the error word and exits normally.  The wait
 * routine is the one every kernel of the library uses (their limit is about
 * two seconds).  Read the result with bi_get_device_error.  Errors:
 * INVALID_ARG, CUDA. */
bi_status bi_selftest_wait_timeout(int32_t limit_us, cudaStream_t stream);

/*
 * bi_rmsnorm -- y[r][i] = bf16( x[r][i] * rsqrt(mean_j x[r][j]^2 + eps) * w[i] )
 *
 * Operation: RMSNorm as in "Defeating Nondeterminism in LLM Inference: The
 * Core Role of Batch Invariance", section "1. Batch-Invariant RMSNorm": each
 * row is reduced entirely by one CTA ("data-parallel RMSNorm"); no split
 * reduction is used at any batch size.  The sum of squares is accumulated in
 * fp32 in an order that depends only on `hidden`.
 *
 *   x      device, bf16 [rows][ld_x], row-major; only the first `hidden`
 *          elements of each row are read.
 *   w      device, bf16 [hidden].
 *   y      device, bf16 [rows][ld_y]; may alias x when ld_y == ld_x.
 *   rows   0 .. 2^31-1 (0 launches nothing).
 *   hidden multiple of 8, 8 .. 32768.
 *   ld_x, ld_y  in elements, >= hidden, multiples of 8 (16-byte rows).
 *   eps    finite, >= 0.
 * Pointers must be 16-byte aligned.  Errors: INVALID_ARG, UNSUPPORTED_SHAPE,
 * MISALIGNED, CUDA.
 */
bi_status bi_rmsnorm(const void* x, const void* w, void* y, int64_t rows, int32_t hidden,
                     int64_t ld_x, int64_t ld_y, float eps, cudaStream_t stream);

/*
 * bi_add_rmsnorm -- the residual add fused with the RMSNorm that follows it:
 *     residual[r][i] = bf16(residual[r][i] + x[r][i])      (written back)
 *     y[r][i]        = RMSNorm(residual[r])[i] * w[i]        as bi_rmsnorm
 * bit-identical to an elementwise add followed by bi_rmsnorm, in one pass.
 * Pointwise adds are batch-invariant ("Achieving Batch-Invariant Kernels");
 * the reduction is bi_rmsnorm's.  y must not overlap residual or x.
 * Arguments and errors as bi_rmsnorm, plus residual [rows][ld_res].
 */
bi_status bi_add_rmsnorm(const void* x, void* residual, const void* w, void* y, int64_t rows,
                         int32_t hidden, int64_t ld_x, int64_t ld_res, int64_t ld_y, float eps,
                         cudaStream_t stream);

/*
 * bi_gemm -- y[M][N] = bf16( x[M][K] . W[N][K]^T ), fp32 accumulation.
 *
 * Operation: "2. Batch-Invariant Matrix Multiplication" of the same page: a
 * data-parallel tiled matmul with ONE kernel configuration for every shape --
 * a fixed 256x256 output tile computed by a pair of CTAs (tcgen05.mma
 * cta_group::2, M=256, N=256, K=16), K walked in ascending 64-wide blocks,
 * each block as four ascending 16-deep MMAs accumulating in TMEM.  No split-K
 * or stream-K for any M, and the same MMA instruction shape always.
 *
 *   x  device, bf16 [M][ld_x] row-major (K contiguous).
 *   W  device, bf16 [N][ld_w] row-major: the nn.Linear weight layout.
 *   y  device, bf16 [M][ld_y] row-major; must not overlap x or W.
 *   M  0 .. 2^31-257;  N, K  >= 8 and multiples of 8.
 *   ld_x, ld_w, ld_y  in elements, multiples of 8, >= K, >= K, >= N.
 * Pointers must be 16-byte aligned.  Errors: INVALID_ARG, UNSUPPORTED_SHAPE,
 * MISALIGNED, CUDA.
 */
bi_status bi_gemm(const void* x, const void* W, void* y, int32_t M, int32_t N, int32_t K,
                  int64_t ld_x, int64_t ld_w, int64_t ld_y, cudaStream_t stream);

/*
 * bi_gemm_swiglu -- the gate|up projection of a SwiGLU MLP fused with the
 * SwiGLU product:
 *     h[M][F] = bf16( silu(g) * u ),  g = bf16((x . W_gate^T)[m][j]),
 *                                     u = bf16((x . W_up^T)[m][j])
 * with silu(g) = g / (1 + exp(-g)) in fp32 -- bit-identical to bi_gemm into a
 * [M][2F] buffer followed by bi_silu_mul, without writing that buffer.
 *
 * Operation: bi_gemm's main loop (same tile, instruction shape and K order,
 * so the same batch invariance) with a pointwise epilogue ("Achieving
 * Batch-Invariant Kernels": pointwise operations are batch-invariant).  The
 * pages do not fuse it; this is a layout choice for the decoder's MLP.
 *
 *   x     device, bf16 [M][ld_x], as bi_gemm.
 *   W_gu  device, bf16 [2F][ld_w]: the gate and up weights (nn.Linear layout)
 *         with rows interleaved in groups of 8 -- rows 16i .. 16i+7 are gate
 *         rows 8i .. 8i+7 and rows 16i+8 .. 16i+15 are up rows 8i .. 8i+7.
 *   h     device, bf16 [M][ld_h]; must not overlap x or W_gu.
 *   M  0 .. 2^31-257;  F >= 8 and a multiple of 8;  K >= 8, multiple of 8.
 *   ld_x, ld_w, ld_h  in elements, multiples of 8, >= K, >= K, >= F.
 * Pointers must be 16-byte aligned.  Errors as bi_gemm.
 */
bi_status bi_gemm_swiglu(const void* x, const void* W_gu, void* h, int32_t M, int32_t F,
                         int32_t K, int64_t ld_x, int64_t ld_w, int64_t ld_h,
                         cudaStream_t stream);

/*
 * Workspace bytes bi_decode_attention needs for B sequences of at most
 * max_seq_len tokens with Hq query heads of size D: BI_DECODE_COUNTER_BYTES of
 * arrival counters, then one fp32 partial (max, sum, D-vector) per (sequence,
 * query head, 256-token chunk).  0 when max_seq_len <= 256 (no sequence has a
 * second chunk, nothing is written) and for invalid arguments.
 */
size_t bi_decode_attention_workspace_size(int32_t B, int32_t Hq, int32_t D, int32_t max_seq_len);

/* Number of 256-token chunks a sequence of `seq_len` tokens is cut into
 * (ceil(seq_len / 256)), and the length of chunk c (256 for all but the last).
 * 0 for invalid arguments. */
int32_t bi_decode_num_chunks(int32_t seq_len);
int32_t bi_decode_chunk_len(int32_t seq_len, int32_t c);

/*
 * bi_decode_attention -- one query row per sequence attends over that
 * sequence's paged KV cache:
 *     out[s][i] = softmax_t( scale * q[s][i] . k_t[g] ) . v_t[g],
 *     g = i / (Hq / Hkv),  t = 0 .. seq_lens[s]-1.
 *
 * Operation: "3. Batch-Invariant Attention" of the same page, with the fixed
 * split-SIZE strategy ("Fixed Size Split KV Strategy"; "Batch Invariance and
 * Numerical Reproducibility": 1000 tokens = 3 x 256 + 232).  Each sequence's
 * keys are cut into consecutive 256-token chunks; one warp computes each
 * chunk's partial (running max, sum of exponentials, unnormalised output)
 * with an online softmax over its 16 pages in a fixed order; the partials are
 * then folded in ascending chunk order with the log-sum-exp rule, by the CTA
 * that holds all of a sequence's chunks or else by the last of its CTAs to
 * finish (an integer arrival counter, no float atomics).  One kernel launch
 * (two only when B * Hkv > BI_DECODE_COUNTER_BYTES / 4).  The
 * arithmetic for a sequence depends only on its own length and data, never on
 * B, on other sequences, or on tokens stored past seq_lens[s].  The cache is
 * read only: the caller writes the current token's K/V into its page slot
 * BEFORE calling (one K/V layout for cached and new tokens).
 *
 *   q            device, bf16 [B][Hq][D].
 *   k_cache,
 *   v_cache      device, bf16 [num_pages][Hkv][page_size][D]: each
 *                (page, kv-head) is one contiguous page_size x D block.
 *   block_table  device, int32 [B][max_pages_per_seq]: page index of each
 *                sequence's token block t / page_size.  Entries past a
 *                sequence's last page are never read.
 *   seq_lens     device, int32 [B]: 1 .. max_seq_len tokens per sequence.
 *   B            0 .. 65535 sequences (0 launches nothing).
 *   Hq, Hkv      query and key/value heads; Hq % Hkv == 0, Hq / Hkv <= 8.
 *   D            128.   page_size  16.
 *   num_pages    pages in each cache; num_pages * Hkv * page_size < 2^31.
 *   max_seq_len  upper bound on every seq_lens entry, >= 1 and
 *                <= max_pages_per_seq * page_size; it sizes the launch grid.
 *   scale        softmax scale (1/sqrt(D) for standard attention), finite, > 0.
 *   out          device, bf16 [B][Hq][D].
 *   workspace    device, >= bi_decode_attention_workspace_size(B, Hq, D,
 *                max_seq_len) bytes, 16-byte aligned; may be null when that
 *                size is 0.  Its first BI_DECODE_COUNTER_BYTES are uint32
 *                arrival counters that MUST BE ZERO when the workspace is
 *                first used (allocate it zero-filled, or clear those bytes
 *                once); every call leaves them zero again, also a call that
 *                reports a device error, so a workspace can serve any later
 *                call without clearing.  Do not share one workspace between
 *                calls that may run at the same time.  After the counters the
 *                call leaves, for every sequence with more than one chunk,
 *                the fp32 chunk partials in the layout [B][Hq][chunks][D]
 *                (unnormalised outputs) followed by [B][Hq][chunks][2] (max
 *                in log2 units of scale*q.k, sum), chunks =
 *                ceil(max_seq_len / 256).
 * Pointers to bf16 data must be 16-byte aligned, int32 arrays 4-byte aligned.
 * Host-side errors: INVALID_ARG, UNSUPPORTED_SHAPE, MISALIGNED,
 * WORKSPACE_TOO_SMALL, CUDA.  A seq_lens entry outside 1 .. max_seq_len or a
 * block_table entry outside 0 .. num_pages-1 is found on the device: the
 * affected sequence's output is left unwritten and bi_get_device_error
 * reports BI_ERR_DEVICE_BAD_INPUT.
 */
bi_status bi_decode_attention(const void* q, const void* k_cache, const void* v_cache,
                              const int32_t* block_table, int32_t max_pages_per_seq,
                              const int32_t* seq_lens, int32_t B, int32_t Hq, int32_t Hkv,
                              int32_t D, int32_t page_size, int32_t num_pages,
                              int32_t max_seq_len, float scale, void* out, void* workspace,
                              size_t workspace_bytes, cudaStream_t stream);

/*
 * bi_prefill_attention -- many query rows per sequence (a prompt, or one
 * chunk of it), causal: sequence i's query rows are q rows
 * q_indptr[i] .. q_indptr[i+1]-1, they are its LAST n_i = q_indptr[i+1] -
 * q_indptr[i] tokens, and its row j (0-based) attends over the first
 * seq_lens[i] - n_i + 1 + j cached tokens:
 *     out[row] = softmax_t( scale * q[row] . k_t[g] ) . v_t[g].
 *
 * Operation: "3. Batch-Invariant Attention" of "Defeating Nondeterminism in
 * LLM Inference: The Core Role of Batch Invariance" (FlashAttention2-style
 * parallelism over queries, with a reduction order that does not depend on
 * how many of the sequence's tokens are processed together).  Every row uses
 * exactly bi_decode_attention's arithmetic for a sequence of its length --
 * 256-token chunks in order, one online softmax over each chunk's pages in
 * order, chunk partials folded in order -- so a token's output is
 * bit-identical whether computed here (whole prompt or any chunking of it) or
 * by bi_decode_attention.  The caller writes all n_i tokens' K/V into the
 * cache first.
 *
 *   q            device, bf16 [T][Hq][D].   out  device, bf16 [T][Hq][D].
 *   q_indptr     device, int32 [S + 1], non-decreasing, q_indptr[S] <= T.
 *   seq_lens     device, int32 [S]: cached tokens of each sequence, including
 *                its query rows (n_i <= seq_lens[i] <= max_seq_len).
 *   block_table  device, int32 [S][max_pages_per_seq], as bi_decode_attention.
 *   max_q_len    host bound on every n_i (sizes the grid).
 *   workspace    device, >= bi_prefill_attention_workspace_size(T, Hq, D,
 *                max_seq_len) bytes, 16-byte aligned; may be null when that
 *                size is 0 (no row longer than 256 tokens).  It holds the fp32
 *                running output of rows longer than one chunk between chunks;
 *                its contents need no initialisation and are undefined after.
 *   S <= 65535; other arguments as bi_decode_attention.
 * Errors: as bi_decode_attention; an inconsistent q_indptr / seq_lens entry
 * is reported on the device (BI_ERR_DEVICE_BAD_INPUT) and the sequence is
 * skipped; an out-of-range page is reported the same way, is read as zeros
 * (no fault), and the 128-column query tiles whose rows reach it are not
 * written (the sequence's other rows are).
 */
bi_status bi_prefill_attention(const void* q, const void* k_cache, const void* v_cache,
                               const int32_t* block_table, int32_t max_pages_per_seq,
                               const int32_t* seq_lens, const int32_t* q_indptr, int32_t S,
                               int32_t T, int32_t Hq, int32_t Hkv, int32_t D, int32_t page_size,
                               int32_t num_pages, int32_t max_q_len, int32_t max_seq_len,
                               float scale, void* out, void* workspace, size_t workspace_bytes,
                               cudaStream_t stream);

/*
 * bi_selftest_tcgen05_vs_mma_sync -- the premise that lets prefill run on
 * tcgen05 and still match decode bit for bit, checked on caller data: one
 * page's score product and output update on both instruction paths, with
 * bi_prefill_attention's descriptors and MMA forms and bi_decode_attention's
 * mma.sync steps (the same 16-deep steps over the same operands; operand
 * roles swapped).  "3. Batch-Invariant Attention" of "Defeating
 * Nondeterminism in LLM Inference: The Core Role of Batch Invariance" warns
 * that different tensor-core instructions may reduce in different orders;
 * this call lets a test confirm that, on the GPU at hand, these two do not.
 *   q   device, bf16 [128][128] (128 query columns)   k, v  bf16 [16][128]
 *   p   device, bf16 [128][16] (weights)                o0   fp32 [128][128]
 *   s_tc, s_mma   device, fp32 [128][16]: S = q . k^T, tcgen05 / mma.sync
 *   o_tc, o_mma   device, fp32 [128][128]: o0 + p . v, tcgen05 / mma.sync
 * Inputs 16-byte aligned.  One CTA; asynchronous on `stream`.
 */
bi_status bi_selftest_tcgen05_vs_mma_sync(const void* q, const void* k, const void* v,
                                          const void* p, const float* o0, float* s_tc,
                                          float* s_mma, float* o_tc, float* o_mma,
                                          cudaStream_t stream);

/* Workspace bytes bi_prefill_attention needs for T query rows of Hq heads of
 * size D when some row may attend over more than one 256-token chunk
 * (max_seq_len > 256): one fp32 D-vector per (row, head).  0 otherwise and for
 * invalid arguments. */
size_t bi_prefill_attention_workspace_size(int32_t T, int32_t Hq, int32_t D, int32_t max_seq_len);

/*
 * bi_qk_norm_rope_append -- the steps between the qkv projection and
 * attention, for T new tokens: per-head RMSNorm of q and k (when a weight is
 * given), rotary position embedding (rotate-half pairing of dims i and
 * 64 + i), q written out, k and v appended into the paged cache.
 *
 *   qkv        device, bf16 [T][ld_qkv]: per token Hq q-heads, then Hkv
 *              k-heads, then Hkv v-heads, 128 values each.
 *   positions  device, int32 [T]: each token's position (0 .. max_pos-1).
 *   slots      device, int32 [T]: each token's cache slot, page * 16 + offset.
 *   rope_table device, fp32 [max_pos][128]: cos(pos * f_i) at i and
 *              sin(pos * f_i) at 64 + i, i < 64 (f_i = theta^(-i/64)).
 *   q_norm_w, k_norm_w  device, bf16 [128], or null for no per-head norm.
 *   q_out      device, bf16 [T][Hq][128].
 *   k_cache, v_cache    as bi_decode_attention, num_pages pages.
 * Per head: x -> bf16(x * rsqrt(mean(x^2) + eps) * w) (fp32, sum of squares
 * in an order fixed by the head size) -> y_i = x_i c - x_{64+i} s,
 * y_{64+i} = x_{64+i} c + x_i s in fp32, rounded once to bf16.  Pointwise
 * and per-head, hence batch-invariant ("Achieving Batch-Invariant Kernels");
 * the append is the "3. Batch-Invariant Attention" rule that new tokens join
 * the one cache layout before attention reads it.  D = 128, page_size = 16.
 * A position or slot out of range is reported on the device
 * (BI_ERR_DEVICE_BAD_INPUT) and that token is skipped.
 */
bi_status bi_qk_norm_rope_append(const void* qkv, int64_t ld_qkv, int32_t T, int32_t Hq,
                                 int32_t Hkv, int32_t D, const int32_t* positions,
                                 const int32_t* slots, const float* rope_table, int32_t max_pos,
                                 const void* q_norm_w, const void* k_norm_w, float eps,
                                 void* q_out, void* k_cache, void* v_cache, int32_t num_pages,
                                 int32_t page_size, cudaStream_t stream);

/*
 * bi_silu_mul -- the SwiGLU product: out[t][j] = bf16(silu(g) * u) with
 * g = gate_up[t][j], u = gate_up[t][F + j], silu(g) = g / (1 + exp(-g)), all
 * in fp32 (exp(-g) as 2^(-g log2 e) by ex2.approx and the quotient as
 * g * rcp(1 + e) by rcp.approx: a few fp32 ulp, far inside bf16 rounding).
 * Pointwise, hence batch-invariant.  F a multiple of 8, at most
 * 2^30 (else BI_ERR_UNSUPPORTED_SHAPE).
 *   gate_up  device, bf16 [T][ld_gate_up] (gate columns 0..F-1, up F..2F-1).
 *   out      device, bf16 [T][ld_out].
 */
bi_status bi_silu_mul(const void* gate_up, int64_t ld_gate_up, int32_t T, int32_t F, void* out,
                      int64_t ld_out, cudaStream_t stream);

/*
 * bi_logprobs -- per-row log-sum-exp of bf16 logits and the log-probability
 * of one target token per row:
 *     lse[r] = log sum_j exp(x[r][j]),   logprob[r] = x[r][targets[r]] - lse[r]   (fp32)
 *
 * Operation: the sampler/trainer agreement that "Defeating Nondeterminism in
 * LLM Inference: The Core Role of Batch Invariance" ("Experimental Validation
 * and Future Prospects", true on-policy RL) needs: the softmax denominator is
 * a reduction over the vocabulary, computed one row per CTA in an order that
 * depends only on `vocab` (one pass: each thread folds its fixed stride of
 * 8-value vectors into a running max and sum of exp(x - max); then a warp
 * butterfly and a warp-ordered fold of those pairs), so a row's results are
 * bit-identical in any batch.  -inf logits (a masked vocabulary) add nothing.
 *   logits   device, bf16 [rows][ld], ld >= vocab, both multiples of 8.
 *   targets  device, int32 [rows] or null;  logprob_out  device, fp32 [rows]
 *            (needed with targets);  lse_out  device, fp32 [rows] or null.
 * A target outside 0 .. vocab-1 gives NaN and BI_ERR_DEVICE_BAD_INPUT.
 */
bi_status bi_logprobs(const void* logits, int64_t rows, int32_t vocab, int64_t ld,
                      const int32_t* targets, float* logprob_out, float* lse_out,
                      cudaStream_t stream);

/*
 * bi_decode_attention_fixed_splits -- the same attention with a fixed split
 * COUNT instead of a fixed split size: each sequence's pages are cut into
 * num_splits nearly equal runs (ceil(ceil(L/16)/num_splits) pages each), so
 * the chunk size -- and the reduction order -- changes as the sequence grows.
 * This is the strategy "Defeating Nondeterminism in LLM Inference: The Core
 * Role of Batch Invariance" warns against (section "3. Batch-Invariant
 * Attention", figure "Fixed Number Split KV Strategy"); it is NOT batch- or
 * growth-invariant and exists only as the non-invariant comparison: a
 * negative control for the growth tests and a same-run cost reference.
 *   num_splits   1 .. ; ceil(ceil(max_seq_len/16)/num_splits) <= 512 pages.
 *   workspace    >= bi_decode_attention_workspace_size(B, Hq, D,
 *                num_splits * 256) bytes when num_splits >= 2.
 * Other arguments and errors: as bi_decode_attention.
 */
bi_status bi_decode_attention_fixed_splits(const void* q, const void* k_cache,
                                           const void* v_cache, const int32_t* block_table,
                                           int32_t max_pages_per_seq, const int32_t* seq_lens,
                                           int32_t B, int32_t Hq, int32_t Hkv, int32_t D,
                                           int32_t page_size, int32_t num_pages,
                                           int32_t max_seq_len, float scale, int32_t num_splits,
                                           void* out, void* workspace, size_t workspace_bytes,
                                           cudaStream_t stream);

/* Kernel launches one bi_decode_attention call makes on the current device:
 * 1 whenever B * Hkv <= BI_DECODE_COUNTER_BYTES / 4 (each sequence is folded
 * by its own CTA or by the last of its CTAs to arrive), else 2 when some
 * sequence spans several CTAs (the separate merge kernel folds it).  A
 * schedule detail -- the results are the same bits either way.  0 for
 * invalid arguments or when no device is available. */
int32_t bi_decode_attention_launches(int32_t B, int32_t Hkv, int32_t max_seq_len);

/*
 * bi_decode_attention_noalloc -- bi_decode_attention for callers that cannot
 * allocate device memory when they call it.
 *
 * Some callers have no way to obtain a workspace: a plugin handed only its
 * input and output buffers by a host framework, a serving loop whose device
 * memory was all reserved up front by a caching allocator (so a fresh
 * cudaMalloc would fail, or would synchronise the device mid-step), or code
 * that must not trigger allocation at all.  This entry point takes the same
 * arguments minus the workspace and computes exactly what bi_decode_attention
 * computes -- same kernels, same reduction order, bit-identical output --
 * keeping the chunk partials in a scratch array that is part of the library's
 * device image instead.  The pages this library follows describe no such
 * entry point; it exists only for those callers.
 *
 * Limits and behaviour:
 *   - the scratch holds 65536 chunk partials: when max_seq_len > 256,
 *     B * Hq * ceil(max_seq_len/256) must not exceed 65536 (for example 64
 *     sequences of 32 heads up to 8192 tokens, or 256 sequences of 32 heads
 *     up to 2048 tokens); larger calls return BI_ERR_WORKSPACE_TOO_SMALL and
 *     launch nothing.  With max_seq_len <= 256 nothing is written to the
 *     scratch and any B up to 65535 is accepted.
 *   - the array takes 32.75 MiB of device memory on every GPU that loads the
 *     library, for as long as the library stays loaded.
 *   - nothing is allocated or freed: no cudaMalloc, no cudaFree, no library
 *     allocator.  The first call on each device that needs the scratch looks
 *     up the array's device address (cudaGetSymbolAddress) and caches it for
 *     the life of the process; make that first call before any stream
 *     capture (made during a capture, it returns BI_ERR_CUDA).  A
 *     cudaDeviceReset discards the array and the cached address with it:
 *     do not call this entry point on a device after resetting it.
 *   - every call on a device shares the one array: its arrival counters
 *     start at zero when the library loads and every call leaves them zero;
 *     the partials keep the last call's values and need no clearing.  Calls
 *     whose kernels may overlap on the GPU (different streams, without
 *     ordering between them) race on it and must be serialised by the
 *     caller.
 * Other arguments, errors and device-side checks: as bi_decode_attention.
 */
bi_status bi_decode_attention_noalloc(const void* q, const void* k_cache, const void* v_cache,
                                      const int32_t* block_table, int32_t max_pages_per_seq,
                                      const int32_t* seq_lens, int32_t B, int32_t Hq,
                                      int32_t Hkv, int32_t D, int32_t page_size,
                                      int32_t num_pages, int32_t max_seq_len, float scale,
                                      void* out, cudaStream_t stream);

#ifdef __cplusplus
}
#endif

#endif /* BI_H_ */
