/*
 * Plain fp64 CPU oracle for the batch-invariant forward kernels.
 *
 * TEST INFRASTRUCTURE ONLY.  Nothing in the product path links, loads or
 * calls this file; only the tests, the smoke check and the CPU-baseline leg
 * of the benchmark do.  It shares no code, header, table or constant with
 * the CUDA library.
 *
 * Every routine computes the plain mathematical definition of its operation
 * in double precision, in the most obvious loop order, with no blocking,
 * chunking or reordering.  bf16 inputs arrive as raw 16-bit patterns and are
 * widened exactly; results are returned as doubles, and oracle_round_bf16
 * rounds them once, to nearest-even, when a caller wants the bf16 value the
 * definition rounds to.
 *
 * Sources (web pages on the batch-invariance method):
 *  - "Thinking Machines Lab - Defeating Nondeterminism in LLM Inference: The
 *    Core Role of Batch Invariance", sections "1. Batch-Invariant RMSNorm",
 *    "2. Batch-Invariant Matrix Multiplication", "3. Batch-Invariant
 *    Attention".
 *  - "Batch Invariance and Numerical Reproducibility", the answer on fixed
 *    split counts versus fixed split sizes (1000 = 3 x 256 + 232).
 *
 * Build: gcc -O2 -fno-fast-math -ffp-contract=off [-fopenmp] -shared -fPIC.
 * With OpenMP the loops over independent rows / outputs run in parallel; the
 * arithmetic of each output is unchanged by that.
 */
#include <math.h>
#include <stdint.h>
#include <string.h>

#ifdef _OPENMP
#include <omp.h>
#endif

/* ---- bf16 <-> double, written from the bit layouts -------------------- */

/* bf16 is the top half of an IEEE binary32: 1 sign, 8 exponent, 7 fraction
 * bits.  Widening is exact: shift into a float's high half, then to double. */
static double bf16_to_double(uint16_t h) {
    uint32_t u = ((uint32_t)h) << 16;
    float f;
    memcpy(&f, &u, sizeof f);
    return (double)f;
}

/* Round a double straight to the nearest bf16, ties to even, with no
 * intermediate float (which would round twice).
 *
 * A finite nonzero double is sig * 2^(e - 1075) with sig the 53-bit
 * significand including the hidden bit.  The bf16 grid spacing (quantum) at
 * unbiased exponent x = e - 1023 is 2^(x - 7) for normals and 2^-133 below the
 * normal range.  The result is q * quantum with q = round(sig * 2^-shift).
 * Because bf16 encodings are monotone in magnitude, (E << 7) + (q - 128)
 * is the encoding of a normal result even when rounding carries into the
 * next binade, and q itself is the encoding of a subnormal (q == 128 lands
 * exactly on the smallest normal, 0x0080). */
static uint16_t double_to_bf16_rne(double d) {
    uint64_t u;
    memcpy(&u, &d, sizeof u);
    uint16_t sign = (uint16_t)((u >> 48) & 0x8000u);
    uint64_t a = u & 0x7fffffffffffffffull;
    if (a > 0x7ff0000000000000ull) return (uint16_t)(sign | 0x7fc0u); /* NaN */
    if (a == 0x7ff0000000000000ull) return (uint16_t)(sign | 0x7f80u); /* inf */
    int e = (int)(a >> 52);
    if (e == 0) return sign; /* double subnormals are far below 2^-134 */
    uint64_t sig = (a & 0x000fffffffffffffull) | 0x0010000000000000ull;
    int x = e - 1023;
    int qe = (x - 7 > -133) ? x - 7 : -133;
    int shift = qe - (e - 1075); /* >= 45 */
    if (shift >= 64) return sign;
    uint64_t q = sig >> shift;
    uint64_t rem = sig & ((1ull << shift) - 1ull);
    uint64_t half = 1ull << (shift - 1);
    if (rem > half || (rem == half && (q & 1ull))) q += 1ull;
    uint32_t bits;
    if (qe == -133) {
        bits = (uint32_t)q;
    } else {
        uint32_t E = (uint32_t)(x + 127);
        bits = (E << 7) + (uint32_t)(q - 128u);
    }
    if (bits >= 0x7f80u) bits = 0x7f80u; /* overflow to infinity */
    return (uint16_t)(sign | bits);
}

void oracle_round_bf16(const double* in, uint16_t* out, int64_t n) {
    for (int64_t i = 0; i < n; ++i) out[i] = double_to_bf16_rne(in[i]);
}

void oracle_bf16_to_double(const uint16_t* in, double* out, int64_t n) {
    for (int64_t i = 0; i < n; ++i) out[i] = bf16_to_double(in[i]);
}

int oracle_num_threads(void) {
#ifdef _OPENMP
    return omp_get_max_threads();
#else
    return 1;
#endif
}

/* ---- RMSNorm ----------------------------------------------------------
 * "1. Batch-Invariant RMSNorm": each row is normalised by the root mean
 * square of its own elements, then scaled elementwise by the weight:
 *     y[r][i] = x[r][i] * w[i] / sqrt( (1/H) * sum_j x[r][j]^2 + eps ).
 * The reduction is over one row only; other rows never enter it. */
int oracle_rmsnorm(const uint16_t* x, const uint16_t* w, int64_t rows,
                   int32_t hidden, double eps, double* y) {
    if (rows < 0 || hidden <= 0) return -1;
#pragma omp parallel for schedule(static)
    for (int64_t r = 0; r < rows; ++r) {
        const uint16_t* xr = x + r * (int64_t)hidden;
        double sumsq = 0.0;
        for (int32_t j = 0; j < hidden; ++j) {
            double v = bf16_to_double(xr[j]);
            sumsq += v * v;
        }
        double denom = sqrt(sumsq / (double)hidden + eps);
        for (int32_t i = 0; i < hidden; ++i)
            y[r * (int64_t)hidden + i] =
                bf16_to_double(xr[i]) * bf16_to_double(w[i]) / denom;
    }
    return 0;
}

/* ---- GEMM -------------------------------------------------------------
 * "2. Batch-Invariant Matrix Multiplication": y = x * W^T with x [M, K]
 * (row-major) and W [N, K] (row-major, the nn.Linear layout), so
 *     y[m][n] = sum_k x[m][k] * W[n][k].
 * Every product of two bf16 values is exact in double. */
int oracle_gemm(const uint16_t* x, const uint16_t* W, int32_t M, int32_t N,
                int32_t K, double* y) {
    if (M < 0 || N < 0 || K < 0) return -1;
#pragma omp parallel for collapse(2) schedule(static)
    for (int64_t m = 0; m < M; ++m) {
        for (int32_t n = 0; n < N; ++n) {
            double acc = 0.0;
            for (int32_t k = 0; k < K; ++k)
                acc += bf16_to_double(x[m * (int64_t)K + k]) *
                       bf16_to_double(W[(int64_t)n * K + k]);
            y[m * (int64_t)N + n] = acc;
        }
    }
    return 0;
}

/* The same dot product at a list of (m, n) positions, for shapes too large
 * to evaluate in full: y[i] = sum_k x[mi][k] * W[ni][k]. */
int oracle_gemm_entries(const uint16_t* x, const uint16_t* W, int32_t M,
                        int32_t N, int32_t K, const int32_t* ms,
                        const int32_t* ns, int64_t count, double* y) {
#pragma omp parallel for schedule(static)
    for (int64_t i = 0; i < count; ++i) {
        int32_t m = ms[i], n = ns[i];
        if (m < 0 || m >= M || n < 0 || n >= N) {
            y[i] = NAN;
            continue;
        }
        double acc = 0.0;
        for (int32_t k = 0; k < K; ++k)
            acc += bf16_to_double(x[(int64_t)m * K + k]) *
                   bf16_to_double(W[(int64_t)n * K + k]);
        y[i] = acc;
    }
    return 0;
}

/* ---- decode attention over a paged KV cache ----------------------------
 * "3. Batch-Invariant Attention": one query row per sequence attends over
 * every cached key of that sequence.  For sequence s, query head i and its
 * key/value head g = i / (Hq / Hkv):
 *     score_t = scale * sum_d q[s][i][d] * k_t[g][d],   t = 0 .. L_s - 1
 *     p_t     = exp(score_t - max_t score_t) / sum_t exp(...)
 *     out[s][i][d] = sum_t p_t * v_t[g][d]
 * Token t of sequence s lives in page block_table[s][t / page_size] at slot
 * t % page_size.  The cache layout is [num_pages][Hkv][page_size][D].
 * No chunking: this is the definition the chunked method must reproduce. */
static const uint16_t* kv_row(const uint16_t* cache, const int32_t* bt_row,
                              int32_t t, int32_t g, int32_t Hkv,
                              int32_t page_size, int32_t D) {
    int64_t page = bt_row[t / page_size];
    int64_t slot = t % page_size;
    return cache + (((page * Hkv + g) * page_size + slot) * (int64_t)D);
}

int oracle_decode_attention(const uint16_t* q, const uint16_t* k_cache,
                            const uint16_t* v_cache, const int32_t* block_table,
                            int32_t max_pages_per_seq, const int32_t* seq_lens,
                            int32_t B, int32_t Hq, int32_t Hkv, int32_t D,
                            int32_t page_size, double scale, double* out) {
    if (B < 0 || Hq <= 0 || Hkv <= 0 || D <= 0 || page_size <= 0) return -1;
    if (Hq % Hkv != 0) return -1;
    const int32_t group = Hq / Hkv;
    int bad = 0;
#pragma omp parallel for schedule(dynamic) reduction(| : bad)
    for (int64_t si = 0; si < (int64_t)B * Hq; ++si) {
        int32_t s = (int32_t)(si / Hq), i = (int32_t)(si % Hq);
        int32_t g = i / group;
        int32_t L = seq_lens[s];
        const int32_t* bt_row = block_table + (int64_t)s * max_pages_per_seq;
        const uint16_t* qi = q + ((int64_t)s * Hq + i) * D;
        double* o = out + ((int64_t)s * Hq + i) * D;
        if (L <= 0 || (L + page_size - 1) / page_size > max_pages_per_seq) {
            for (int32_t d = 0; d < D; ++d) o[d] = NAN;
            bad = 1;
            continue;
        }
        double mx = -INFINITY;
        for (int32_t t = 0; t < L; ++t) {
            const uint16_t* kt = kv_row(k_cache, bt_row, t, g, Hkv, page_size, D);
            double sc = 0.0;
            for (int32_t d = 0; d < D; ++d)
                sc += bf16_to_double(qi[d]) * bf16_to_double(kt[d]);
            sc *= scale;
            if (sc > mx) mx = sc;
        }
        double denom = 0.0;
        for (int32_t d = 0; d < D; ++d) o[d] = 0.0;
        for (int32_t t = 0; t < L; ++t) {
            const uint16_t* kt = kv_row(k_cache, bt_row, t, g, Hkv, page_size, D);
            const uint16_t* vt = kv_row(v_cache, bt_row, t, g, Hkv, page_size, D);
            double sc = 0.0;
            for (int32_t d = 0; d < D; ++d)
                sc += bf16_to_double(qi[d]) * bf16_to_double(kt[d]);
            double p = exp(sc * scale - mx);
            denom += p;
            for (int32_t d = 0; d < D; ++d) o[d] += p * bf16_to_double(vt[d]);
        }
        for (int32_t d = 0; d < D; ++d) o[d] /= denom;
    }
    return bad ? -2 : 0;
}

/* The fixed split-size form of the same computation, in fp64, following the
 * steps "3. Batch-Invariant Attention" and "Batch Invariance and Numerical
 * Reproducibility" describe: the keys of a sequence are cut into consecutive
 * chunks of exactly `chunk` tokens (the last one shorter), each chunk yields
 * a partial (running max m_c, sum of exponentials l_c, unnormalised output
 * a_c), and the partials are folded in ascending chunk order with the
 * log-sum-exp rule
 *     M' = max(M, m_c),  L' = L e^(M - M') + l_c e^(m_c - M'),
 *     A' = A e^(M - M') + a_c e^(m_c - M'),
 * and out = A / L at the end.  Algebraically this equals the unchunked
 * definition above; the tests check that it does to fp64 rounding.
 * When `partials` is non-null it receives, per (s, i, c) for c < nchunks(L_s),
 * the triple (m_c, l_c, a_c[0..D-1]) in a [B][Hq][max_chunks][D + 2] array. */
int oracle_decode_attention_chunked(
    const uint16_t* q, const uint16_t* k_cache, const uint16_t* v_cache,
    const int32_t* block_table, int32_t max_pages_per_seq,
    const int32_t* seq_lens, int32_t B, int32_t Hq, int32_t Hkv, int32_t D,
    int32_t page_size, double scale, int32_t chunk, int32_t max_chunks,
    double* out, double* partials) {
    if (B < 0 || Hq <= 0 || Hkv <= 0 || D <= 0 || page_size <= 0 || chunk <= 0)
        return -1;
    if (Hq % Hkv != 0) return -1;
    const int32_t group = Hq / Hkv;
    int bad = 0;
#pragma omp parallel for schedule(dynamic) reduction(| : bad)
    for (int64_t si = 0; si < (int64_t)B * Hq; ++si) {
        int32_t s = (int32_t)(si / Hq), i = (int32_t)(si % Hq);
        int32_t g = i / group;
        int32_t L = seq_lens[s];
        const int32_t* bt_row = block_table + (int64_t)s * max_pages_per_seq;
        const uint16_t* qi = q + ((int64_t)s * Hq + i) * D;
        double* o = out + ((int64_t)s * Hq + i) * D;
        int32_t nch = (L + chunk - 1) / chunk;
        if (L <= 0 || (L + page_size - 1) / page_size > max_pages_per_seq ||
            (partials && nch > max_chunks)) {
            for (int32_t d = 0; d < D; ++d) o[d] = NAN;
            bad = 1;
            continue;
        }
        double Mrun = -INFINITY, Lrun = 0.0;
        for (int32_t d = 0; d < D; ++d) o[d] = 0.0;
        for (int32_t c = 0; c < nch; ++c) {
            int32_t t0 = c * chunk;
            int32_t t1 = (t0 + chunk < L) ? t0 + chunk : L;
            /* partial over this chunk alone */
            double m = -INFINITY;
            for (int32_t t = t0; t < t1; ++t) {
                const uint16_t* kt = kv_row(k_cache, bt_row, t, g, Hkv, page_size, D);
                double sc = 0.0;
                for (int32_t d = 0; d < D; ++d)
                    sc += bf16_to_double(qi[d]) * bf16_to_double(kt[d]);
                sc *= scale;
                if (sc > m) m = sc;
            }
            double l = 0.0;
            double a[1024];
            if (D > 1024) { bad = 1; break; }
            for (int32_t d = 0; d < D; ++d) a[d] = 0.0;
            for (int32_t t = t0; t < t1; ++t) {
                const uint16_t* kt = kv_row(k_cache, bt_row, t, g, Hkv, page_size, D);
                const uint16_t* vt = kv_row(v_cache, bt_row, t, g, Hkv, page_size, D);
                double sc = 0.0;
                for (int32_t d = 0; d < D; ++d)
                    sc += bf16_to_double(qi[d]) * bf16_to_double(kt[d]);
                double p = exp(sc * scale - m);
                l += p;
                for (int32_t d = 0; d < D; ++d) a[d] += p * bf16_to_double(vt[d]);
            }
            if (partials) {
                double* pp = partials +
                             (((int64_t)s * Hq + i) * max_chunks + c) * (D + 2);
                pp[0] = m;
                pp[1] = l;
                for (int32_t d = 0; d < D; ++d) pp[2 + d] = a[d];
            }
            /* fold into the running state, ascending chunk order */
            double Mnew = (m > Mrun) ? m : Mrun;
            double fo = exp(Mrun - Mnew); /* exp(-inf) = 0 on the first chunk */
            double fc = exp(m - Mnew);
            Lrun = Lrun * fo + l * fc;
            for (int32_t d = 0; d < D; ++d) o[d] = o[d] * fo + a[d] * fc;
            Mrun = Mnew;
        }
        for (int32_t d = 0; d < D; ++d) o[d] /= Lrun;
    }
    return bad ? -2 : 0;
}

/* ---- log-probabilities ---------------------------------------------------
 * "Experimental Validation and Future Prospects" (true on-policy RL): the
 * log-probability of a token under the softmax of a logits row,
 *     lse = log sum_j exp(x_j),   logprob(t) = x_t - lse,
 * evaluated as m + log(sum_j exp(x_j - m)) with m = max_j x_j. */
int oracle_logprobs(const uint16_t* logits, int64_t rows, int32_t vocab,
                    const int32_t* targets, double* logprob, double* lse) {
    if (rows < 0 || vocab <= 0) return -1;
    int bad = 0;
#pragma omp parallel for schedule(static) reduction(| : bad)
    for (int64_t r = 0; r < rows; ++r) {
        const uint16_t* x = logits + r * (int64_t)vocab;
        double m = -INFINITY;
        for (int32_t j = 0; j < vocab; ++j) {
            double v = bf16_to_double(x[j]);
            if (v > m) m = v;
        }
        double s = 0.0;
        for (int32_t j = 0; j < vocab; ++j) s += exp(bf16_to_double(x[j]) - m);
        double l = m + log(s);
        if (lse) lse[r] = l;
        if (targets && logprob) {
            int32_t t = targets[r];
            if (t < 0 || t >= vocab) {
                logprob[r] = NAN;
                bad = 1;
            } else {
                logprob[r] = bf16_to_double(x[t]) - l;
            }
        }
    }
    return bad ? -2 : 0;
}
