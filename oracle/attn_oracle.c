/*
 * Oracle for fused scaled-dot-product attention -- TEST INFRASTRUCTURE ONLY.
 *
 * Only tests/, the smoke check in __graft_entry__.py and the cpu_baseline /
 * reference legs of bench.py may load this code.  The product path (the CUDA
 * library under attention_online_softmax_gb300/) never links, loads or calls it,
 * and this file shares no code, header or table with that library.
 *
 * What it computes is the plain two-pass definition of attention, in double
 * precision, one query row at a time:
 *
 *   "Compilers and Kernels", section "FlashAttention changes the algorithm
 *   around IO", first display equation and the one after it:
 *       S = Q K^T / sqrt(d) + C,   m_i = max_j S_ij,
 *       l_i = sum_j exp(S_ij - m_i),   P_ij = exp(S_ij - m_i) / l_i,   O = P V.
 *   The additive mask C takes the values 0 (key allowed) or -inf (key
 *   disallowed); a disallowed key is simply left out of the max and the sum.
 *
 *   "Don't Write Kernels, Derive Them", section "What happened": logsumexp is
 *   one of the derived operations.  The row logsumexp of the scaled, masked
 *   scores is  LSE_i = m_i + ln(l_i).
 *
 * Readings where the pages are silent (each one is listed with its reason in
 * the design notes of the repository):
 *   - scale: the caller passes the float it wants (1/sqrt(d) in every workload);
 *     it is widened to double unchanged, so the oracle and the GPU use the same
 *     number.
 *   - causal alignment for Nq != Nk is bottom-right: key j is allowed for query
 *     i iff j <= i + (Nk - Nq).  For Nq == Nk this is "query i attends keys
 *     0..i".
 *   - grouped-query attention: query head h reads key/value head
 *     h / (Hq / Hkv) (consecutive groups).
 *   - a row with no allowed key (the page assumes there is none) is defined as
 *     O = 0 and LSE = -inf.
 *   - inputs arrive as bfloat16 bit patterns; each is widened exactly to double.
 *
 * Paged decode is the same definition with one query row per sequence, over
 * all seqlens[s] cached tokens, where token t of sequence s sits in page
 * block_table[s][t / page_size], slot t % page_size, of a cache laid out as
 * [num_pages][page_size][Hkv][d].
 *
 * The test-suite builds copies of this file with one deliberate mistake
 * planted (tests/oracle_mutants.py) to show that its pins catch each kind of
 * mistake; this file itself holds none.
 */
#include <math.h>
#include <stdint.h>
#include <stdlib.h>
#include <string.h>
#ifdef _OPENMP
#include <omp.h>
#endif

/* bfloat16 is the upper half of an IEEE binary32; widening is exact. */
static double bf16_to_double(uint16_t bits) {
    uint32_t w = ((uint32_t)bits) << 16;
    float f;
    memcpy(&f, &w, sizeof f);
    return (double)f;
}

/*
 * One query row against n_keys keys.
 *   q:  d values (bf16 bits), kv rows fetched through key_row()/val_row().
 *   Writes d_v doubles to o and returns the row LSE through *lse.
 * The key/value rows are given as arrays of row pointers so that the same
 * routine serves contiguous prefill and paged decode.
 */
static void attend_row(const uint16_t* q, const uint16_t* const* krows,
                       const uint16_t* const* vrows, int64_t n_keys, int d,
                       double scale, double* scratch, double* o, double* lse) {
    int64_t j;
    int c;
    if (n_keys <= 0) {
        for (c = 0; c < d; ++c) o[c] = 0.0;
        *lse = -INFINITY;
        return;
    }
    /* pass 1: scores and their maximum */
    double m = -INFINITY;
    for (j = 0; j < n_keys; ++j) {
        double s = 0.0;
        for (c = 0; c < d; ++c) {
            s += bf16_to_double(q[c]) * bf16_to_double(krows[j][c]);
        }
        s *= scale;
        scratch[j] = s;
        if (s > m) m = s;
    }
    /* pass 2: normaliser and the weighted sum of value rows */
    double l = 0.0;
    for (c = 0; c < d; ++c) o[c] = 0.0;
    for (j = 0; j < n_keys; ++j) {
        double p = exp(scratch[j] - m);
        l += p;
        for (c = 0; c < d; ++c) o[c] += p * bf16_to_double(vrows[j][c]);
    }
    for (c = 0; c < d; ++c) o[c] /= l;
    *lse = m + log(l);
}

static int oracle_threads(int nthreads) {
#ifdef _OPENMP
    if (nthreads <= 0) nthreads = omp_get_max_threads();
#else
    nthreads = 1;
#endif
    return nthreads;
}

/*
 * Additive bias C of the attention definition, beyond the causal mask:
 *   window_left > 0: key j is allowed for query i only if
 *                    j > i + (Nk - Nq) - window_left;
 *   alibi (may be NULL): adds alibi[h] * (j - i - (Nk - Nq)) to S_ij;
 *   bias (may be NULL): bf16 bits, adds bias[b*sb + h*sh + i*Nk + j] to S_ij
 *                       (-inf disallows the key).
 * A key the mask disallows is left out; a row with no allowed key (or whose
 * every allowed score is -inf) has O = 0 and LSE = -inf.
 */
static void attend_row_biased(const uint16_t* q, const uint16_t* const* krows,
                              const uint16_t* const* vrows, int64_t n_keys, int d, double scale,
                              const double* cbias, double* scratch, double* o, double* lse) {
    int64_t j;
    int c;
    double m = -INFINITY;
    for (j = 0; j < n_keys; ++j) {
        double s = 0.0;
        for (c = 0; c < d; ++c) s += bf16_to_double(q[c]) * bf16_to_double(krows[j][c]);
        s = s * scale + cbias[j];
        scratch[j] = s;
        if (s > m) m = s;
    }
    for (c = 0; c < d; ++c) o[c] = 0.0;
    if (m == -INFINITY) {
        *lse = -INFINITY;
        return;
    }
    double l = 0.0;
    for (j = 0; j < n_keys; ++j) {
        double p = exp(scratch[j] - m);
        l += p;
        for (c = 0; c < d; ++c) o[c] += p * bf16_to_double(vrows[j][c]);
    }
    for (c = 0; c < d; ++c) o[c] /= l;
    *lse = m + log(l);
}

int oracle_attention_masked(const uint16_t* q, const uint16_t* k, const uint16_t* v,
                            int B, int Hq, int Hkv, int Nq, int Nk, int d, int causal,
                            float scale, int window_left, const float* alibi,
                            const uint16_t* bias, int64_t bias_sb, int64_t bias_sh,
                            const int64_t* rows, int64_t nrows,
                            double* o_out, double* lse_out, int nthreads) {
    if (B < 0 || Hq <= 0 || Hkv <= 0 || Nq < 0 || Nk < 0 || d <= 0 || window_left < 0) return -1;
    if (Hq % Hkv != 0) return -1;
    const int group = Hq / Hkv;
    const int64_t total = (int64_t)B * Hq * Nq;
    if (rows == NULL) nrows = total;
    nthreads = oracle_threads(nthreads);
    int bad = 0;
#pragma omp parallel num_threads(nthreads)
    {
        const size_t cap = (size_t)(Nk > 0 ? Nk : 1);
        double* scratch = (double*)malloc(sizeof(double) * cap);
        double* cb = (double*)malloc(sizeof(double) * cap);
        const uint16_t** krows = (const uint16_t**)malloc(sizeof(void*) * cap);
        const uint16_t** vrows = (const uint16_t**)malloc(sizeof(void*) * cap);
        int64_t r;
#pragma omp for schedule(dynamic, 4)
        for (r = 0; r < nrows; ++r) {
            int64_t flat = rows ? rows[r] : r;
            if (flat < 0 || flat >= total) {
#pragma omp atomic write
                bad = 1;
                continue;
            }
            int64_t i = flat % Nq;
            int64_t bh = flat / Nq;
            int64_t h = bh % Hq;
            int64_t b = bh / Hq;
            int64_t g = h / group;
            int64_t diag = (int64_t)Nk - (int64_t)Nq;
            const uint16_t* kb = k + ((b * Hkv + g) * (int64_t)Nk) * d;
            const uint16_t* vb = v + ((b * Hkv + g) * (int64_t)Nk) * d;
            int64_t n = 0, j;
            for (j = 0; j < Nk; ++j) {
                if (causal && j > i + diag) continue;
                if (window_left > 0 && j <= i + diag - window_left) continue;
                double c = 0.0;
                if (alibi) c += (double)alibi[h] * (double)(j - i - diag);
                if (bias) c += bf16_to_double(bias[b * bias_sb + h * bias_sh + i * (int64_t)Nk + j]);
                krows[n] = kb + j * d;
                vrows[n] = vb + j * d;
                cb[n] = c;
                ++n;
            }
            attend_row_biased(q + flat * d, krows, vrows, n, d, (double)scale, cb, scratch,
                              o_out + r * d, lse_out + r);
        }
        free(scratch);
        free(cb);
        free(krows);
        free(vrows);
    }
    return bad ? -2 : nthreads;
}

/*
 * Prefill / general attention.
 *   q: [B][Hq][Nq][d], k and v: [B][Hkv][Nk][d], all bf16 bits, contiguous.
 *   rows: flat query-row ids ((b*Hq + h)*Nq + i), or NULL for every row in
 *   order; nrows: their count.
 *   o_out: [nrows][d] doubles, lse_out: [nrows] doubles.
 *   nthreads <= 0 uses every core OpenMP offers.
 * Returns the number of threads used, or a negative value on a bad argument.
 */
int oracle_attention(const uint16_t* q, const uint16_t* k, const uint16_t* v,
                     int B, int Hq, int Hkv, int Nq, int Nk, int d, int causal,
                     float scale, const int64_t* rows, int64_t nrows,
                     double* o_out, double* lse_out, int nthreads) {
    if (B < 0 || Hq <= 0 || Hkv <= 0 || Nq < 0 || Nk < 0 || d <= 0) return -1;
    if (Hq % Hkv != 0) return -1;
    const int group = Hq / Hkv;
    const int64_t total = (int64_t)B * Hq * Nq;
    if (rows == NULL) nrows = total;
    nthreads = oracle_threads(nthreads);
    int bad = 0;

#pragma omp parallel num_threads(nthreads)
    {
        double* scratch = (double*)malloc(sizeof(double) * (size_t)(Nk > 0 ? Nk : 1));
        const uint16_t** krows = (const uint16_t**)malloc(sizeof(void*) * (size_t)(Nk > 0 ? Nk : 1));
        const uint16_t** vrows = (const uint16_t**)malloc(sizeof(void*) * (size_t)(Nk > 0 ? Nk : 1));
        int64_t r;
#pragma omp for schedule(dynamic, 4)
        for (r = 0; r < nrows; ++r) {
            int64_t flat = rows ? rows[r] : r;
            if (flat < 0 || flat >= total) {
#pragma omp atomic write
                bad = 1;
                continue;
            }
            int64_t i = flat % Nq;
            int64_t bh = flat / Nq;
            int64_t h = bh % Hq;
            int64_t b = bh / Hq;
            int64_t g = h / group;
            int64_t n_allowed = Nk;
            if (causal) {
                int64_t last = i + (int64_t)Nk - (int64_t)Nq;
                n_allowed = last + 1;
                if (n_allowed < 0) n_allowed = 0;
                if (n_allowed > Nk) n_allowed = Nk;
            }
            const uint16_t* kb = k + ((b * Hkv + g) * (int64_t)Nk) * d;
            const uint16_t* vb = v + ((b * Hkv + g) * (int64_t)Nk) * d;
            int64_t j;
            for (j = 0; j < n_allowed; ++j) {
                krows[j] = kb + j * d;
                vrows[j] = vb + j * d;
            }
            attend_row(q + flat * d, krows, vrows, n_allowed, d, (double)scale,
                       scratch, o_out + r * d, lse_out + r);
        }
        free(scratch);
        free(krows);
        free(vrows);
    }
    return bad ? -2 : nthreads;
}

/*
 * Paged decode: one query row per sequence and query head.
 *   q: [num_seqs][Hq][d]; kcache, vcache: [num_pages][page_size][Hkv][d];
 *   block_table: [num_seqs][max_pages_per_seq] int32; seqlens: [num_seqs].
 *   seqs: sequence ids to evaluate (NULL = all, in order), nseqs their count.
 *   o_out: [nseqs][Hq][d] doubles, lse_out: [nseqs][Hq] doubles.
 * Returns threads used, or a negative value when an argument or a block-table
 * entry is out of range.
 */
int oracle_decode_paged(const uint16_t* q, const uint16_t* kcache, const uint16_t* vcache,
                        const int32_t* block_table, const int32_t* seqlens,
                        int num_seqs, int Hq, int Hkv, int d, int page_size,
                        int num_pages, int max_pages_per_seq, float scale,
                        const int32_t* seqs, int nseqs,
                        double* o_out, double* lse_out, int nthreads) {
    if (num_seqs < 0 || Hq <= 0 || Hkv <= 0 || d <= 0 || page_size <= 0) return -1;
    if (Hq % Hkv != 0) return -1;
    const int group = Hq / Hkv;
    if (seqs == NULL) nseqs = num_seqs;
    int64_t max_len = 0;
    int s;
    for (s = 0; s < num_seqs; ++s) {
        if (seqlens[s] < 0 || (int64_t)seqlens[s] > (int64_t)max_pages_per_seq * page_size) return -1;
        if (seqlens[s] > max_len) max_len = seqlens[s];
    }
    nthreads = oracle_threads(nthreads);
    const int64_t work = (int64_t)nseqs * Hq;
    int bad = 0;

#pragma omp parallel num_threads(nthreads)
    {
        double* scratch = (double*)malloc(sizeof(double) * (size_t)(max_len > 0 ? max_len : 1));
        const uint16_t** krows = (const uint16_t**)malloc(sizeof(void*) * (size_t)(max_len > 0 ? max_len : 1));
        const uint16_t** vrows = (const uint16_t**)malloc(sizeof(void*) * (size_t)(max_len > 0 ? max_len : 1));
        int64_t w;
#pragma omp for schedule(dynamic, 1)
        for (w = 0; w < work; ++w) {
            int si = (int)(w / Hq);
            int h = (int)(w % Hq);
            int seq = seqs ? seqs[si] : si;
            if (seq < 0 || seq >= num_seqs) {
#pragma omp atomic write
                bad = 1;
                continue;
            }
            int g = h / group;
            int64_t n = seqlens[seq];
            int64_t t;
            int ok = 1;
            for (t = 0; t < n; ++t) {
                int32_t page = block_table[(int64_t)seq * max_pages_per_seq + t / page_size];
                if (page < 0 || page >= num_pages) { ok = 0; break; }
                int64_t off = (((int64_t)page * page_size + t % page_size) * Hkv + g) * d;
                krows[t] = kcache + off;
                vrows[t] = vcache + off;
            }
            if (!ok) {
#pragma omp atomic write
                bad = 1;
                continue;
            }
            attend_row(q + ((int64_t)seq * Hq + h) * d, krows, vrows, n, d, (double)scale,
                       scratch, o_out + w * d, lse_out + w);
        }
        free(scratch);
        free(krows);
        free(vrows);
    }
    return bad ? -2 : nthreads;
}

/*
 * Chunked prefill against a paged KV cache, ragged over sequences.
 *
 * "Don't Write Kernels, Derive Them", section "What happened": paged KV-cache
 * access is one of the operations the method covers; "Compilers and Kernels",
 * section "FlashAttention changes the algorithm around IO", gives the
 * attention each query row computes (the definition above).
 *
 * Sequence s owns query tokens [cu_seqlens_q[s], cu_seqlens_q[s+1]) of the
 * packed q [total_q][Hq][d]; they are the LAST q_len = cu_seqlens_q[s+1] -
 * cu_seqlens_q[s] tokens of its context of k_len = seqlens_k[s] tokens, whose
 * keys and values sit in the paged cache exactly as for paged decode.  Query i
 * of the chunk (0 <= i < q_len) sees keys j in [lo, hi):
 *     hi = min(k_len, i + (k_len - q_len) + 1) when causal, else k_len;
 *     lo = max(0, i + (k_len - q_len) - window_left + 1) when window_left > 0,
 *          else 0
 * (the bottom-right causal reading of the plain oracle, with the chunk's
 * tokens at the end of the context).  q_len = 1 with causal is paged decode.
 *
 * rows: NULL for every (token, head) of the batch, else flat indices
 * token * Hq + h; o_out [nrows][d], lse_out [nrows].  Returns the threads
 * used, -1 on invalid sizes, -2 on a block-table entry outside the pool.
 */
int oracle_prefill_paged(const uint16_t* q, const uint16_t* kcache, const uint16_t* vcache,
                         const int32_t* block_table, const int32_t* cu_seqlens_q,
                         const int32_t* seqlens_k, int num_seqs, int Hq, int Hkv, int d,
                         int page_size, int num_pages, int max_pages_per_seq, int causal,
                         int window_left, float scale, const int64_t* rows, int64_t nrows,
                         double* o_out, double* lse_out, int nthreads) {
    if (num_seqs < 0 || Hq <= 0 || Hkv <= 0 || d <= 0 || page_size <= 0 || window_left < 0) return -1;
    if (Hq % Hkv != 0) return -1;
    const int group = Hq / Hkv;
    if (num_seqs > 0 && cu_seqlens_q[0] != 0) return -1;
    int64_t max_len = 1;
    int s;
    for (s = 0; s < num_seqs; ++s) {
        if (cu_seqlens_q[s + 1] < cu_seqlens_q[s]) return -1;
        if (seqlens_k[s] < 0 || (int64_t)seqlens_k[s] > (int64_t)max_pages_per_seq * page_size) return -1;
        if (seqlens_k[s] > max_len) max_len = seqlens_k[s];
    }
    const int64_t total_q = num_seqs > 0 ? cu_seqlens_q[num_seqs] : 0;
    if (rows == NULL) nrows = total_q * Hq;
    nthreads = oracle_threads(nthreads);
    int bad = 0;

#pragma omp parallel num_threads(nthreads)
    {
        double* scratch = (double*)malloc(sizeof(double) * (size_t)max_len);
        const uint16_t** krows = (const uint16_t**)malloc(sizeof(void*) * (size_t)max_len);
        const uint16_t** vrows = (const uint16_t**)malloc(sizeof(void*) * (size_t)max_len);
        int64_t w;
#pragma omp for schedule(dynamic, 16)
        for (w = 0; w < nrows; ++w) {
            const int64_t r = rows ? rows[w] : w;
            if (r < 0 || r >= total_q * Hq) {
#pragma omp atomic write
                bad = 1;
                continue;
            }
            const int64_t token = r / Hq;
            const int h = (int)(r % Hq);
            /* the sequence holding this token: last s with cu_seqlens_q[s] <= token */
            int a = 0, b = num_seqs - 1;
            while (a < b) {
                int mid = (a + b + 1) / 2;
                if (cu_seqlens_q[mid] <= token) a = mid; else b = mid - 1;
            }
            const int seq = a;
            const int64_t q_len = cu_seqlens_q[seq + 1] - cu_seqlens_q[seq];
            const int64_t k_len = seqlens_k[seq];
            const int64_t i = token - cu_seqlens_q[seq];
            const int64_t diag = k_len - q_len;
            int64_t hi = causal ? i + diag + 1 : k_len;
            if (hi > k_len) hi = k_len;
            int64_t lo = window_left > 0 ? i + diag - window_left + 1 : 0;
            if (lo < 0) lo = 0;
            const int g = h / group;
            int64_t t, n = 0;
            int ok = 1;
            for (t = lo; t < hi; ++t, ++n) {
                int32_t page = block_table[(int64_t)seq * max_pages_per_seq + t / page_size];
                if (page < 0 || page >= num_pages) { ok = 0; break; }
                int64_t off = (((int64_t)page * page_size + t % page_size) * Hkv + g) * d;
                krows[n] = kcache + off;
                vrows[n] = vcache + off;
            }
            if (!ok) {
#pragma omp atomic write
                bad = 1;
                continue;
            }
            attend_row(q + r * d, krows, vrows, n, d, (double)scale, scratch, o_out + w * d, lse_out + w);
        }
        free(scratch);
        free(krows);
        free(vrows);
    }
    return bad ? -2 : nthreads;
}

/*
 * Backward pass: the gradients of the attention output with respect to Q, K
 * and V for an upstream gradient dO.
 *
 * The pages fix the forward only ("Compilers and Kernels", section
 * "FlashAttention changes the algorithm around IO": O = softmax(S) V with
 * S = scale * Q K^T + C); "Tang: a compiler that derives GPU kernels ...",
 * abstract: gradients of comprehensions are comprehensions, and a flash-style
 * attention backward recomputes instead of storing intermediates.  This is the
 * derivative of that definition, written out by the chain rule, in double
 * precision, from the exact softmax (two passes per row, no stored state):
 *
 *   P_ij  = exp(S_ij - m_i) / l_i            (the forward's weights)
 *   O_i   = sum_j P_ij V_j                    (exact, not a rounded input)
 *   dV_j  = sum_i P_ij dO_i
 *   dP_ij = dO_i . V_j
 *   D_i   = dO_i . O_i  ( = sum_j P_ij dP_ij )
 *   dS_ij = P_ij (dP_ij - D_i)                (softmax Jacobian)
 *   dQ_i  = scale * sum_j dS_ij K_j
 *   dK_j  = scale * sum_i dS_ij Q_i
 * With grouped-query attention dK and dV of a kv head sum over the query
 * heads that read it.  Masked keys (causal, bottom-right) have P = 0 and take
 * no gradient; a row with no allowed key contributes nothing.
 *
 * q, dout: [B][Hq][Nq][d]; k, v: [B][Hkv][Nk][d] (bf16 bits).  dq: [B][Hq][Nq][d],
 * dk, dv: [B][Hkv][Nk][d] (double).  Returns the threads used, -1 on invalid
 * sizes.
 */
int oracle_attention_bwd(const uint16_t* q, const uint16_t* k, const uint16_t* v, const uint16_t* dout,
                         int B, int Hq, int Hkv, int Nq, int Nk, int d, int causal, float scale,
                         double* dq, double* dk, double* dv, int nthreads) {
    if (B < 0 || Hq <= 0 || Hkv <= 0 || Nq < 0 || Nk < 0 || d <= 0) return -1;
    if (Hq % Hkv != 0) return -1;
    const int group = Hq / Hkv;
    const double sc = (double)scale;
    nthreads = oracle_threads(nthreads);
    memset(dq, 0, sizeof(double) * (size_t)B * Hq * Nq * d);
    memset(dk, 0, sizeof(double) * (size_t)B * Hkv * Nk * d);
    memset(dv, 0, sizeof(double) * (size_t)B * Hkv * Nk * d);
    const int64_t pairs = (int64_t)B * Hkv;

#pragma omp parallel num_threads(nthreads)
    {
        double* p = (double*)malloc(sizeof(double) * (size_t)(Nk > 0 ? Nk : 1));
        double* dp = (double*)malloc(sizeof(double) * (size_t)(Nk > 0 ? Nk : 1));
        double* o = (double*)malloc(sizeof(double) * (size_t)d);
        int64_t w;
        /* one (batch, kv head) per task: its dK and dV rows are written by it alone */
#pragma omp for schedule(dynamic, 1)
        for (w = 0; w < pairs; ++w) {
            const int64_t b = w / Hkv, g = w % Hkv;
            const uint16_t* kb = k + (b * Hkv + g) * (int64_t)Nk * d;
            const uint16_t* vb = v + (b * Hkv + g) * (int64_t)Nk * d;
            double* dkb = dk + (b * Hkv + g) * (int64_t)Nk * d;
            double* dvb = dv + (b * Hkv + g) * (int64_t)Nk * d;
            int hh;
            for (hh = 0; hh < group; ++hh) {
                const int64_t h = g * group + hh;
                int64_t i;
                for (i = 0; i < Nq; ++i) {
                    const int64_t row = (b * Hq + h) * (int64_t)Nq + i;
                    const uint16_t* qi = q + row * d;
                    const uint16_t* doi = dout + row * d;
                    int64_t n = Nk;
                    if (causal) {
                        n = i + (int64_t)Nk - (int64_t)Nq + 1;
                        if (n < 0) n = 0;
                        if (n > Nk) n = Nk;
                    }
                    if (n == 0) continue;
                    int64_t j;
                    int c;
                    double m = -INFINITY;
                    for (j = 0; j < n; ++j) {
                        double s = 0.0;
                        for (c = 0; c < d; ++c) s += bf16_to_double(qi[c]) * bf16_to_double(kb[j * d + c]);
                        p[j] = s * sc;
                        if (p[j] > m) m = p[j];
                    }
                    double l = 0.0;
                    for (j = 0; j < n; ++j) {
                        p[j] = exp(p[j] - m);
                        l += p[j];
                    }
                    for (c = 0; c < d; ++c) o[c] = 0.0;
                    for (j = 0; j < n; ++j) {
                        p[j] /= l;
                        for (c = 0; c < d; ++c) o[c] += p[j] * bf16_to_double(vb[j * d + c]);
                    }
                    double D = 0.0;
                    for (c = 0; c < d; ++c) D += bf16_to_double(doi[c]) * o[c];
                    for (j = 0; j < n; ++j) {
                        double s = 0.0;
                        for (c = 0; c < d; ++c) s += bf16_to_double(doi[c]) * bf16_to_double(vb[j * d + c]);
                        dp[j] = s;
                    }
                    double* dqi = dq + row * d;
                    for (j = 0; j < n; ++j) {
                        const double ds = p[j] * (dp[j] - D);
                        for (c = 0; c < d; ++c) {
                            dqi[c] += sc * ds * bf16_to_double(kb[j * d + c]);
                            dkb[j * d + c] += sc * ds * bf16_to_double(qi[c]);
                            dvb[j * d + c] += p[j] * bf16_to_double(doi[c]);
                        }
                    }
                }
            }
        }
        free(p);
        free(dp);
        free(o);
    }
    return nthreads;
}

/*
 * dQ for selected query rows only, by the per-row steps of
 * oracle_attention_bwd above (the weights of the row from its scores, its
 * output, D = dO . O, dP = dO V^T over the row's keys, dQ = scale * sum_j
 * P_j (dP_j - D) K_j): rows[r] = (b * Hq + h) * Nq + i, out[r][d].  The
 * cost is one row's keys per row, so rows of a long sequence can be checked
 * one by one.  Returns the threads used, or -1 on invalid arguments.
 */
int oracle_attention_bwd_dq_rows(const uint16_t* q, const uint16_t* k, const uint16_t* v, const uint16_t* dout,
                                 int B, int Hq, int Hkv, int Nq, int Nk, int d, int causal, float scale,
                                 const int64_t* rows, int64_t nrows, double* out, int threads) {
    const double sc = (double)scale;
    if (B < 0 || Hq <= 0 || Hkv <= 0 || Hq % Hkv != 0 || Nq < 0 || Nk < 0 || d <= 0 || nrows < 0) return -1;
    {
        int64_t r;
        for (r = 0; r < nrows; ++r)
            if (rows[r] < 0 || rows[r] >= (int64_t)B * Hq * Nq) return -1;
    }
    const int group = Hq / Hkv;
    const int nthreads = oracle_threads(threads);
#pragma omp parallel num_threads(nthreads)
    {
        double* p = (double*)malloc(sizeof(double) * (size_t)(Nk > 0 ? Nk : 1));
        double* dp = (double*)malloc(sizeof(double) * (size_t)(Nk > 0 ? Nk : 1));
        double* o = (double*)malloc(sizeof(double) * (size_t)d);
        int64_t r;
#pragma omp for schedule(dynamic, 1)
        for (r = 0; r < nrows; ++r) {
            const int64_t row = rows[r];
            const int64_t bh = row / Nq, i = row % Nq;
            const int64_t b = bh / Hq, h = bh % Hq, g = h / group;
            const uint16_t* kb = k + (b * Hkv + g) * (int64_t)Nk * d;
            const uint16_t* vb = v + (b * Hkv + g) * (int64_t)Nk * d;
            const uint16_t* qi = q + row * d;
            const uint16_t* doi = dout + row * d;
            double* dqi = out + r * d;
            int64_t n = Nk, j;
            int c;
            for (c = 0; c < d; ++c) dqi[c] = 0.0;
            if (causal) {
                n = i + (int64_t)Nk - (int64_t)Nq + 1;
                if (n < 0) n = 0;
                if (n > Nk) n = Nk;
            }
            if (n == 0) continue;
            double m = -INFINITY;
            for (j = 0; j < n; ++j) {
                double s = 0.0;
                for (c = 0; c < d; ++c) s += bf16_to_double(qi[c]) * bf16_to_double(kb[j * d + c]);
                p[j] = s * sc;
                if (p[j] > m) m = p[j];
            }
            double l = 0.0;
            for (j = 0; j < n; ++j) {
                p[j] = exp(p[j] - m);
                l += p[j];
            }
            for (c = 0; c < d; ++c) o[c] = 0.0;
            for (j = 0; j < n; ++j) {
                p[j] /= l;
                for (c = 0; c < d; ++c) o[c] += p[j] * bf16_to_double(vb[j * d + c]);
            }
            double D = 0.0;
            for (c = 0; c < d; ++c) D += bf16_to_double(doi[c]) * o[c];
            for (j = 0; j < n; ++j) {
                double s = 0.0;
                for (c = 0; c < d; ++c) s += bf16_to_double(doi[c]) * bf16_to_double(vb[j * d + c]);
                dp[j] = s;
            }
            for (j = 0; j < n; ++j) {
                const double ds = p[j] * (dp[j] - D);
                for (c = 0; c < d; ++c) dqi[c] += sc * ds * bf16_to_double(kb[j * d + c]);
            }
        }
        free(p);
        free(dp);
        free(o);
    }
    return nthreads;
}

/*
 * Backward of oracle_attention_masked: the same derivative as
 * oracle_attention_bwd (dV = P^T dO, dS = P * (dP - D), dQ = scale dS K,
 * dK = scale dS^T Q), with the weights P of the biased scores
 * S_ij = scale q_i . k_j + C_ij over the keys the causal mask and the left
 * window allow, C_ij = alibi[h] (j - i - (Nk - Nq)) + bias[b sb + h sh + i Nk + j].
 * A key whose score is -inf, and every key of a row with no finite score,
 * takes no gradient.  Layouts and return value as oracle_attention_bwd.
 */
int oracle_attention_masked_bwd(const uint16_t* q, const uint16_t* k, const uint16_t* v, const uint16_t* dout,
                                int B, int Hq, int Hkv, int Nq, int Nk, int d, int causal, float scale,
                                int window_left, const float* alibi, const uint16_t* bias, int64_t bias_sb,
                                int64_t bias_sh, double* dq, double* dk, double* dv, int nthreads) {
    if (B < 0 || Hq <= 0 || Hkv <= 0 || Nq < 0 || Nk < 0 || d <= 0 || window_left < 0) return -1;
    if (Hq % Hkv != 0) return -1;
    const int group = Hq / Hkv;
    const double sc = (double)scale;
    nthreads = oracle_threads(nthreads);
    memset(dq, 0, sizeof(double) * (size_t)B * Hq * Nq * d);
    memset(dk, 0, sizeof(double) * (size_t)B * Hkv * Nk * d);
    memset(dv, 0, sizeof(double) * (size_t)B * Hkv * Nk * d);
    const int64_t pairs = (int64_t)B * Hkv;
    const int64_t diag = (int64_t)Nk - (int64_t)Nq;

#pragma omp parallel num_threads(nthreads)
    {
        const size_t cap = (size_t)(Nk > 0 ? Nk : 1);
        double* p = (double*)malloc(sizeof(double) * cap);
        double* dp = (double*)malloc(sizeof(double) * cap);
        int64_t* keys = (int64_t*)malloc(sizeof(int64_t) * cap);
        double* o = (double*)malloc(sizeof(double) * (size_t)d);
        int64_t w;
        /* one (batch, kv head) per task: its dK and dV rows are written by it alone */
#pragma omp for schedule(dynamic, 1)
        for (w = 0; w < pairs; ++w) {
            const int64_t b = w / Hkv, g = w % Hkv;
            const uint16_t* kb = k + (b * Hkv + g) * (int64_t)Nk * d;
            const uint16_t* vb = v + (b * Hkv + g) * (int64_t)Nk * d;
            double* dkb = dk + (b * Hkv + g) * (int64_t)Nk * d;
            double* dvb = dv + (b * Hkv + g) * (int64_t)Nk * d;
            int hh;
            for (hh = 0; hh < group; ++hh) {
                const int64_t h = g * group + hh;
                int64_t i;
                for (i = 0; i < Nq; ++i) {
                    const int64_t row = (b * Hq + h) * (int64_t)Nq + i;
                    const uint16_t* qi = q + row * d;
                    const uint16_t* doi = dout + row * d;
                    int64_t n = 0, j, t;
                    int c;
                    double m = -INFINITY;
                    /* the allowed keys of row i and their biased scores */
                    for (j = 0; j < Nk; ++j) {
                        if (causal && j > i + diag) continue;
                        if (window_left > 0 && j <= i + diag - window_left) continue;
                        double s = 0.0;
                        for (c = 0; c < d; ++c) s += bf16_to_double(qi[c]) * bf16_to_double(kb[j * d + c]);
                        s *= sc;
                        if (alibi) s += (double)alibi[h] * (double)(j - i - diag);
                        if (bias) s += bf16_to_double(bias[b * bias_sb + h * bias_sh + i * (int64_t)Nk + j]);
                        keys[n] = j;
                        p[n] = s;
                        if (s > m) m = s;
                        ++n;
                    }
                    if (n == 0 || m == -INFINITY) continue;
                    double l = 0.0;
                    for (t = 0; t < n; ++t) {
                        p[t] = exp(p[t] - m);
                        l += p[t];
                    }
                    for (c = 0; c < d; ++c) o[c] = 0.0;
                    for (t = 0; t < n; ++t) {
                        p[t] /= l;
                        for (c = 0; c < d; ++c) o[c] += p[t] * bf16_to_double(vb[keys[t] * d + c]);
                    }
                    double D = 0.0;
                    for (c = 0; c < d; ++c) D += bf16_to_double(doi[c]) * o[c];
                    for (t = 0; t < n; ++t) {
                        double s = 0.0;
                        for (c = 0; c < d; ++c) s += bf16_to_double(doi[c]) * bf16_to_double(vb[keys[t] * d + c]);
                        dp[t] = s;
                    }
                    double* dqi = dq + row * d;
                    for (t = 0; t < n; ++t) {
                        const double ds = p[t] * (dp[t] - D);
                        const int64_t jj = keys[t];
                        for (c = 0; c < d; ++c) {
                            dqi[c] += sc * ds * bf16_to_double(kb[jj * d + c]);
                            dkb[jj * d + c] += sc * ds * bf16_to_double(qi[c]);
                            dvb[jj * d + c] += p[t] * bf16_to_double(doi[c]);
                        }
                    }
                }
            }
        }
        free(p);
        free(dp);
        free(keys);
        free(o);
    }
    return nthreads;
}
