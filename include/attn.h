/*
 * attn.h -- C ABI of the GB300 fused-attention library (libattn_gb300.so).
 *
 * The operation ("Compilers and Kernels", section "FlashAttention changes the
 * algorithm around IO", the definition of scaled dot-product attention and the
 * block recurrence that follows it):
 *
 *     S = scale * Q K^T + C,  m_i = max_j S_ij,  l_i = sum_j exp(S_ij - m_i),
 *     O_i = sum_j exp(S_ij - m_i) V_j / l_i,  LSE_i = m_i + ln l_i,
 *
 * computed in one fused pass in which the per-row state (m, l, o) is carried
 * over key blocks and merged associatively ("Tang: a compiler that derives GPU
 * kernels ...", abstract: online softmax as a monoid), so the N x N score
 * matrix never reaches memory.  The logsumexp output is the one named in
 * "Don't Write Kernels, Derive Them", section "What happened".
 *
 * Conventions shared by every entry point
 * ---------------------------------------
 *  - Every tensor pointer is a DEVICE pointer owned by the caller; the library
 *    never frees or retains it after the call returns.  Inputs are read only;
 *    outputs must not alias inputs or each other.
 *  - Tensors are dense and row-major with the head dimension innermost
 *    (strided views are not accepted: copy them first).  bf16 means IEEE
 *    bfloat16 bit patterns (uint16_t).  Pointers must be 16-byte aligned.
 *  - C is 0 or -inf: with causal != 0, key j is allowed for query i iff
 *    j <= i + (Nk - Nq) (bottom-right alignment; "query i attends keys 0..i"
 *    when Nq == Nk).  A row with no allowed key gets O = 0 and LSE = -inf.
 *  - Grouped-query attention: query head h reads key/value head
 *    h / (Hq / Hkv); Hq must be a multiple of Hkv.
 *  - Head dimension d (for Q, K and V alike) must be 64, 128 or 256.
 *  - LSE is natural-log, float32.  O is bf16 (o_dtype = ATTN_BF16) or float32
 *    (ATTN_F32, for diagnostics).  Accumulation is float32 throughout; P is
 *    rounded to bf16 (round-to-nearest-even) before the P V product.
 *  - Calls are asynchronous on `stream` (NULL = the legacy default stream):
 *    arguments are checked synchronously and an error status is returned
 *    before anything is launched; a launch failure returns ATTN_ERR_LAUNCH.
 *    Faults the kernels detect while running (a wait that timed out, an
 *    out-of-range block-table entry or sequence length) are recorded in a
 *    device status word read by attn_get_device_status().
 *  - Forward and decode results are deterministic run to run (fixed work
 *    split, no atomics in any reduction); attn_bwd's dQ is the one exception
 *    (see there).
 *  - The GPU must be compute capability 10.3 (GB300, sm_103a); otherwise
 *    ATTN_ERR_UNSUPPORTED.
 *  - Every wait inside a kernel is bounded (1 s).  A wait that gives up
 *    records ATTN_ERR_TIMEOUT and its kernel unwinds and exits instead of
 *    hanging; its outputs are then incomplete, and copies it had issued may
 *    not have landed when it exited.  After ATTN_ERR_TIMEOUT treat the CUDA
 *    context, and this library's state on that device, as suspect: finish
 *    the process (or reset the device from a fresh process) before trusting
 *    further results.
 *  - Each declaration below names the passage of the pages its operation
 *    follows ("Source:"), or says that the pages have no counterpart.
 */
#ifndef ATTN_GB300_H
#define ATTN_GB300_H

#include <stddef.h>
#include <stdint.h>

#ifdef __cplusplus
extern "C" {
#endif

#if defined(__GNUC__)
#define ATTN_API __attribute__((visibility("default")))
#else
#define ATTN_API
#endif

/* Same object as cudaStream_t / CUstream; declared here so that this header
 * needs no CUDA header. */
struct CUstream_st;
typedef struct CUstream_st* attn_stream_t;

typedef enum {
    ATTN_OK = 0,
    ATTN_ERR_INVALID_ARG = 1,  /* a size is negative, zero where it may not be, or inconsistent */
    ATTN_ERR_UNSUPPORTED = 2,  /* d, page size or query-head group outside what the call takes; wrong GPU */
    ATTN_ERR_MISALIGNED = 3,   /* a pointer is NULL or not 16-byte aligned */
    ATTN_ERR_WORKSPACE = 4,    /* decode workspace NULL or smaller than attn_decode_workspace_size() */
    ATTN_ERR_LAUNCH = 5,       /* the CUDA runtime refused a launch or an attribute */
    ATTN_ERR_TIMEOUT = 6,      /* device: a pipeline wait exceeded its time limit (see below) */
    ATTN_ERR_BOUNDS = 7,       /* device: block-table entry or sequence length out of range */
    ATTN_ERR_NO_DEVICE = 8     /* no CUDA device is usable */
} attn_status;

typedef enum { ATTN_BF16 = 0, ATTN_F32 = 1 } attn_dtype;

/*
 * Prefill / general forward attention.
 * Source: "Compilers and Kernels", section "FlashAttention changes the
 * algorithm around IO" (the definition of attention, the block recurrence
 * over key blocks and its exactness); LSE as in "Don't Write Kernels, Derive
 * Them", section "What happened".
 *   q:   [B, Hq, Nq, d] bf16          k, v: [B, Hkv, Nk, d] bf16
 *   o:   [B, Hq, Nq, d] bf16 or f32   lse:  [B, Hq, Nq] f32
 *   scale: multiplies Q K^T (1/sqrt(d) for the textbook operator); finite
 *          and > 0.
 * B, Hq, Hkv, Nq, Nk >= 0; nothing is launched when the output is empty.
 * With Nk == 0 (or every key masked) each row is O = 0, LSE = -inf.
 *
 * Work distribution: one persistent CTA per SM takes units from a counter in
 * a ring of 64 slots built into the library; each call takes the next slot.
 * Calls in flight at the same time (any streams) use different slots unless
 * more than 64 are in flight: a call whose slot is still held by an earlier
 * call waits, on the GPU, until that call has handed out its last unit
 * (bounded: ATTN_ERR_TIMEOUT after 1 s, e.g. when the earlier call cannot
 * run because this one occupies the GPU).  A call captured into a CUDA graph
 * keeps its slot in every replay; two replays of one graph must not overlap
 * on the GPU (the same holds for attn_fwd_masked and attn_prefill_paged).
 */
ATTN_API attn_status attn_fwd(const void* q, const void* k, const void* v, void* o, float* lse,
                     int B, int Hq, int Hkv, int Nq, int Nk, int d, int causal,
                     float scale, attn_dtype o_dtype, attn_stream_t stream);

/*
 * Additive bias C beyond the causal mask.
 * Source: "Compilers and Kernels", section "FlashAttention changes the
 * algorithm around IO" (S = Q K^T / sqrt(d) + C, C in R U {-inf}).  Every
 * field may be left zero.
 *   window_left:   > 0 keeps, for query i, only keys j > i + (Nk - Nq) - window_left
 *                  (with causal: the window_left most recent keys up to the
 *                  diagonal); key tiles wholly outside the window are skipped.
 *   alibi_slopes:  NULL or a device [Hq] float32 array; adds
 *                  alibi_slopes[h] * (j - i - (Nk - Nq)) to S_ij.
 *   bias:          NULL or a device bf16 array read as
 *                  bias[b*bias_stride_b + h*bias_stride_h + i*Nk + j] (strides in
 *                  elements, 0 to broadcast); -inf disallows a key.  A dense bias
 *                  costs one read of Nq*Nk values per (batch, head).
 * alibi_slopes and bias must be 4-byte aligned.
 */
typedef struct {
    int window_left;
    const float* alibi_slopes;
    const void* bias;
    long long bias_stride_b;
    long long bias_stride_h;
} attn_mask;

/*
 * attn_fwd with the additive bias `mask` (NULL: same as attn_fwd).  A row
 * whose keys are all disallowed (or all -inf after the bias) gets O = 0 and
 * LSE = -inf.
 * Source: "Compilers and Kernels", section "FlashAttention changes the
 * algorithm around IO" (the additive term C of the score definition).
 */
ATTN_API attn_status attn_fwd_masked(const void* q, const void* k, const void* v, void* o, float* lse,
                     int B, int Hq, int Hkv, int Nq, int Nk, int d, int causal,
                     float scale, const attn_mask* mask, attn_dtype o_dtype, attn_stream_t stream);

/*
 * Bytes of scratch memory attn_prefill_paged() needs: the unit prefix sums
 * (num_seqs + 1 int32) and the sequences' dispatch order (num_seqs int32),
 * each rounded up to 256.  0 on invalid input.
 * Source: "Compilers and Kernels", section "A kernel implements a bounded
 * contract" (a kernel states the workspace it needs).
 */
ATTN_API size_t attn_prefill_paged_workspace_size(int num_seqs);

/*
 * Chunked prefill against a paged KV cache, ragged over sequences.
 * Source: "Don't Write Kernels, Derive Them", section "What happened" (paged
 * KV-cache access); the attention of each row as in attn_fwd.
 *   q:            [total_q, Hq, d] bf16, the sequences' new tokens packed in order
 *   kcache/vcache: [num_pages, page_size, Hkv, d] bf16 (the layout of
 *                 attn_decode_paged), already holding every context token,
 *                 the new ones included
 *   block_table:  [num_seqs, max_pages_per_seq] int32 device
 *   cu_seqlens_q: [num_seqs + 1] int32 device: sequence s owns query tokens
 *                 [cu_seqlens_q[s], cu_seqlens_q[s+1]); cu_seqlens_q[0] = 0 and
 *                 the last entry <= total_q
 *   seqlens_k:    [num_seqs] int32 device: context length k_len of sequence s
 *                 (<= max_pages_per_seq * page_size)
 *   o:            [total_q, Hq, d] bf16 or f32;  lse: [total_q, Hq] f32
 * The q_len new tokens are the last q_len of the context: with causal, query
 * i of the chunk sees keys j <= i + k_len - q_len (bottom-right alignment);
 * window_left > 0 also drops keys j <= i + k_len - q_len - window_left.  A row
 * with no key gets O = 0 and LSE = -inf.  page_size must be 16, 32, 64 or
 * 128; workspace: device scratch of attn_prefill_paged_workspace_size()
 * bytes, 16-byte aligned, caller-owned, not shared by overlapping calls.
 * Cache slots past a sequence's context are never read as values (they may
 * hold anything).  Inconsistent lengths or a block-table entry outside the
 * pool are reported through attn_get_device_status() (ATTN_ERR_BOUNDS); the
 * affected sequence is skipped or the entry not read.
 */
ATTN_API attn_status attn_prefill_paged(const void* q, const void* kcache, const void* vcache,
                                        const int32_t* block_table, const int32_t* cu_seqlens_q,
                                        const int32_t* seqlens_k, void* o, float* lse, int num_seqs,
                                        int total_q, int Hq, int Hkv, int d, int page_size, int num_pages,
                                        int max_pages_per_seq, int causal, int window_left, float scale,
                                        void* workspace, size_t workspace_bytes, attn_dtype o_dtype,
                                        attn_stream_t stream);

/*
 * Bytes of scratch memory attn_bwd() needs: D = rowsum(dO * O) per query row
 * (f32) and an f32 dQ accumulator [B, Hq, Nq, d] (used when the gradients
 * are bf16; f32 gradients accumulate in dq itself), each rounded up to 256.
 * 0 on invalid input (including d other than 64, 128, 256).
 * Source: "Compilers and Kernels", section "A kernel implements a bounded
 * contract" (a kernel states the workspace it needs).
 */
ATTN_API size_t attn_bwd_workspace_size(int B, int Hq, int Nq, int d);

/*
 * Backward pass of attn_fwd: the gradients of O with respect to Q, K and V
 * for an upstream gradient dO, recomputing the weights from the saved LSE.
 * Source: "Tang: a compiler that derives GPU kernels and bounds how fast they
 * can run", abstract (a fused flash-style attention backward); "Compilers and
 * Kernels", section "FlashAttention changes the algorithm around IO" (the
 * backward recomputes score and probability tiles instead of storing them).  With P = softmax(S) the forward's
 * weights and D_i = dO_i . O_i:  dV = P^T dO,  dS = P * (dO V^T - D),
 * dQ = scale * dS K,  dK = scale * dS^T Q  (dK, dV summed over the query heads
 * of a kv group).
 *   q, o, dout: [B, Hq, Nq, d] bf16 (o: the forward's output); lse: [B, Hq, Nq]
 *   f32 from attn_fwd; k, v: [B, Hkv, Nk, d] bf16; causal, scale as passed to
 *   attn_fwd.  dq: [B, Hq, Nq, d]; dk, dv: [B, Hkv, Nk, d], bf16 or f32 by
 *   grad_dtype.  d must be 64, 128 or 256 (else ATTN_ERR_UNSUPPORTED).
 *   workspace: device scratch of attn_bwd_workspace_size() bytes, 16-byte
 *   aligned, caller-owned, not shared by overlapping calls.
 * Two or three kernels on `stream` (rows D and a zeroed dQ accumulator; the fused
 * backward, one CTA per (batch, kv head, 128-key tile), two at d = 256 (one
 * per half of the head dim); the bf16 dQ conversion, when grad_dtype is bf16).
 * dK and dV are deterministic; dQ sums its per-key-tile parts with TMA
 * reduce-adds in no fixed order, so its last bits can differ from run to run.
 */
ATTN_API attn_status attn_bwd(const void* q, const void* k, const void* v, const void* o, const void* dout,
                              const float* lse, void* dq, void* dk, void* dv, int B, int Hq, int Hkv, int Nq,
                              int Nk, int d, int causal, float scale, attn_dtype grad_dtype, void* workspace,
                              size_t workspace_bytes, attn_stream_t stream);

/*
 * Backward pass of attn_fwd_masked: attn_bwd for the biased scores
 * S = scale Q K^T + C, with `mask` the one passed to the forward (NULL: same
 * as attn_bwd).  The formulas of attn_bwd hold with P the biased weights; a
 * key the mask disallows, or whose bias is -inf, takes no gradient, and no
 * gradient with respect to C is formed.  Key tiles wholly outside a left
 * window are skipped.  Arguments, workspace, kernels and determinism as
 * attn_bwd; the bias is read once per (key tile, query tile) pair it covers.
 * Source: "Compilers and Kernels", section "FlashAttention changes the
 * algorithm around IO" (the additive term C of the score definition; the
 * backward recomputes the weights); "Tang: a compiler that derives GPU
 * kernels and bounds how fast they can run", abstract (fused backward).
 */
ATTN_API attn_status attn_bwd_masked(const void* q, const void* k, const void* v, const void* o, const void* dout,
                                     const float* lse, void* dq, void* dk, void* dv, int B, int Hq, int Hkv,
                                     int Nq, int Nk, int d, int causal, float scale, const attn_mask* mask,
                                     attn_dtype grad_dtype, void* workspace, size_t workspace_bytes,
                                     attn_stream_t stream);

/*
 * Measurement aid for the decode time floor: one thread follows
 * idx = chain[idx] (starting at 0) for `hops` dependent loads that bypass L1
 * and writes the elapsed nanoseconds to out_ns[0] (out_ns[1] receives the last
 * index).  chain: device uint32 array of chain_len entries (chain_len < 2^32)
 * whose every visited entry should hold an index < chain_len (the caller
 * builds a cycle through a buffer larger than L2, one entry per 128-byte
 * line, and flushes L2 first); an entry >= chain_len stops the walk and is
 * reported (ATTN_ERR_BOUNDS; out_ns[0] = 0, out_ns[1] = the entry).
 * out_ns: device array of 2 uint64.  One DRAM round trip = out_ns[0] / hops.
 * Source: "Tang: a compiler that derives GPU kernels and bounds how fast they
 * can run", abstract (a time floor from the traffic bound, the measured
 * launch cost and the DRAM latency).
 */
ATTN_API attn_status attn_probe_dram_latency(const uint32_t* chain, size_t chain_len, int hops,
                                             unsigned long long* out_ns, attn_stream_t stream);

/*
 * Bytes of scratch memory attn_decode_paged() needs for these sizes (the
 * split partials: one float32 O row and one float32 LSE per sequence, split
 * and query head).  Pure function of its arguments; 0 on invalid input.
 * It takes Hkv as well as Hq: the number of key chunks per sequence (and so
 * the partials) is chosen from the number of (sequence, kv-head group) work
 * items, which depends on the grouping of query heads over kv heads.
 * Source: "Compilers and Kernels", section "A kernel implements a bounded
 * contract" (a kernel states the workspace it needs); the partials are the
 * monoid states of "Tang: a compiler that derives GPU kernels and bounds how
 * fast they can run", abstract (online softmax as a monoid).
 */
ATTN_API size_t attn_decode_workspace_size(int num_seqs, int Hq, int Hkv, int d, int max_seqlen);

/*
 * Paged decode: one query row per sequence and query head against that
 * sequence's cached keys/values, split over key chunks whose partial states
 * are merged by the online-softmax monoid (a split kernel, then a combine
 * kernel launched as its programmatic dependent; sequences that fit one chunk
 * are finished by the split kernel).
 * Source: "Don't Write Kernels, Derive Them", section "What happened" (paged
 * KV-cache access, logsumexp); "Tang: a compiler that derives GPU kernels and
 * bounds how fast they can run", abstract (online softmax as a monoid; decode
 * as a narrow GEMV-class stage).
 *   q:           [num_seqs, Hq, d] bf16
 *   kcache/vcache: [num_pages, page_size, Hkv, d] bf16; page_size 16, 32, 64
 *                or 128
 *   block_table: [num_seqs, max_pages_per_seq] int32; token t of sequence s is
 *                slot t % page_size of page block_table[s][t / page_size]
 *   seqlens:     [num_seqs] int32, each in [0, max_seqlen] and
 *                <= max_pages_per_seq * page_size (checked on the device)
 *   o:           [num_seqs, Hq, d] bf16 or f32;  lse: [num_seqs, Hq] f32
 *   max_seqlen:  host-side upper bound of seqlens (sizes the work split)
 *   scale:       as for attn_fwd: finite and > 0
 *   workspace:   device scratch of at least attn_decode_workspace_size() bytes,
 *                16-byte aligned, owned by the caller, contents ignored; it
 *                must not be shared by two calls that overlap on the GPU.
 * Hq / Hkv (query heads per key/value head) must be 1, 2, 4, 8 or 16.  The
 * query row attends every cached token (no mask).
 */
ATTN_API attn_status attn_decode_paged(const void* q, const void* kcache, const void* vcache,
                              const int32_t* block_table, const int32_t* seqlens,
                              void* o, float* lse,
                              int num_seqs, int Hq, int Hkv, int d, int page_size,
                              int num_pages, int max_pages_per_seq, int max_seqlen,
                              float scale, void* workspace, size_t workspace_bytes,
                              attn_dtype o_dtype, attn_stream_t stream);

/*
 * Paged decode that allocates nothing and takes no workspace argument.
 *
 * Same inputs, outputs, checks and results as attn_decode_paged(), but the
 * split partials live in a scratch array compiled into this library (a
 * file-scope device array of ATTN_STATIC_SCRATCH_BYTES on every GPU that
 * loads the library, held until the process exits).  It is meant for callers
 * that cannot call cudaMalloc or hand over a buffer of their own -- for
 * example code whose device memory is all owned by a host framework's fixed
 * pool, or a latency-critical loop where an allocation (which may synchronise
 * the device) is not acceptable.  The paper has no counterpart to this entry
 * point; it is a deployment convenience of this library.
 *
 *  - Sizes whose attn_decode_workspace_size() exceeds ATTN_STATIC_SCRATCH_BYTES
 *    are rejected with ATTN_ERR_WORKSPACE before anything is launched.
 *  - The first call on each device looks up the array's device address
 *    (cudaGetSymbolAddress) with that device current; make that first call
 *    before any stream capture begins.
 *  - Every call on a device shares the one array.  Calls that may overlap on
 *    the GPU (different streams without ordering between them) race on it and
 *    corrupt each other's results; order them on one stream.  Nothing in the
 *    array needs to start at zero: every value a call reads back was written
 *    earlier in that same call.
 */
#define ATTN_STATIC_SCRATCH_BYTES (64u << 20)
ATTN_API attn_status attn_decode_paged_static(const void* q, const void* kcache, const void* vcache,
                              const int32_t* block_table, const int32_t* seqlens,
                              void* o, float* lse,
                              int num_seqs, int Hq, int Hkv, int d, int page_size,
                              int num_pages, int max_pages_per_seq, int max_seqlen,
                              float scale, attn_dtype o_dtype, attn_stream_t stream);

/*
 * Waits for `stream`, then returns and clears the device status word of the
 * current device (ATTN_OK when no kernel recorded a fault since the last
 * call).  Not for the hot path: it synchronises.
 * Source: "Compilers and Kernels", section "A kernel implements a bounded
 * contract" (a kernel states how it reports errors).
 */
ATTN_API attn_status attn_get_device_status(attn_stream_t stream);

/*
 * Failure-detection self-test (diagnostics, not part of the attention path).
 * Launches one CTA whose thread waits on a shared-memory barrier that nothing
 * will ever complete, using the same bounded-wait routine as the kernels but
 * with a limit of `limit_us` microseconds (1..1000000).  The wait gives up,
 * records ATTN_ERR_TIMEOUT in the device status word and the kernel returns,
 * leaving the CUDA context usable.  Returns ATTN_OK once launched (read the
 * outcome with attn_get_device_status), ATTN_ERR_INVALID_ARG for a limit out
 * of range.  No GPU work waits on anything the host or another kernel does.
 * The pages have no counterpart: it exercises the error path that "Compilers
 * and Kernels", section "A kernel implements a bounded contract", asks a
 * kernel to state.
 */
ATTN_API attn_status attn_selftest_wait_timeout(uint32_t limit_us, attn_stream_t stream);

/* Static, human-readable name of a status code.  The pages have no
 * counterpart (a library convenience). */
ATTN_API const char* attn_status_string(attn_status s);

/* Number of kernels this library has launched in this process.  The pages
 * have no counterpart (a measurement convenience). */
ATTN_API uint64_t attn_launch_count(void);

/* Version of this ABI (bumped on any incompatible change).  The pages have no
 * counterpart (a library convenience). */
ATTN_API int attn_abi_version(void);

/* The kernel instantiation attn_fwd() launches for these sizes on the current
 * device, e.g. "prefill_fwd_kernel<128,2,4,0,0>" (head dim, query tiles per
 * unit, K/V ring stages, bias variant, paged); "" for sizes it rejects.  The
 * string lives in thread-local storage until the next call on that thread.
 * The pages have no counterpart (a measurement convenience: it names the
 * kernel a profile or a roofline figure belongs to). */
ATTN_API const char* attn_fwd_kernel_name(int B, int Hq, int Nq, int d);

/* The kernels attn_decode_paged() launches for these sizes, e.g.
 * "decode_split_kernel<128,4,1> + decode_combine_kernel" (head dim, query
 * heads per warp, warps per key/value head); "" for sizes it rejects.  Thread-local storage as for
 * attn_fwd_kernel_name.  The pages have no counterpart (a measurement
 * convenience). */
ATTN_API const char* attn_decode_kernel_name(int num_seqs, int Hq, int Hkv, int d, int max_seqlen);

#ifdef __cplusplus
}
#endif

#endif /* ATTN_GB300_H */
