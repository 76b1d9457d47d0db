/*
 * b300attn: exact softmax attention for NVIDIA B300 (sm_103a), C ABI.
 *
 *   O = softmax(scale * Q K^T + mask) V,   LSE_i = ln sum_j exp(scale * q_i.k_j + mask_ij)
 *
 * computed by tiling with an online softmax, so the N x N score matrix never
 * reaches global memory ("FlashAttention" learn page, aiunderstanding.org,
 * sections "Deep dive" and "Technical insight"; FAQ on exactness: the result
 * is the same as standard attention, only the order of the work changes).
 *
 * Conventions shared by every entry point
 * ---------------------------------------
 *  - Every pointer argument is a DEVICE pointer owned by the caller.  The
 *    library never allocates or frees memory and never synchronises the
 *    stream; all work is enqueued on `stream` (0 = legacy default stream).
 *  - Layouts are row-major with the head dimension d contiguous; bf16 means
 *    IEEE bfloat16, f32 means IEEE binary32.
 *  - Query head h reads key/value head h / (Hq / Hkv) (grouped-query heads).
 *  - A row with no visible key gets O = 0 and LSE = -inf.
 *  - Return value: B300ATTN_OK, or a negative b300attn_status.  On a host-side
 *    error nothing is enqueued and attn_last_error() describes the problem.
 *    B300ATTN_ERR_CUDA means a CUDA call (e.g. the launch) failed.
 *  - Inputs with nothing to compute (B == 0, N == 0, rows == 0) return OK and
 *    enqueue nothing; pointers may then be NULL.
 *  - Thread safety: stateless apart from a thread-local error message and a
 *    per-device status word written only when a kernel's bounded wait expires.
 */
#ifndef B300ATTN_H
#define B300ATTN_H

#include <stddef.h>

#ifdef __cplusplus
extern "C" {
#endif

/* Same definition as the CUDA runtime's; passing a cudaStream_t works as is. */
typedef struct CUstream_st* cudaStream_t;

typedef enum {
  B300ATTN_OK = 0,
  B300ATTN_ERR_INVALID = -1,     /* bad argument: NULL, negative size, misaligned, ... */
  B300ATTN_ERR_UNSUPPORTED = -2, /* valid but not implemented (e.g. d not in {64,128}) */
  B300ATTN_ERR_WORKSPACE = -3,   /* workspace missing or smaller than required */
  B300ATTN_ERR_CUDA = -4,        /* a CUDA runtime/driver call failed */
  B300ATTN_ERR_TIMEOUT = -5      /* a kernel gave up on a bounded wait (see attn_device_status) */
} b300attn_status;

typedef enum { B300ATTN_BF16 = 0, B300ATTN_F32 = 1 } b300attn_dtype;

/*
 * attn_fwd -- prefill attention (causal, sliding-window or non-causal).
 *
 * Implements the tiled, online-softmax form of attention: Q, K, V move through
 * on-chip memory in tiles, a running row maximum and row sum are kept and
 * partial outputs rescaled as new tiles arrive ("FlashAttention" learn page,
 * "Technical insight" and FAQ on how softmax is computed without seeing all
 * scores); key tiles a row cannot see are skipped.  The window is the local
 * attention of the Arabic thread on extending context length (point 1:
 * tokens attend only to their neighbours).
 *
 *   q    bf16 [B, N, Hq,  d]       k, v  bf16 [B, N, Hkv, d]
 *   o    [B, N, Hq, d], bf16 or f32 as o_dtype says
 *   lse  f32  [B, Hq, N], natural logarithm
 *   causal  0/1: row i sees keys j <= i (square, top-left aligned)
 *   window  < 0: no window; w >= 0: row i sees keys with |i - j| <= w
 *           (with causal: i - w <= j <= i)
 *   scale   finite, >= 0 (1/sqrt(d) is the usual choice)
 *   d in {64, 128}; Hq % Hkv == 0; every pointer 16-byte aligned.
 * Errors: INVALID (NULL/negative/misaligned/bad scale or dtype), UNSUPPORTED (d),
 * CUDA (launch failure).
 */
int attn_fwd(const void* q, const void* k, const void* v, void* o, float* lse, int B, int Hq,
             int Hkv, int N, int d, int causal, int window, float scale, cudaStream_t stream,
             int o_dtype);

/*
 * attn_fwd_varlen -- prefill over a batch of sequences of different lengths,
 * packed back to back along the token axis (no padding).
 *
 * The same tiled online-softmax attention as attn_fwd, applied within each
 * sequence: sequence s owns tokens [cu_seqlens[s], cu_seqlens[s+1]) and its
 * queries see only its own keys (with the causal / window masks of attn_fwd,
 * positions counted from the sequence's first token).  This is the
 * "variable-length" form that long-document and serving workloads use
 * ("FlashAttention" learn page, "The future of FlashAttention": variants for
 * irregular and sliding-window attention).
 *
 *   q    bf16 [T, Hq, d]        k, v  bf16 [T, Hkv, d]      (T = total_rows)
 *   o    [T, Hq, d], bf16 or f32 as o_dtype says;  lse  f32 [Hq, T]
 *   cu_seqlens  int32 [num_seqs + 1], DEVICE, non-decreasing, cu_seqlens[0] = 0,
 *               cu_seqlens[num_seqs] <= total_rows.  Values are clamped to
 *               [0, total_rows] on the device (a decreasing entry gives an
 *               empty sequence); rows outside every sequence are not written.
 *   max_seqlen  upper bound of the sequence lengths (sizes the launch only).
 *   1 <= num_seqs <= 4096; other arguments as for attn_fwd.
 * Errors: INVALID, UNSUPPORTED (d, num_seqs > 4096), CUDA.
 */
int attn_fwd_varlen(const void* q, const void* k, const void* v, void* o, float* lse,
                    const int* cu_seqlens, int num_seqs, int total_rows, int max_seqlen, int Hq,
                    int Hkv, int d, int causal, int window, float scale, cudaStream_t stream,
                    int o_dtype);

/*
 * FP8 (e4m3) prefill.  FlashAttention-3 computes attention in low-precision
 * FP8 ("FlashAttention" learn page, aiunderstanding.org, section on the
 * future of FlashAttention; FlashAttention-3 article, ybx.com,
 * "FlashAttention-3 innovations" item 3).  The pages fix no format or scaling;
 * this library uses:
 *   - e4m3 codes (1 sign, 4 exponent bits with bias 7, 3 mantissa bits, no
 *     infinities, largest finite value 448), conversion rounding to nearest
 *     even and saturating at +-448;
 *   - one int32 exponent e per tile: the largest e with amax * 2^e <= 448
 *     (amax = max |x| over the tile; 0 for an all-zero tile; clamped to
 *     [-126, 126]); a code c stands for c * 2^-e;
 *   - tiles: Q and K per 128 rows (tokens) of one (batch, head); V per
 *     (batch, head) over the whole sequence.  V is stored transposed,
 *     [B, Hkv, d, Np] with Np = attn_fp8_padded_len(N) (N rounded up to 16),
 *     keys N..Np-1 zero.
 * d = 128 only; dense [B, N, H, d] layout only.
 */

/* attn_fp8_padded_len -- key-axis length Np of the transposed FP8 V (0 for N <= 0). */
int attn_fp8_padded_len(int N);

/*
 * attn_fp8_workspace_size -- bytes of workspace attn_fp8_quantize needs (the
 * f32 maximum of every 128-key tile of V, [B, Hkv, ceil(N/128)]), a multiple
 * of 256; 256 on empty or invalid sizes.
 */
size_t attn_fp8_workspace_size(int B, int Hkv, int N);

/*
 * attn_fp8_quantize -- bf16 Q, K, V to e4m3 codes with per-tile exponents.
 *
 *   q          bf16 [B, N, Hq, d]      k, v  bf16 [B, N, Hkv, d]
 *   q8         e4m3 [B, N, Hq, d]      k8    e4m3 [B, N, Hkv, d]
 *   v8t        e4m3 [B, Hkv, d, Np]    (V transposed; Np as above)
 *   q_exp      int32 [B, Hq, ceil(N/128)]   k_exp  int32 [B, Hkv, ceil(N/128)]
 *   v_exp      int32 [B, Hkv]
 *   workspace  >= attn_fp8_workspace_size(B, Hkv, N) bytes, 256-byte aligned
 *   d == 128; Hq % Hkv == 0; q, k, v, q8, k8, v8t 16-byte aligned.
 * Two kernel launches.  The outputs are a function of the inputs alone (no
 * state, bit-identical on every call).
 * Errors: INVALID, UNSUPPORTED (d), WORKSPACE, CUDA.
 */
int attn_fp8_quantize(const void* q, const void* k, const void* v, void* q8, void* k8, void* v8t,
                      int* q_exp, int* k_exp, int* v_exp, int B, int Hq, int Hkv, int N, int d,
                      void* workspace, size_t workspace_bytes, cudaStream_t stream);

/*
 * attn_fwd_fp8 -- prefill attention on e4m3 operands from attn_fp8_quantize.
 *
 * The same tiled online-softmax computation as attn_fwd, with both tensor-core
 * products in e4m3 and f32 accumulation: S = Q8 K8^T is scaled by
 * scale * 2^-(e_Q + e_K) of its tile pair; the softmax numerators P (at most
 * 2^8) are rounded to e4m3 before O += P V8; O is divided by the row sum and
 * by 2^e_V.  LSE uses the unrounded numerators.
 *
 *   q8, k8, v8t, q_exp, k_exp, v_exp   as written by attn_fp8_quantize
 *   o    [B, N, Hq, d], bf16 or f32 as o_dtype says
 *   lse  f32 [B, Hq, N], natural logarithm
 *   causal, window, scale as for attn_fwd; d == 128; one kernel launch.
 * Errors: INVALID, UNSUPPORTED (d), CUDA.
 */
int attn_fwd_fp8(const void* q8, const void* k8, const void* v8t, const int* q_exp,
                 const int* k_exp, const int* v_exp, void* o, float* lse, int B, int Hq, int Hkv,
                 int N, int d, int causal, int window, float scale, cudaStream_t stream,
                 int o_dtype);

/*
 * attn_fwd_paged -- attn_fwd with K and V kept in a paged pool, the layout an
 * inference server keeps its KV cache in ("FlashAttention" learn page, "The
 * future of FlashAttention": integration into inference servers, and variants
 * for irregular attention).  Sequence b's key/value j is row j % page_size of
 * page block_table[b * pages_per_seq + j / page_size]; each 128-key tile is
 * gathered by two 64-row TMA copies.  Queries, masks, O and LSE are exactly
 * those of attn_fwd with the gathered K and V.
 *
 *   q            bf16 [B, N, Hq, d]
 *   k_pages, v_pages  bf16 [num_pages, page_size, Hkv, d]
 *   block_table  int32 [B, pages_per_seq], device; entries for keys < N must
 *                lie in [0, num_pages); entries past a sequence's N keys are
 *                not read.  The kernel checks each entry it reads: one out of
 *                range is never dereferenced, its keys read as zeros, and the
 *                next attn_device_status returns B300ATTN_ERR_INVALID.
 *   page_size    a positive multiple of 64;  pages_per_seq * page_size >= N
 *   o, lse, causal, window, scale, o_dtype, stream  as for attn_fwd.
 * Errors: INVALID, UNSUPPORTED, CUDA.
 */
int attn_fwd_paged(const void* q, const void* k_pages, const void* v_pages,
                   const int* block_table, void* o, float* lse, int B, int Hq, int Hkv, int N,
                   int d, int page_size, int num_pages, int pages_per_seq, int causal,
                   int window, float scale, cudaStream_t stream, int o_dtype);

/*
 * attn_bwd_workspace_size -- bytes of workspace attn_bwd needs: the f32 row
 * terms D = rowsum(dO * O) [B, Hq, N], 256-byte aligned.  0 on invalid input.
 */
size_t attn_bwd_workspace_size(int B, int Hq, int N);

/*
 * attn_bwd -- gradients dQ, dK, dV of attn_fwd's O with respect to q, k, v,
 * given dO, the forward's O and its LSE.
 *
 * The forward's softmax weights are recomputed tile by tile from the saved
 * LSE (P = exp(scale q.k - LSE)), so that, as in the forward, the N x N
 * matrices stay on chip; then dV = P^T dO, dP = dO V^T,
 * dS = P * (dP - rowsum(dO * O)), dQ = scale dS K, dK = scale dS^T Q.  Query
 * heads of a group add into their kv head's dK and dV.  (The pages stress
 * faster training, "FlashAttention-3" article, "Benefits": the backward pass
 * is what training runs besides the forward.)  Three launches: the row terms,
 * dK/dV (one CTA per kv head and 128-key tile), dQ (one CTA per query head and
 * 128-query tile); no atomics, so the result is deterministic.
 *
 *   q, o, dO   [B, N, Hq, d] (q, dO bf16; o bf16 or f32 as o_dtype says)
 *   k, v       bf16 [B, N, Hkv, d]
 *   lse        f32 [B, Hq, N] from attn_fwd with the same causal/window/scale
 *   dq         bf16 [B, N, Hq, d];   dk, dv  bf16 [B, N, Hkv, d]
 *   workspace  >= attn_bwd_workspace_size(B, Hq, N) bytes, 256-byte aligned
 *   d in {64, 128}; other arguments as for attn_fwd.
 * Errors: INVALID, UNSUPPORTED, WORKSPACE, CUDA.
 */
int attn_bwd(const void* q, const void* k, const void* v, const void* o, const float* lse,
             const void* dO, void* dq, void* dk, void* dv, void* workspace,
             size_t workspace_bytes, int B, int Hq, int Hkv, int N, int d, int causal, int window,
             float scale, cudaStream_t stream, int o_dtype);

/*
 * attn_decode_chunk -- keys per split used by attn_decode_splitkv:
 * ceil(max_kv_len / num_splits) rounded up to a multiple of 64.  Returns a
 * negative status on invalid arguments.
 */
int attn_decode_chunk(int max_kv_len, int num_splits);

/*
 * attn_decode_workspace_size -- bytes of workspace attn_decode_splitkv needs
 * for the split partials: f32 m and l [B, Hq, num_splits] and f32 o
 * [B, Hq, num_splits, d], each region 256-byte aligned; with more than 64
 * splits, followed by the second level of the merge (the same three arrays
 * with nseg = ceil(num_splits / 64) in place of num_splits).  0 on invalid
 * input.
 */
size_t attn_decode_workspace_size(int B, int Hq, int num_splits, int d);

/*
 * attn_decode_splitkv -- single-query decode over a (possibly ragged) KV cache.
 *
 * The key axis of every sequence is cut into num_splits chunks of
 * attn_decode_chunk(max_kv_len, num_splits) keys.  One kernel computes, per
 * (sequence, kv head, chunk), the partial triple of every query head in the
 * group -- m = max score, l = sum exp(s - m), o = sum exp(s - m) v -- streaming
 * each K/V byte once per group; a second kernel merges the partials with the
 * logsumexp tree (two levels when there are more than 64 splits: segments of
 * 64 partials, then the segment triples).  The split and the tree follow the
 * Tree Attention page (express24.ir), abstract: the reduction along the
 * sequence axis is associative and can be computed as a tree.
 *
 *   q        bf16 [B, Hq, d]
 *   k_cache, v_cache  bf16 [B, max_kv_len, Hkv, d]; only rows < kv_len[b] are read
 *                     into the result (rows beyond may hold anything, even NaN)
 *   kv_len   int32 [B], device; values are clamped to [0, max_kv_len]
 *   o        [B, Hq, d] bf16 or f32 (o_dtype);  lse  f32 [B, Hq]
 *   workspace  device buffer of at least attn_decode_workspace_size(B, Hq,
 *              num_splits, d) bytes, 256-byte aligned; contents on return are
 *              the partials (m in natural-log units).
 *   d in {64, 128}; Hq % Hkv == 0; 1 <= num_splits <= 65535.
 * Errors: INVALID, UNSUPPORTED, WORKSPACE (NULL or too small), CUDA.
 */
int attn_decode_splitkv(const void* q, const void* k_cache, const void* v_cache,
                        const int* kv_len, void* o, float* lse, int B, int Hq, int Hkv,
                        int max_kv_len, int d, float scale, int num_splits, void* workspace,
                        size_t workspace_bytes, cudaStream_t stream, int o_dtype);

/*
 * attn_decode_splitkv_noalloc -- attn_decode_splitkv without a caller-supplied
 * workspace, for callers that cannot allocate device memory at the point where
 * they run decode.  Examples: a plugin whose host framework owns all device
 * memory and forbids allocation inside its execution step, or a
 * latency-critical loop where cudaMalloc, which may synchronise the whole
 * device, is not acceptable.  Those callers still pass q, the caches, kv_len,
 * o and lse; this entry point allocates nothing itself (no cudaMalloc, no
 * cudaFree, no allocating library call).
 *
 * The split partials go to a scratch array compiled into the library (a
 * file-scope __device__ array of 40 MiB = 41943040 bytes).  Every device that
 * loads the library holds that array until the process exits.  A call whose
 * partials would need more than that (attn_decode_workspace_size(B, Hq,
 * num_splits, d) > 40 MiB) returns B300ATTN_ERR_WORKSPACE with a message; e.g.
 * 1 sequence x 32 heads x 2048 splits x d=128 needs 33.0 MiB
 * (34,611,200 bytes) and fits.
 *
 * The first call on a device looks up the scratch array's device address
 * (cudaGetSymbolAddress, with that device current) and caches it; make that
 * first call before any stream capture.  All calls share the one array and it
 * keeps the last call's contents, so calls that overlap on the GPU (different
 * streams, or host threads without ordering between them) race and corrupt
 * each other's results: serialise them.  Nothing in the array needs clearing
 * between calls, because each call rewrites every partial it later reads.
 *
 * The paper has no counterpart to this entry point; it exists for the
 * allocation constraint above.  Arguments, layouts and errors are otherwise
 * those of attn_decode_splitkv.
 */
int attn_decode_splitkv_noalloc(const void* q, const void* k_cache, const void* v_cache,
                                const int* kv_len, void* o, float* lse, int B, int Hq, int Hkv,
                                int max_kv_len, int d, float scale, int num_splits,
                                cudaStream_t stream, int o_dtype);

/*
 * attn_decode_splitkv_paged -- attn_decode_splitkv over a paged KV cache, the
 * layout inference servers keep for many sequences of changing length
 * ("FlashAttention" learn page, "The future of FlashAttention": integration
 * into inference servers).  Keys and values live in fixed-size pages of a
 * shared pool; sequence b's logical key k is row k % page_size of physical
 * page block_table[b * pages_per_seq + k / page_size].
 *
 *   k_pages, v_pages  bf16 [num_pages, page_size, Hkv, d]
 *   block_table       int32 [B, pages_per_seq], device; entries for keys
 *                     < kv_len[b] must lie in [0, num_pages) (others are not read).
 *                     The kernel checks each entry it reads: one outside that range
 *                     is never dereferenced, its page counts as holding no keys, and
 *                     the next attn_device_status returns B300ATTN_ERR_INVALID.
 *   kv_len            int32 [B], device; clamped to [0, pages_per_seq * page_size]
 *   page_size         a positive multiple of 64
 *   other arguments, the split, the workspace and the errors as for
 *   attn_decode_splitkv with max_kv_len = pages_per_seq * page_size.
 */
int attn_decode_splitkv_paged(const void* q, const void* k_pages, const void* v_pages,
                              const int* block_table, const int* kv_len, void* o, float* lse,
                              int B, int Hq, int Hkv, int page_size, int num_pages,
                              int pages_per_seq, int d, float scale, int num_splits,
                              void* workspace, size_t workspace_bytes, cudaStream_t stream,
                              int o_dtype);

/*
 * attn_decode_partials -- the first half of attn_decode_splitkv on its own:
 * writes the per-split partial triples (m, l, o) of every query head into
 * `workspace` (layout as described for attn_decode_splitkv) and does not merge
 * them.  Partials produced on different devices or streams for disjoint key
 * ranges can be merged with lse_tree_combine, which is the cross-device
 * decoding scheme of the Tree Attention page (abstract).  Arguments as for
 * attn_decode_splitkv, without o, lse and o_dtype.  Split c of sequence b
 * covers keys [c*chunk, min((c+1)*chunk, kv_len[b])); an empty split gets
 * m = -inf, l = 0, o = 0.
 */
int attn_decode_partials(const void* q, const void* k_cache, const void* v_cache,
                         const int* kv_len, int B, int Hq, int Hkv, int max_kv_len, int d,
                         float scale, int num_splits, void* workspace, size_t workspace_bytes,
                         cudaStream_t stream);

/*
 * lse_tree_combine -- merge split partials in a logsumexp tree.
 *
 * For each of `rows` rows, merges num_splits triples (m, l, o) with
 *   (m,l,o) + (m',l',o') = (M, l e^(m-M) + l' e^(m'-M), o e^(m-M) + o' e^(m'-M)),
 *   M = max(m, m'),
 * (Tree Attention page, abstract: the sequence-axis reduction as a tree), then
 * writes O = o / l and LSE = M + ln l.  A partial with m = -inf is the empty
 * identity and its o is never read.
 *
 * One thread-block cluster of up to 8 CTAs merges a row: each CTA a
 * contiguous segment of the partials, the CTAs' triples merged through
 * distributed shared memory.
 *
 *   part_m, part_l  f32 [rows, num_splits]   (m in natural-log units)
 *   part_o          f32 [rows, num_splits, d], 16-byte aligned
 *   o               [rows, d] bf16 or f32 (o_dtype), 16-byte aligned;  lse  f32 [rows]
 *   d in {64, 128}; num_splits >= 1.
 * Errors: INVALID, UNSUPPORTED, CUDA.
 */
int lse_tree_combine(const float* part_m, const float* part_l, const float* part_o, void* o,
                     float* lse, int rows, int num_splits, int d, cudaStream_t stream,
                     int o_dtype);

/*
 * attn_device_status -- synchronises `stream`, then reads and clears this
 * library's device status words for the current device.  Returns
 * B300ATTN_ERR_TIMEOUT if any kernel gave up on a bounded wait since the last
 * call (the kernel then stopped early and its outputs are not valid),
 * B300ATTN_ERR_INVALID if the only event was a paged decode reading a
 * block_table entry outside [0, num_pages), B300ATTN_ERR_CUDA if the
 * synchronisation failed, else B300ATTN_OK.
 *
 * Debug build (libb300attn_debug.so, compiled with -DB300ATTN_DEBUG): the
 * kernels also check caller data that the release build clamps (a decode
 * kv_len entry outside [0, max_kv_len]; cu_seqlens that decrease or leave
 * [0, total_rows]) and their own tile and index invariants.  A failed check
 * makes this call return B300ATTN_ERR_INVALID, with the check's bits in
 * attn_last_error(); the kernels themselves carry on with the clamped values
 * and compute what the release build computes.
 */
int attn_device_status(cudaStream_t stream);

/*
 * attn_selftest_bounded_wait -- exercises the failure path that every
 * pipeline wait of the kernels above shares.  One thread of a one-warp kernel
 * waits on a shared-memory barrier that nothing ever arrives on, with no copy
 * and no tensor-core work in flight; the wait gives up after `limit_ns`
 * nanoseconds of %globaltimer, records its status bit and the kernel returns.
 * The next attn_device_status(stream) then returns B300ATTN_ERR_TIMEOUT once
 * and clears the bit, and the context stays usable.  (Not a step of the
 * method: a test of the library's bounded waits, which exist so that a stuck
 * pipeline stops instead of hanging the GPU.)
 *   limit_ns  in [1000, 100000000] (1 us .. 100 ms), else B300ATTN_ERR_INVALID.
 * Errors: INVALID, CUDA.
 */
int attn_selftest_bounded_wait(unsigned long long limit_ns, cudaStream_t stream);

/* Message describing the last non-OK status returned on this thread ("" if none). */
const char* attn_last_error(void);

/* Library version, major * 10000 + minor * 100 + patch. */
int attn_version(void);

#ifdef __cplusplus
}
#endif

#endif /* B300ATTN_H */
