/*
 * rkv_attn.h -- C ABI of the GB300 resident-attention library (librkv_attn.so).
 *
 * Three operations on GPU-resident f32 data, computing
 *     output = softmax(Q . K^T * scale) . V          per query head
 * as defined on the trueno-gpu 0.4.11 page (src/memory/resident/attention.rs,
 * fn batched_multihead_attention: the doc comment's softmax(Q K^T / sqrt(d_k)) V)
 * and the trustformers-core 0.2.0 page (src/gpu_ops/cuda/oxicuda/attention.rs,
 * fn attention_prefill_gpu_to_gpu / fn attention_decode_gpu_to_gpu).
 *
 * Conventions shared by every entry point
 *  - Every tensor pointer is a DEVICE pointer to row-major float32 (int32 for
 *    lengths), 16-byte aligned.  The caller owns all memory; the library
 *    allocates nothing, copies nothing to the host and never synchronises.
 *  - Work is enqueued on `stream` and the call returns at once (the pages'
 *    "no sync, caller chains on its stream" convention: trueno-gpu,
 *    fn incremental_attention_gpu_with_stream / fn kv_cache_scatter_gpu).
 *  - Shapes are validated on the host before anything is launched
 *    (the pages' InvalidParameter / shape_error pattern); a rejected call
 *    launches nothing and returns RKV_ERR_INVALID_ARG or RKV_ERR_UNSUPPORTED,
 *    with a message in rkv_last_error().
 *  - Values that live in device memory (lengths, positions) cannot be checked
 *    on the host without a sync; kernels clamp or skip them and record the
 *    event in a device flag word read by rkv_read_device_flags().
 *  - GQA: query head h uses kv head h / (n_heads / n_kv_heads); n_heads must
 *    be a multiple of n_kv_heads (realizar 0.8.5, cache_from_cache_from_kv_cache.rs,
 *    fn init_kv_cache_gpu sizes the cache by num_kv_heads <= num_heads).
 *  - head_dim must be one of 16, 32, 64, 128 (RKV_ERR_UNSUPPORTED otherwise).
 *  - scale == 0 selects 1/sqrt(head_dim) (trueno-gpu,
 *    fn batched_multihead_attention); a negative or non-finite scale is
 *    rejected.
 *  - Zero-sized work (batch, seq_len, M or T == 0) is a successful no-op.
 */
#ifndef RKV_ATTN_H
#define RKV_ATTN_H

#include <stddef.h>

#ifdef __cplusplus
extern "C" {
#endif

#if !defined(__DRIVER_TYPES_H__)
typedef struct CUstream_st* cudaStream_t;   /* same type as the CUDA runtime's */
#endif

typedef enum {
    RKV_OK = 0,
    RKV_ERR_INVALID_ARG = 1,   /* bad pointer, shape, alignment or workspace */
    RKV_ERR_UNSUPPORTED = 2,   /* valid request outside what the kernels implement */
    RKV_ERR_LAUNCH = 3,        /* the CUDA runtime reported an error */
    RKV_ERR_DEVICE = 4         /* a device-side condition, see rkv_read_device_flags */
} rkv_status;

/* Device flag bits (rkv_read_device_flags). */
#define RKV_FLAG_WAIT_TIMEOUT    0x1u  /* a bounded on-chip wait gave up; outputs invalid */
#define RKV_FLAG_LEN_CLAMPED     0x2u  /* a seq_lens entry exceeded its bound and was clamped */
#define RKV_FLAG_NEGATIVE_INPUT  0x4u  /* a negative length or position was treated as 0 / skipped */
#define RKV_FLAG_BAD_POINTER     0x8u  /* a per-sequence cache pointer was NULL or not 16-byte aligned: that
                                          sequence was skipped (no row read or written, zero output) */
#define RKV_FLAG_BOUNDS          0x10u /* checked build only (librkv_attn_checked.so, device checks compiled
                                          in): an index a kernel computed fell outside its buffer and that
                                          access was skipped -- a defect in the library, never expected */

/* Bytes at the head of a decode workspace that hold its completion tickets
 * (attn_decode_batched and the other decode entry points).  Their place does
 * not depend on the call's sizes. */
#define RKV_DECODE_TICKET_BYTES 32768

/* Library version, (major << 16) | minor. */
int rkv_version(void);

/* Static text for a status code. */
const char* rkv_status_string(rkv_status status);

/* Message describing the most recent failing call made on this host thread
 * ("" if none).  The pointer stays valid until the next call on this thread. */
const char* rkv_last_error(void);

/*
 * Reads (and, if clear != 0, resets) the device flag word of the current
 * device.  Synchronises `stream`.  Returns RKV_OK and *flags, or
 * RKV_ERR_LAUNCH.  Diagnostic only; the compute entry points never sync.
 */
rkv_status rkv_read_device_flags(unsigned int* flags, int clear, cudaStream_t stream);

/*
 * Self-check of the failure path of the on-chip waits.  Every mbarrier wait in
 * the kernels is bounded (2 s per phase); on expiry the kernel sets
 * RKV_FLAG_WAIT_TIMEOUT, unwinds (lets its copies and MMAs in flight finish,
 * frees tensor memory) and returns, so the context stays usable.  This call
 * runs the same bounded wait in one warp on a barrier that nothing completes,
 * with a limit of limit_us microseconds: it must give up, set
 * RKV_FLAG_WAIT_TIMEOUT and return.  limit_us in [1, 1000000]
 * (RKV_ERR_INVALID_ARG otherwise).  Asynchronous on `stream`; read the flag
 * with rkv_read_device_flags.
 */
rkv_status rkv_check_wait_timeout(unsigned int limit_us, cudaStream_t stream);

/*
 * Self-check of the operand rounding of the prefill.  The tensor core reads an
 * f32 operand of a TF32 product by dropping its 13 low mantissa bits; the
 * prefill first adds half a TF32 unit in the last place to the bit pattern of
 * each element of Q and V, which makes the drop a round to nearest, ties away
 * from zero (infinities stay infinite, positive NaNs stay NaN; a negative NaN
 * at 0xFFFFF000 or above is read as +0).  For each of the n f32 bit patterns in
 * x this writes ours[i] = that rounding with the low 13 bits cleared, and
 * ref[i] = the hardware conversion cvt.rna.tf32.f32 of x[i]; the two agree bit
 * for bit on every finite input.  Device pointers, 4-byte aligned; n >= 0.
 * Asynchronous on `stream`.  No counterpart on the pages.
 */
rkv_status rkv_check_tf32_round(const unsigned int* x, unsigned int* ours, unsigned int* ref, int n,
                                cudaStream_t stream);

/*
 * Prefill attention over interleaved activations, causal or not, with GQA.
 *
 * Cites: trueno-gpu attention.rs, fn batched_multihead_attention_optimized
 * (interleaved [seq, n_heads*head_dim] in and out); trustformers-core
 * attention.rs, fn attention_prefill_gpu_to_gpu (causal: query i sees keys
 * 0..=i, from an empty cache).
 *
 *   q        [batch, seq_len, n_heads*head_dim]      input
 *   k, v     [batch, seq_len, n_kv_heads*head_dim]   input
 *   o        [batch, seq_len, n_heads*head_dim]      output, fully written
 *   causal   0: every query sees keys 0..len-1; 1: query i sees keys 0..min(i, len-1)
 *   seq_lens device int32[batch] valid lengths (<= seq_len), or NULL for all
 *            seq_len.  Query rows i >= len are written as 0; keys j >= len are
 *            ignored.  Entries > seq_len are clamped (RKV_FLAG_LEN_CLAMPED),
 *            negative entries count as 0 (RKV_FLAG_NEGATIVE_INPUT).
 *   scale    0 -> 1/sqrt(head_dim)
 * Heads are read in place (no head-split copies); no score matrix is stored.
 * Arithmetic: QK^T and PV on TF32 tensor cores with f32 accumulation; softmax
 * in f32.  Q and V are rounded to the nearest TF32 value (rkv_check_tf32_round),
 * K and the probabilities are truncated to TF32 (the probabilities' row sum is
 * taken over the truncated values).  Non-finite inputs give unspecified rows
 * (a NaN need not propagate).  o must not alias q, k or v.
 */
rkv_status attn_prefill(const float* q, const float* k, const float* v, float* o,
                        int batch, int seq_len, int n_heads, int n_kv_heads, int head_dim,
                        int causal, const int* seq_lens, float scale, cudaStream_t stream);

/*
 * Prefill of fresh sequences fused with their cache fill: attn_prefill (without
 * seq_lens) plus kv_cache_scatter of all seq_len rows at positions 0..seq_len-1,
 * in one kernel.
 *
 * Cites: trueno-gpu attention.rs, fn batched_multihead_attention_optimized and
 * trustformers-core attention.rs, fn attention_prefill_gpu_to_gpu (the
 * attention); realizar cache_from_cache_from_kv_cache.rs, cache filled after a
 * prefill into [M, num_kv_heads, max_len, head_dim] (the fill).
 *
 *   q, k, v, o  as attn_prefill (every row of every sequence valid)
 *   k_cache,
 *   v_cache     [batch, n_kv_heads, max_len, head_dim], updated in place:
 *               cache[b, kh, t, :] = k[b, t, kh*head_dim : (kh+1)*head_dim] for
 *               t < seq_len (same for v); rows t >= seq_len are untouched.
 * o is the same as attn_prefill's to the bit, and the cache rows are bit-exact
 * copies.  Two kernels on `stream`: the prefill, and the fill launched as its
 * programmatic dependent, which starts at once beside the prefill (in the
 * registers and shared memory a prefill CTA leaves free on each SM), reads the
 * K/V rows while the prefill has them in L2, and completes only after the
 * prefill, so later work on `stream` is ordered after both.  0 <= batch <= 32,
 * seq_len <= max_len; o and the caches must not alias the inputs or each other.
 */
rkv_status attn_prefill_fill_cache(const float* q, const float* k, const float* v, float* o,
                                   int batch, int seq_len, int n_heads, int n_kv_heads,
                                   int head_dim, int causal, float scale, float* k_cache,
                                   float* v_cache, int max_len, cudaStream_t stream);

/*
 * Prefill appended behind rows already in the resident cache (chunked prefill).
 *
 * Cites: trustformers-core attention.rs, fn attention_prefill_gpu_to_gpu (its
 * doc: the causal mask is the from-empty-cache one, and a prefill appended to
 * an existing cache must run the decode path once per token) and
 * fn attention_decode_gpu_to_gpu (one query against every cached row).  This
 * call computes that per-token result for a whole chunk in one launch.
 *
 *   q          [M, T, n_heads*head_dim]             input, T new tokens per sequence
 *   k_cache,
 *   v_cache    [M, n_kv_heads, max_len, head_dim]   input; must already hold the
 *              chunk's own K/V rows at start_pos .. start_pos+n-1 (kv_cache_scatter)
 *   o          [M, T, n_heads*head_dim]             output, fully written
 *   start_pos  device int32[M]: p0, cache rows present before the chunk
 *   q_lens     device int32[M]: valid tokens n of the chunk (<= T), or NULL for T;
 *              rows i >= n are written as 0
 *   causal     1: token i (position p0+i) sees cache rows 0..p0+i;
 *              0: every valid token sees rows 0..p0+n-1
 * Device values out of range are clamped and flagged: n > T or p0 + n > max_len
 * (keys past max_len are not read; RKV_FLAG_LEN_CLAMPED), negative p0 or n
 * (treated as 0; RKV_FLAG_NEGATIVE_INPUT).  Cache rows past p0+n are never
 * used, even if they hold NaN.  Same kernel and arithmetic as attn_prefill
 * (TF32 tensor cores, f32 accumulation; K/V tiles by tensor copies straight
 * from the cache).  0 <= M <= 32, T <= max_len; o must not alias q or the caches.
 */
rkv_status attn_prefill_chunked(const float* q, const float* k_cache, const float* v_cache,
                                float* o, int M, int T, int n_heads, int n_kv_heads,
                                int head_dim, int max_len, int causal, const int* start_pos,
                                const int* q_lens, float scale, cudaStream_t stream);

/*
 * Bytes of device workspace attn_decode_batched needs for these sizes:
 * RKV_DECODE_TICKET_BYTES of tickets, then the split-KV partial records.
 * Returns 0 for invalid sizes (including M * n_kv_heads above
 * RKV_DECODE_TICKET_BYTES / 4).
 */
size_t attn_decode_workspace_bytes(int M, int n_heads, int n_kv_heads, int head_dim,
                                   int max_len);

/*
 * Batched single-token decode attention against the resident KV cache.
 *
 * Cites: trueno-gpu attention.rs, fn incremental_attention_gpu (one query per
 * head against cache rows 0..seq_len-1; seq_len == 0 gives a zero row);
 * trustformers-core attention.rs, fn attention_decode_gpu_to_gpu (no mask);
 * realizar cache_from_cache_from_kv_cache.rs, fn init_batched_kv_cache_gpu
 * (M <= 32 sequences, cache [M, num_kv_heads, max_len, head_dim], per-sequence
 * lengths).
 *
 *   q          [M, n_heads*head_dim]               input, one token per sequence
 *   k_cache,
 *   v_cache    [M, n_kv_heads, max_len, head_dim]  input
 *   o          [M, n_heads*head_dim]               output, fully written
 *   seq_lens   device int32[M]: rows 0..len-1 of each sequence are attended
 *              (the length INCLUDING the token just appended).  len > max_len
 *              is clamped (RKV_FLAG_LEN_CLAMPED); len <= 0 gives a zero row.
 *   workspace  device buffer of >= attn_decode_workspace_bytes(...) bytes,
 *              256-byte aligned, ZERO-FILLED before its first use.  Its first
 *              RKV_DECODE_TICKET_BYTES bytes are completion tickets, one per
 *              (sequence m, kv head kh) at int index m * n_kv_heads + kh,
 *              whatever the sizes; every call that completes leaves them zero,
 *              so one workspace sized for the largest call can be reused by
 *              calls of any sizes without clearing.  A call that raised
 *              RKV_FLAG_WAIT_TIMEOUT may leave tickets non-zero: zero the first
 *              RKV_DECODE_TICKET_BYTES bytes before the workspace is used again.
 *              Calls sharing one workspace must not overlap on the GPU (use one
 *              workspace per concurrent stream).
 * 1 <= M <= 32; n_heads / n_kv_heads in {1, 2, 4, 8}; M * n_kv_heads <=
 * RKV_DECODE_TICKET_BYTES / 4 (RKV_ERR_UNSUPPORTED otherwise).  Split-KV: the cache rows
 * of all sequences are cut into equal contiguous pieces, one per CTA; pieces
 * of one (sequence, kv head) are merged with a log-sum-exp combine inside the
 * same launch.  Arithmetic is f32.
 */
rkv_status attn_decode_batched(const float* q, const float* k_cache, const float* v_cache,
                               float* o, int M, int n_heads, int n_kv_heads, int head_dim,
                               int max_len, const int* seq_lens, float scale,
                               void* workspace, size_t workspace_bytes, cudaStream_t stream);

/*
 * attn_decode_batched without a caller workspace, for callers that cannot
 * allocate device memory when they decode (an allocator owned by someone
 * else, a plugin host that forbids allocation after start-up, a real-time
 * loop that must not block in cudaMalloc).  The reference pages have no
 * counterpart: their decode paths allocate per call.
 *
 * Same arguments, semantics and results as attn_decode_batched, minus the
 * workspace.  The scratch is a fixed 4 MiB array in the library's own device
 * memory, held on every GPU that loads the library until the process exits;
 * sizes whose workspace (attn_decode_workspace_bytes) exceeds it are rejected
 * with RKV_ERR_UNSUPPORTED.  Nothing is allocated: no cudaMalloc, no library
 * allocator.  The first call on a device looks up the array's device address,
 * and so does the first call after that device's context changed (for
 * instance after cudaDeviceReset); make the first call before any stream
 * capture.  The lookup is guarded by a lock.  Each call clears the part of the
 * array that must start at zero with an asynchronous memset on `stream`.
 * All calls share the one array: calls that overlap on the GPU (different
 * streams or host threads on one device) race and give wrong results.
 */
rkv_status attn_decode_batched_noalloc(const float* q, const float* k_cache,
                                       const float* v_cache, float* o, int M, int n_heads,
                                       int n_kv_heads, int head_dim, int max_len,
                                       const int* seq_lens, float scale, cudaStream_t stream);

/*
 * One decode step in one launch: append each sequence's new K/V row at
 * position seq_lens[m] - 1, then decode over seq_lens[m] rows -- the same
 * results, cache and output, as kv_cache_scatter(k_new, v_new, ..., T = 1,
 * start_pos = seq_lens - 1) followed by attn_decode_batched.
 *
 * Cites: trueno-gpu attention.rs, fn kv_cache_scatter_gpu then
 * fn incremental_attention_gpu (append the token, then attend to rows
 * 0..seq_len-1); realizar batched cache layout.
 *
 *   k_new, v_new  [M, n_kv_heads*head_dim]  the step's new rows
 *   k_cache, v_cache                        updated in place at row seq_lens[m]-1
 *                                           (not written when that row is
 *                                           outside [0, max_len))
 * Every other argument as attn_decode_batched.  The new row is the last row
 * each (sequence, kv head) attends to; the one CTA that reads it takes it
 * straight from k_new / v_new and writes it into the cache when it is done
 * with its rows, so no separate launch, grid-wide ordering or wait on the
 * write is needed.  Outputs must not alias the inputs.
 */
rkv_status attn_decode_append(const float* q, const float* k_new, const float* v_new,
                              float* k_cache, float* v_cache, float* o, int M, int n_heads,
                              int n_kv_heads, int head_dim, int max_len, const int* seq_lens,
                              float scale, void* workspace, size_t workspace_bytes,
                              cudaStream_t stream);

/*
 * attn_decode_batched over per-sequence caches instead of one batched cache:
 * the pointer-array layout of realizar cache_from_cache_from_kv_cache.rs, which
 * keeps device arrays of per-sequence K and V pointers (batched_k_ptrs,
 * batched_v_ptrs) so each sequence's cache can live anywhere.
 *
 *   k_ptrs, v_ptrs  device arrays of M device pointers (8-byte aligned); entry m
 *                   addresses sequence m's cache [n_kv_heads, max_len, head_dim]
 *                   and must be 16-byte aligned.  A NULL or misaligned entry is
 *                   never dereferenced: the sequence is decoded as empty (zero
 *                   output) and RKV_FLAG_BAD_POINTER is raised.  A pointer to
 *                   memory that is not a valid cache of that size is the caller's
 *                   error (it cannot be checked on the device).
 * Everything else as attn_decode_batched (same kernel, same results).  Rollback
 * (realizar fn rollback_kv_cache_gpu) needs no call: decoding with a smaller
 * seq_lens ignores the rows past it.
 */
rkv_status attn_decode_batched_ptrs(const float* q, const float* const* k_ptrs,
                                    const float* const* v_ptrs, float* o, int M, int n_heads,
                                    int n_kv_heads, int head_dim, int max_len,
                                    const int* seq_lens, float scale, void* workspace,
                                    size_t workspace_bytes, cudaStream_t stream);

/*
 * kv_cache_scatter into per-sequence caches (k_ptrs / v_ptrs as for
 * attn_decode_batched_ptrs; a NULL or misaligned entry skips that sequence's
 * tokens and raises RKV_FLAG_BAD_POINTER).  Everything else as kv_cache_scatter.
 */
rkv_status kv_cache_scatter_ptrs(const float* k_new, const float* v_new, float* const* k_ptrs,
                                 float* const* v_ptrs, int M, int T, int n_kv_heads, int head_dim,
                                 int max_len, const int* start_pos, int* overflow,
                                 cudaStream_t stream);

/*
 * Appends T new K/V rows per sequence into the resident cache.
 *
 * Cites: trueno-gpu attention.rs, fn kv_cache_scatter_gpu (interleaved
 * [n_heads*head_dim] row -> cache[head, pos, :], position must be below
 * max_seq_len); batched layout from realizar fn init_batched_kv_cache_gpu.
 *
 *   k_new, v_new      [M, T, n_kv_heads*head_dim]        input
 *   k_cache, v_cache  [M, n_kv_heads, max_len, head_dim] updated in place:
 *       cache[m, kh, start_pos[m] + t, :] = new[m, t, kh*head_dim : (kh+1)*head_dim]
 *   start_pos  device int32[M]
 *   overflow   device int32*, or NULL.  Tokens whose target row is outside
 *              [0, max_len) are skipped and each is added once to *overflow
 *              (the page's host-side pos < max_seq_len check, moved on chip
 *              because positions live in device memory).
 * Bit-exact copy; rows not targeted are untouched.  1 <= M <= 32, T <= max_len.
 */
rkv_status kv_cache_scatter(const float* k_new, const float* v_new, float* k_cache,
                            float* v_cache, int M, int T, int n_kv_heads, int head_dim,
                            int max_len, const int* start_pos, int* overflow,
                            cudaStream_t stream);

/*
 * Rotary position embedding fused with the append: the prologue of a decode
 * step (T = 1) or of a prefill (T = S) in one pass.
 *
 * Cites: trustformers-core attention.rs, fn rope_neox_gpu_to_gpu (GPT-NeoX
 * half-split partial RoPE over the first rotary_ndims dims of each head, at an
 * absolute position offset) and realizar cache_from_cache_from_kv_cache.rs,
 * fn apply_rope_to_buffer (pair (i, i + half), frequency theta^(-2i/dim),
 * x1' = x1 cos - x2 sin, x2' = x1 sin + x2 cos); the append as kv_cache_scatter.
 *
 * For every sequence m and token t, at position p = start_pos[m] + t:
 *   q      [M, T, n_heads*head_dim]     rotated in place at p (every head)
 *   k_new  [M, T, n_kv_heads*head_dim]  rotated in place at p
 *   v_new  [M, T, n_kv_heads*head_dim]  input
 *   k_cache, v_cache [M, n_kv_heads, max_len, head_dim]: row p receives the
 *          rotated k and the v row (tokens with p outside [0, max_len) are not
 *          written and are counted once each in *overflow, if not NULL)
 * Pair i < rotary_ndims/2 joins dims i and i + rotary_ndims/2 of a head and turns
 * by p * theta^(-2i/rotary_ndims); dims rotary_ndims.. are unchanged.  The angle
 * is formed and reduced mod 2*pi in double (frequencies from the host), then
 * sincosf.  A negative p raises RKV_FLAG_NEGATIVE_INPUT and rotates as p = 0.
 * 0 <= M <= 32, T <= max_len, rotary_ndims even in (0, head_dim] (a multiple of
 * 8 is required: RKV_ERR_UNSUPPORTED otherwise), theta > 0; the five tensors
 * must be distinct.  A decode step is kv_append_rope(T = 1, start_pos = len-1)
 * then attn_decode_batched with lens; a prefill is kv_append_rope(T = S,
 * start_pos = 0) then attn_prefill on the rotated q, k (or attn_prefill_chunked
 * from the cache).
 */
rkv_status kv_append_rope(float* q, float* k_new, const float* v_new, float* k_cache,
                          float* v_cache, int M, int T, int n_heads, int n_kv_heads,
                          int head_dim, int max_len, const int* start_pos, int rotary_ndims,
                          float theta, int* overflow, cudaStream_t stream);

#ifdef __cplusplus
}
#endif

#endif /* RKV_ATTN_H */
