/*
 * pa.h -- C ABI of the paged KV-cache decode-attention library (libpa.so).
 *
 * Decode-time attention over a paged KV cache, for NVIDIA GB300 (sm_103a):
 *
 *   pa_reshape_and_cache  scatter each new token's key/value into the pool
 *   pa_decode             one-pass paged decode attention
 *   pa_decode_splitk      partitioned decode attention + log-sum-exp reduce
 *   pa_copy_blocks        copy whole blocks (the device half of copy-on-write)
 *   pa_prefill            prefill / chunked prefill attention over the pool
 *   pa_decode_splitk_lse  split-K decode that also returns the log-sum-exps
 *   pa_merge_attn_states  merge two partial attention results
 *   pa_cascade_decode     decode for sequences sharing a prefix (cascade)
 *   pa_*_fp8              the cache write and decode with an FP8 (e4m3) pool
 *   pa_stage_copy         move a step's data between pinned host memory and
 *                         the device on the SMs
 *
 * Data layout (all tensors contiguous, row-major, caller-owned):
 *
 *   kv_cache      [2, num_blocks, block_size, num_kv_heads, head_size]
 *                 index 0 holds keys, index 1 values ("PagedAttention 在 vLLM
 *                 中的实现分析", section 3.3 "KV Cache 布局", the NHD layout).
 *   block_tables  int32 [num_seqs, max_blocks_per_seq]; entry j of row s is the
 *                 physical block holding tokens [j*block_size, (j+1)*block_size)
 *                 of sequence s (same page, section 3.1; "Paged attention",
 *                 k4i.top, section "block table").  Entries past a sequence's
 *                 last block are never read.
 *   seq_lens      int32 [num_seqs]; number of cached tokens of each sequence,
 *                 the token just written included.
 *   slot_mapping  int64 [num_tokens]; slot = block_number * block_size +
 *                 block_offset; a negative slot marks a padding token that is
 *                 skipped (same page, section 3.2 "Slot Mapping").
 *   q, out        [num_seqs, num_heads, head_size]; one query token per
 *                 sequence (same page, section 7.2, stage 5 output shape).
 *
 * Grouped-query attention: query head h reads kv head h / (num_heads /
 * num_kv_heads).
 *
 * Conventions for every entry point:
 *   - Tensor arguments are DEVICE pointers on the current CUDA device, 16-byte
 *     aligned.  The library never takes ownership and never frees them.
 *   - `stream` is a cudaStream_t passed as void* (NULL = the legacy default
 *     stream).  Calls only enqueue work on it and return; results are ready
 *     once the stream reaches that point.
 *   - The library allocates no device memory.  The split-K path uses a
 *     workspace the caller provides.
 *   - Arguments are checked on the host before any launch.  Bad arguments
 *     return PA_ERR_INVALID_ARG, shapes outside the supported set return
 *     PA_ERR_UNSUPPORTED, and nothing is launched in either case.
 *     PA_ERR_CUDA reports a failed launch (the CUDA error is left for the
 *     caller's next cudaGetLastError/synchronize).
 *   - Supported: head_size in {64, 128}; block_size in {16, 32};
 *     num_heads / num_kv_heads in {1, 2, 4, 8}; fp16 or bf16 for q, cache and
 *     out alike.
 *   - Device-side guards: a block id outside [0, num_blocks), a seq_len
 *     outside [0, max_blocks_per_seq*block_size] (or, for split-K, above
 *     max_seq_len), or a slot at or beyond num_blocks*block_size is never
 *     dereferenced.  The kernel skips it (ids read as zeros, lengths are
 *     clamped, slots write nothing) and sets a bit in a sticky per-device
 *     error word that pa_device_errors reads.  Kernels never trap.
 *   - Every wait inside a kernel is bounded; a wait that runs out sets
 *     PA_DEVERR_TIMEOUT and the kernel returns.  A timeout is a device-side
 *     event that happens after the call has returned, so it has no status
 *     code of its own: it is reported by the sticky word, like the other
 *     device-side guards.
 */
#ifndef PA_H
#define PA_H

#include <stddef.h>
#include <stdint.h>

#ifdef __cplusplus
extern "C" {
#endif

typedef enum pa_status {
    PA_OK = 0,
    PA_ERR_INVALID_ARG = 1, /* null pointer, bad size, misaligned pointer */
    PA_ERR_UNSUPPORTED = 2, /* head_size / block_size / group size not built */
    PA_ERR_WORKSPACE = 3,   /* split-K workspace missing or too small */
    PA_ERR_CUDA = 4,        /* a CUDA runtime/driver call or launch failed */
    PA_ERR_OUT_OF_RANGE = 5 /* host validation found a bad id/length/slot */
} pa_status;

typedef enum pa_dtype { PA_FP16 = 0, PA_BF16 = 1 } pa_dtype;

/* Bits of the sticky device error word (pa_device_errors). */
#define PA_DEVERR_BLOCK_ID 0x1u /* a block id outside [0, num_blocks) */
#define PA_DEVERR_SEQ_LEN 0x2u  /* a seq_len outside its allowed range */
#define PA_DEVERR_SLOT 0x4u     /* a slot >= num_blocks * block_size */
#define PA_DEVERR_TIMEOUT 0x8u  /* a bounded in-kernel wait ran out */
#define PA_DEVERR_PREFIX 0x10u  /* cascade: a table does not start with the shared
                                   prefix blocks, or a seq_len is shorter than it */

/*
 * Write new tokens into the pool ("PagedAttention 在 vLLM 中的实现分析",
 * sections 3.2 and 7.4: for each token, slot = slot_mapping[token]; if
 * slot >= 0, key[token] goes to key_cache[slot] and value[token] to
 * value_cache[slot]).
 *
 *   key, value    [num_tokens, num_kv_heads, head_size] rows; row i starts
 *                 at key + i*key_stride elements (key_stride >=
 *                 num_kv_heads*head_size, multiple of 8), likewise value.
 *   kv_cache      the pool, updated in place at block slot / block_size,
 *                 offset slot % block_size.  Bytes are copied unchanged.
 *   slot_mapping  int64 [num_tokens]; negative = padding, nothing written.
 *                 Two tokens must not share a non-negative slot.
 * num_tokens == 0 is a no-op.
 */
pa_status pa_reshape_and_cache(const void *key, const void *value, void *kv_cache,
                               const int64_t *slot_mapping, int num_tokens,
                               int num_kv_heads, int head_size, int block_size,
                               int num_blocks, int64_t key_stride, int64_t value_stride,
                               pa_dtype dtype, void *stream);

/*
 * One-pass paged decode attention.  For every sequence s and query head h:
 *   out[s,h,:] = sum_t softmax_t(scale * q[s,h,:] . K_t) V_t  over the
 * sequence's tokens t < seq_lens[s], with K_t/V_t found through the block
 * table ("Paged attention", k4i.top, section "对非连续 blocks 做 attention":
 * blocks gathered through the table, softmax merged block by block online,
 * equal to softmax over the whole sequence).  seq_lens[s] == 0 gives a zero
 * row.  Accumulation is fp32; out is rounded to the input dtype (nearest
 * even).
 */
pa_status pa_decode(void *out, const void *q, const void *kv_cache,
                    const int32_t *block_tables, const int32_t *seq_lens, int num_seqs,
                    int num_heads, int num_kv_heads, int head_size, int block_size,
                    int num_blocks, int max_blocks_per_seq, float scale, pa_dtype dtype,
                    void *stream);

/*
 * Bytes of workspace pa_decode_splitk needs for these sizes: a work-list
 * header, one list entry per (sequence, partition), and the partial states
 * (running max, normaliser, unnormalised head_size-vector, fp32) for every
 * (sequence, query head, partition), partitions = ceil(max_seq_len /
 * partition_size).  Returns 0 for invalid sizes.
 */
size_t pa_decode_splitk_workspace_size(int num_seqs, int num_heads, int head_size,
                                       int max_seq_len, int partition_size);

/*
 * Partitioned ("V2") paged decode attention ("PagedAttention 在 vLLM 中的实现
 * 分析", section 7.3: each sequence's tokens are cut into partitions of
 * partition_size tokens that are processed independently, then merged by
 * rescaling with the online-softmax correction).  Same result as pa_decode
 * within fp32 rounding.  Arguments as pa_decode, plus:
 *   max_seq_len     upper bound on every seq_lens[s] (sizes the workspace)
 *   partition_size  tokens per partition, a positive multiple of 64 (512 is
 *                   the pages' choice)
 *   workspace       device buffer of at least
 *                   pa_decode_splitk_workspace_size(...) bytes, 256-byte
 *                   aligned; its contents on entry do not matter and it is
 *                   scratch after return.  Calls that overlap in time must
 *                   not share a workspace.
 */
pa_status pa_decode_splitk(void *out, const void *q, const void *kv_cache,
                           const int32_t *block_tables, const int32_t *seq_lens, int num_seqs,
                           int num_heads, int num_kv_heads, int head_size, int block_size,
                           int num_blocks, int max_blocks_per_seq, float scale,
                           pa_dtype dtype, int max_seq_len, int partition_size,
                           void *workspace, size_t workspace_bytes, void *stream);

/*
 * pa_decode_splitk without a caller-provided workspace, for callers that
 * cannot allocate device memory (for example code hosted inside a framework
 * that owns all device memory and gives it no allocator, or a latency-critical
 * loop where an allocation, which may synchronise the device, is not
 * allowed).  The pages have no counterpart of this entry point.
 *
 * Arguments and result are those of pa_decode_splitk.  Its scratch is a fixed
 * array of PA_NOALLOC_SCRATCH_BYTES inside the library; the call allocates
 * nothing.  Sizes whose pa_decode_splitk_workspace_size exceeds that return
 * PA_ERR_WORKSPACE before any launch.
 *   - The array occupies PA_NOALLOC_SCRATCH_BYTES of device memory on every
 *     GPU where the library's module is loaded, until the process exits.
 *   - The first call on a device looks up the array's device address and
 *     caches it for that device and its current driver context; make that
 *     first call before any stream capture.  After cudaDeviceReset, or from
 *     another driver context on the same device, the array is a new one and
 *     its address is looked up again on the next call, which should then
 *     also come before any capture.
 *   - All calls on one device share the array.  Calls that overlap on the GPU
 *     race; order them (one stream, or events).  Nothing in the array needs
 *     to start at zero.
 */
#define PA_NOALLOC_SCRATCH_BYTES (16u << 20)

pa_status pa_decode_splitk_noalloc(void *out, const void *q, const void *kv_cache,
                                   const int32_t *block_tables, const int32_t *seq_lens,
                                   int num_seqs, int num_heads, int num_kv_heads, int head_size,
                                   int block_size, int num_blocks, int max_blocks_per_seq,
                                   float scale, pa_dtype dtype, int max_seq_len,
                                   int partition_size, void *stream);

/*
 * FP8 KV cache ("PagedAttention 在 vLLM 中的实现分析", section 6.3: with an
 * FP8 cache dtype the cache write converts K/V using k_scale / v_scale).  The
 * pool is uint8 [2, num_blocks, block_size, num_kv_heads, head_size] of e4m3
 * codes (1 sign, 4 exponent bits with bias 7, 3 fraction bits; 0x7F/0xFF are
 * NaN; largest magnitude 448).  head_size 128.
 *
 * pa_reshape_and_cache_fp8: for token i with slot_mapping[i] >= 0 the codes
 *   e4m3(fp32(key[i][..] / k_scale)) and e4m3(fp32(value[i][..] / v_scale))
 *   go to pool row `slot`, rounded to nearest (ties to even), magnitudes
 *   above 448 saturating to 448.  key/value are src_dtype rows as in
 *   pa_reshape_and_cache (strides multiples of 8 elements); k_scale and
 *   v_scale are positive finite floats.  Slots past the pool are skipped and
 *   flagged (PA_DEVERR_SLOT).
 * pa_decode_fp8 / pa_decode_splitk_fp8: pa_decode / pa_decode_splitk over
 *   keys k_scale * e4m3(K) and values v_scale * e4m3(V); q and out are
 *   `dtype`.  The split-K call runs on the tensor cores (kind::f8f6f4, the
 *   query carried as three e4m3 parts with a row scale) and needs
 *   pa_decode_splitk_fp8_workspace_size bytes of workspace (256-byte
 *   aligned); the one-pass call runs on the CUDA cores and needs none.
 */
size_t pa_decode_splitk_fp8_workspace_size(int num_seqs, int num_heads, int head_size,
                                           int max_seq_len, int partition_size);
pa_status pa_reshape_and_cache_fp8(const void *key, const void *value, void *kv_cache,
                                   const int64_t *slot_mapping, int num_tokens, int num_kv_heads,
                                   int head_size, int block_size, int num_blocks,
                                   int64_t key_stride, int64_t value_stride, pa_dtype src_dtype,
                                   float k_scale, float v_scale, void *stream);
pa_status pa_decode_fp8(void *out, const void *q, const void *kv_cache,
                        const int32_t *block_tables, const int32_t *seq_lens, int num_seqs,
                        int num_heads, int num_kv_heads, int head_size, int block_size,
                        int num_blocks, int max_blocks_per_seq, float scale, float k_scale,
                        float v_scale, pa_dtype dtype, void *stream);
pa_status pa_decode_splitk_fp8(void *out, const void *q, const void *kv_cache,
                               const int32_t *block_tables, const int32_t *seq_lens,
                               int num_seqs, int num_heads, int num_kv_heads, int head_size,
                               int block_size, int num_blocks, int max_blocks_per_seq,
                               float scale, float k_scale, float v_scale, pa_dtype dtype,
                               int max_seq_len, int partition_size, void *workspace,
                               size_t workspace_bytes, void *stream);

/*
 * pa_decode_splitk that also writes each row's log-sum-exp: lse[s][h] =
 * log sum_t exp(scale * q . k_t), natural log, float32 [num_seqs, num_heads]
 * (-inf for an empty sequence).  The pieces of a cascade are merged with it
 * (pa_merge_attn_states).  Arguments and errors as pa_decode_splitk; lse must
 * be non-NULL and 4-byte aligned.
 */
pa_status pa_decode_splitk_lse(void *out, float *lse, const void *q, const void *kv_cache,
                               const int32_t *block_tables, const int32_t *seq_lens,
                               int num_seqs, int num_heads, int num_kv_heads, int head_size,
                               int block_size, int num_blocks, int max_blocks_per_seq,
                               float scale, pa_dtype dtype, int max_seq_len, int partition_size,
                               void *workspace, size_t workspace_bytes, void *stream);

/*
 * Merge two attention results over disjoint key sets ("PagedAttention 在 vLLM
 * 中的实现分析", section 6.4, merge_attn_states: the online-softmax
 * correction).  Per row (token, head), with M = max(lse_a, lse_b) and
 * w_x = exp(lse_x - M):
 *   out = (w_a o_a + w_b o_b) / (w_a + w_b),  out_lse = M + log(w_a + w_b).
 * A row whose lse is -inf is an empty part; two empty parts give 0 and -inf.
 *   out, o_a, o_b   [num_tokens, num_heads, head_size], dtype, 16-byte aligned
 *                   (out may alias o_a or o_b).
 *   lse_a, lse_b    float32 [num_tokens, num_heads]; out_lse the same or NULL.
 * head_size 64 or 128.
 */
pa_status pa_merge_attn_states(void *out, float *out_lse, const void *o_a, const float *lse_a,
                               const void *o_b, const float *lse_b, int num_tokens,
                               int num_heads, int head_size, pa_dtype dtype, void *stream);

/*
 * Workspace bytes of pa_cascade_decode for these sizes (0 on bad sizes).
 */
size_t pa_cascade_decode_workspace_size(int num_seqs, int num_heads, int head_size,
                                        int max_blocks_per_seq, int prefix_blocks,
                                        int max_seq_len, int block_size, int partition_size);

/*
 * Cascade decode attention for sequences that share a prefix ("PagedAttention
 * 在 vLLM 中的实现分析", section 6.4: the common prefix is attended once,
 * without the causal mask, for all requests; each request's own suffix
 * separately; merge_attn_states combines them).  The result equals
 * pa_decode over the full tables.
 *
 * The first prefix_blocks entries of every block_tables row must be the same
 * physical blocks (row 0's), and every seq_len >= prefix_blocks * block_size;
 * a table or length that breaks this is flagged (PA_DEVERR_PREFIX) and its
 * output is not defined.  Steps: one prefill pass of the B queries over the
 * prefix (tensor cores); a setup kernel (suffix lengths and tables) and a
 * split-K decode of the suffixes with log-sum-exp; the merge.  The prefix
 * pass runs on a stream of the library's own (one per host thread and
 * device, created on the first call outside a graph capture, at the
 * device's highest stream priority), forked from `stream` when the call
 * starts and joined back into it before the merge, so that the two passes
 * share the SMs; the call stays ordered on `stream` like any other work
 * (and can be captured into a graph).  Without that stream (its creation
 * failed, or the first call comes inside a capture) every step runs on
 * `stream`.  prefix_blocks == 0 is plain pa_decode_splitk.  Other
 * arguments, layouts and errors as pa_decode_splitk; the workspace must hold
 * pa_cascade_decode_workspace_size bytes, 256-byte aligned.
 */
pa_status pa_cascade_decode(void *out, const void *q, const void *kv_cache,
                            const int32_t *block_tables, const int32_t *seq_lens, int num_seqs,
                            int num_heads, int num_kv_heads, int head_size, int block_size,
                            int num_blocks, int max_blocks_per_seq, int prefix_blocks,
                            float scale, pa_dtype dtype, int max_seq_len, int partition_size,
                            void *workspace, size_t workspace_bytes, void *stream);

/*
 * Prefill / chunked prefill over the paged cache ("PagedAttention 在 vLLM 中的
 * 实现分析", section 6.2: the FlashAttention backend attends the batch's new
 * query tokens, packed by query_start_loc, to each request's paged keys with
 * seqlen_k = seq_lens, the block table and causal masking; section 6.4: the
 * shared-prefix pass of cascade attention is the same call without the
 * causal mask).  On the tensor cores (tcgen05).
 *
 *   out              [num_tokens, num_heads, head_size], dtype; rows of tokens
 *                    outside every request's range are left untouched.
 *   lse              NULL, or float32 [num_tokens, num_heads]: the natural log
 *                    of each row's softmax denominator, log sum_t exp(scale q.k_t).
 *   q                [num_tokens, num_heads, head_size], dtype.  The q_len =
 *                    query_start_loc[r+1] - query_start_loc[r] rows of request
 *                    r are its last q_len tokens: row i sits at position
 *                    seq_lens[r] - q_len + i, and its keys/values must already
 *                    be in the pool (pa_reshape_and_cache first).
 *   kv_cache         the pool [2, num_blocks, block_size, num_kv_heads, head_size].
 *   block_tables     int32, row r at block_tables + r * block_table_stride,
 *                    its first ceil(seq_lens[r] / block_size) entries used
 *                    (max_blocks_per_seq <= block_table_stride entries per row).
 *   seq_lens         int32 [num_reqs]: cached tokens of request r, the new
 *                    ones included (q_len <= seq_len).
 *   query_start_loc  int32 [num_reqs + 1], non-decreasing, from 0 to at most
 *                    num_tokens.
 *   max_query_len    an upper bound of every q_len (sets the grid).
 *   causal           1: position p attends keys 0..p; 0: every key of the
 *                    request.
 * Query head h reads kv head h / (num_heads / num_kv_heads).  head_size 64
 * or 128, block_size 16 or 32.  A request whose metadata breaks these rules
 * (q_len < 0 or > max_query_len, seq_len < q_len or beyond its table,
 * query_start_loc outside [0, num_tokens]) is skipped and flagged
 * (PA_DEVERR_SEQ_LEN); block ids outside the pool read zeros and are flagged
 * (PA_DEVERR_BLOCK_ID).
 */
pa_status pa_prefill(void *out, float *lse, const void *q, const void *kv_cache,
                     const int32_t *block_tables, int64_t block_table_stride,
                     const int32_t *seq_lens, const int32_t *query_start_loc, int num_reqs,
                     int num_tokens, int max_query_len, int num_heads, int num_kv_heads,
                     int head_size, int block_size, int num_blocks, int max_blocks_per_seq,
                     float scale, int causal, pa_dtype dtype, void *stream);

/*
 * Copy whole blocks of the pool, for copy-on-write (k4i.top "paged
 * attention" explainer, section on copy-on-write in parallel sampling and its
 * Figure 3; the ATB PagedAttention blog's Copy-on-Write section: when a
 * sequence must write into a block it shares, a fresh block receives a copy of
 * the shared block, the sequence's table is repointed to it, and the new token
 * is written there).
 *
 *   kv_cache       the pool, updated in place: for each pair i, the key rows
 *                  and the value rows of block block_mapping[2i] are copied
 *                  into block block_mapping[2i+1].
 *   block_mapping  int64 [num_pairs, 2] (src, dst), device memory.  No dst
 *                  may repeat or also appear as a src in the same call (the
 *                  pairs are copied concurrently); pa_validate_block_mapping
 *                  checks this on a host copy.  Ids outside [0, num_blocks)
 *                  are skipped and flagged (PA_DEVERR_BLOCK_ID).
 * num_pairs == 0 is a no-op; num_pairs <= 65535.
 */

pa_status pa_copy_blocks(void *kv_cache, const int64_t *block_mapping, int num_pairs,
                         int num_blocks, int block_size, int num_kv_heads, int head_size,
                         pa_dtype dtype, void *stream);

/*
 * Copy bytes from src to dst on the GPU's SMs (16-byte moves), stream-
 * ordered on stream.  Either pointer may be device memory or pinned host
 * memory with a device mapping (page-locked by the CUDA runtime, for example
 * through cudaHostAlloc); the SMs then read or write the host memory directly
 * over the host link, which for the few MB of a decode step's inputs and
 * outputs is faster than a copy-engine transfer.  Pointers without a device
 * mapping, or not 16-byte aligned, or a size that is not a multiple of 16,
 * are handed to cudaMemcpyAsync (cudaMemcpyDefault) instead.  src and dst
 * must not overlap; both stay owned by the caller.  The pages have no
 * counterpart of this call: it stages a step's data.
 * Errors: PA_ERR_INVALID_ARG for a null pointer with bytes > 0; PA_ERR_CUDA
 * for a failed launch or copy.
 */
pa_status pa_stage_copy(void *dst, const void *src, size_t bytes, void *stream);

/*
 * Host-side check of a HOST copy of a block mapping for pa_copy_blocks: ids in
 * [0, num_blocks), destinations distinct, no destination also a source.
 * Returns PA_OK, PA_ERR_OUT_OF_RANGE, or PA_ERR_INVALID_ARG.  No CUDA call.
 */
pa_status pa_validate_block_mapping(const int64_t *block_mapping, int num_pairs,
                                    int num_blocks);

/*
 * Host-side check of the decode preconditions on HOST copies of the tables:
 * 0 <= seq_lens[s] <= max_blocks_per_seq*block_size and every block id a
 * sequence uses (entries j < ceil(seq_lens[s]/block_size)) in [0, num_blocks).
 * Returns PA_OK, PA_ERR_OUT_OF_RANGE, or PA_ERR_INVALID_ARG.  No CUDA call.
 */
pa_status pa_validate_tables(const int32_t *block_tables, const int32_t *seq_lens,
                             int num_seqs, int max_blocks_per_seq, int block_size,
                             int num_blocks);

/*
 * Host-side check of a HOST copy of slot_mapping: every non-negative slot
 * below num_blocks*block_size and no slot used twice.  Returns PA_OK,
 * PA_ERR_OUT_OF_RANGE, or PA_ERR_INVALID_ARG.  No CUDA call.
 */
pa_status pa_validate_slots(const int64_t *slot_mapping, int num_tokens, int block_size,
                            int num_blocks);

/*
 * Read (and with clear != 0, reset) the current device's sticky error word
 * (PA_DEVERR_* bits).  Synchronises the device.  Returns PA_ERR_CUDA if the
 * read fails.
 */
pa_status pa_device_errors(unsigned int *flags, int clear);

/*
 * Self-test of the in-kernel failure detection: launches one thread that
 * waits on a barrier phase nothing will complete.  The wait gives up after
 * its time limit (about 2 s), the kernel sets PA_DEVERR_TIMEOUT in the device
 * error word and returns; the CUDA context stays usable.  No counterpart on
 * the pages (it checks the library's own bounded-wait rule).
 */
pa_status pa_selftest_wait_timeout(void *stream);

/*
 * Measurement aid.  For every later decode call made by the calling host
 * thread (pa_decode, pa_decode_splitk, pa_decode_splitk_lse,
 * pa_decode_splitk_noalloc and the FP8 decodes), record the CUDA event
 * `before` on the call's stream just before its main attention kernel is
 * launched and `after` just after, so that the elapsed time between them is
 * that kernel's alone (the split-K plan and reduce kernels fall outside).
 * Both are cudaEvent_t passed as void*, created and owned by the caller, and
 * must stay valid while set; (NULL, NULL) turns the recording off, one NULL
 * alone is PA_ERR_INVALID_ARG.  While set, the main kernel no longer
 * overlaps its launch with the kernel before it.  No counterpart on the
 * pages: it serves the library's own roofline measurement.
 */
pa_status pa_profile_kernel_events(void *before, void *after);

/* Static, human-readable name of a status code. */
const char *pa_status_string(pa_status status);

/* Library ABI version (major*10000 + minor*100 + patch). */
int pa_version(void);

#ifdef __cplusplus
}
#endif

#endif /* PA_H */
