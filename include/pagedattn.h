/*
 * libpagedattn -- paged KV cache decode path for NVIDIA GB300 (sm_103a).
 *
 * C ABI. Plain pointers and sizes only; no exceptions cross this boundary.
 * Every entry point returns an int status (PA_OK = 0, negative on error).
 *
 * Sources (web pages, by title and section):
 *  [P1] "PagedAttention实现" (ainanfeng.cn teaching version), sections
 *       "Block定义" (one physical block holds block_size tokens' K and V),
 *       "页表" (a per-sequence logical->physical block list) and
 *       "PagedAttention管理器" (free list, reference counts, write_kv,
 *       cow_write, free_sequence).
 *  [P2] "CS349E lecture 7: 01_paged_attention.py", demo 1 (block-table
 *       growth), demo 2 (paper eq. 4: block-wise scores, one softmax over the
 *       whole context, block-wise V; equal to contiguous attention), demo 3
 *       (prefix sharing with copy-on-write).
 *  [P3] "04 - Paged Attention 实现进度", section A.2 (the five components) and
 *       B.2 (slot_mapping [total_tokens], block_tables
 *       [batch, max_blocks_per_seq], context_lens [batch]).
 *
 * Layouts (all row-major, C-contiguous):
 *   key_cache, value_cache : [num_blocks, block_size, num_kv_heads, head_dim]
 *   k, v (new tokens)      : [num_tokens, num_kv_heads, head_dim]
 *   q, out                 : [num_seqs, num_heads, head_dim]
 *   block_tables           : int32 [num_seqs, max_blocks_per_seq]
 *   context_lens           : int32 [num_seqs]
 *   slot_mapping           : int32 [num_tokens], slot = block * block_size + offset
 *   src_dst_pairs          : int32 [num_pairs, 2]
 * Query head h reads kv head h / (num_heads / num_kv_heads).
 *
 * Ownership and timing: the caller owns every buffer. Device pointers must be
 * 16-byte aligned. Compute calls are asynchronous on the caller's CUDA stream
 * (passed as void*, NULL = the legacy default stream); they validate shapes on
 * the host and never read device data on the host. Index errors found on the
 * device (a bad slot, block id, copy pair or context length) skip the bad
 * access and set a bit in a per-device error word, read and cleared by
 * pa_get_device_error(). No kernel traps or asserts.
 *
 * Launch chaining: the decode and merge kernels are launched as programmatic
 * dependents of the kernel before them on the stream, and the decode kernels read
 * context_lens (and prefix_lens) before they wait for it. A kernel the caller
 * launches just before a decode call therefore must not write those two arrays
 * after it signals its dependents early (griddepcontrol.launch_dependents); a
 * kernel that never signals is waited for in full, as usual.
 */
#ifndef PAGEDATTN_H
#define PAGEDATTN_H

#include <stddef.h>
#include <stdint.h>

#ifdef __cplusplus
extern "C" {
#endif

/* ---- status codes --------------------------------------------------------- */
#define PA_OK                 0
#define PA_ERR_INVALID_ARG   -1   /* bad shape, pointer, alignment or value      */
#define PA_ERR_UNSUPPORTED   -2   /* valid but not implemented (e.g. head_dim)   */
#define PA_ERR_OUT_OF_BLOCKS -3   /* allocator: free list too short              */
#define PA_ERR_CUDA          -4   /* a CUDA runtime call failed                  */
#define PA_ERR_DEVICE_INDEX  -5   /* pa_get_device_error: a device check fired   */
#define PA_ERR_UNKNOWN_SEQ   -6   /* allocator: no such sequence id              */
#define PA_ERR_WORKSPACE     -7   /* decode: workspace given but too small       */
#define PA_ERR_EXISTS        -8   /* allocator: sequence id already present      */

/* ---- element types -------------------------------------------------------- */
#define PA_DTYPE_F32  0
#define PA_DTYPE_F16  1
#define PA_DTYPE_BF16 2
#define PA_DTYPE_E4M3 3   /* 8-bit cache storage (see the _fp8 calls); also   */
                          /* accepted by pa_copy_blocks                        */

/* ---- device error bits (pa_get_device_error) ------------------------------ */
#define PA_DEVERR_SLOT       0x1u  /* slot not -1 and outside [0, NB*bs)          */
#define PA_DEVERR_BLOCK_ID   0x2u  /* live table entry outside [0, num_blocks)    */
#define PA_DEVERR_CONTEXT    0x4u  /* context_len < 0, > max_blocks_per_seq*bs,   */
                                   /* or > max_context_len                        */
#define PA_DEVERR_COPY_PAIR  0x8u  /* copy pair id outside [0, num_blocks)        */
#define PA_DEVERR_WAIT       0x10u /* an internal pipeline wait hit its bound     */

/* Name of a status code (static string). */
const char *pa_status_string(int status);

/* Library version, major*10000 + minor*100 + patch. */
int pa_version(void);

/*
 * Scatter new tokens' K and V rows into their cache slots.
 * [P1 write_kv: page = position / block_size, offset = position % block_size,
 *  then the token's values are copied; P3 B.2: slot_mapping]
 *
 * Token t's row k[t] (num_kv_heads*head_dim elements) is copied to
 * key_cache[slot / block_size, slot % block_size], and v[t] likewise, where
 * slot = slot_mapping[t]. slot == -1 skips the token (padding). Any other slot
 * outside [0, num_blocks*block_size) is skipped and sets PA_DEVERR_SLOT.
 * Two tokens with the same slot are a caller error (the survivor is undefined).
 * Requires num_kv_heads*head_dim*sizeof(dtype) to be a multiple of 16 bytes.
 */
int pa_paged_kv_write(const void *k, const void *v, const int32_t *slot_mapping,
                      int64_t num_tokens, void *key_cache, void *value_cache,
                      int64_t num_blocks, int block_size, int num_kv_heads, int head_dim,
                      int dtype, void *stream);

/*
 * Bytes of split-K workspace pa_paged_attention_decode needs for these sizes
 * (0 when every sequence fits one partition). partition_size 0 = automatic.
 */
size_t pa_decode_workspace_bytes(int num_seqs, int num_heads, int head_dim,
                                 int max_context_len, int partition_size);

/*
 * The partition size a decode call uses for these arguments: partition_size
 * itself when it is not 0, else the automatic choice -- 1024 tokens when
 * num_seqs * ceil(max_context_len / 1024) >= 64, otherwise 512 (small batches
 * keep more, shorter partitions to spread over the SMs). max_context_len is the
 * call's bound (max_blocks_per_seq * block_size when the call passes 0).
 * Applies to pa_paged_attention_decode, _append, _noalloc and the _fp8 calls;
 * the sharing-aware decode has its own rule (pa_decode_shared_partition_size).
 */
int pa_decode_partition_size(int num_seqs, int max_context_len, int partition_size);

/*
 * Single-query decode attention over the paged cache.
 * [P2 demo 2, eq. 4: for each sequence and query head, scores against every
 *  cached key are formed block by block through the block table, ONE softmax
 *  is taken over the whole context, and V is accumulated block by block;
 *  P3 B.2: block_tables, context_lens]
 *
 *   out[b,h,:] = sum_t softmax_t(scale * q[b,h,:] . K[b,t,h/G,:]) * V[b,t,h/G,:]
 *
 * over t < context_lens[b]; position t lives in physical block
 * block_tables[b, t / block_size] at offset t % block_size. Accumulation is
 * fp32; out has q's dtype. context_lens[b] == 0 gives a zero row.
 *
 * Long contexts are split into partitions of partition_size tokens
 * (0 = automatic, see pa_decode_partition_size; else a positive multiple of
 * 128). Each partition keeps its
 * running max, sum and unnormalised output in fp32 workspace, and a second
 * kernel merges them. max_context_len is a host-side upper bound on every
 * context_lens[b] (0 = max_blocks_per_seq * block_size); it sizes the grid
 * and the workspace. A context above it, or above max_blocks_per_seq *
 * block_size, or negative, sets PA_DEVERR_CONTEXT and is clamped to the
 * covered range; a live table entry outside [0, num_blocks) sets
 * PA_DEVERR_BLOCK_ID and that block reads as zeros.
 *
 * workspace: caller-owned device memory of workspace_bytes >=
 * pa_decode_workspace_bytes(...). When workspace is NULL and one is needed,
 * the library takes it with cudaMallocAsync on the stream and releases it with
 * cudaFreeAsync after the merge. Too small a workspace returns PA_ERR_WORKSPACE.
 *
 * Supported: dtype f32/f16/bf16 (q, caches and out share it), head_dim 64 or
 * 128, num_heads a multiple of num_kv_heads with num_heads/num_kv_heads <= 16,
 * block_size a power of two in [1, 256].
 */
int pa_paged_attention_decode(void *out, const void *q, const void *key_cache,
                              const void *value_cache, const int32_t *block_tables,
                              int max_blocks_per_seq, const int32_t *context_lens,
                              int num_seqs, int num_heads, int num_kv_heads, int head_dim,
                              int block_size, int64_t num_blocks, float scale,
                              int max_context_len, int partition_size, void *workspace,
                              size_t workspace_bytes, int dtype, void *stream);

/*
 * One decode step: pa_paged_kv_write of each sequence's new token, then
 * pa_paged_attention_decode. [P2 demo 1: a decode step writes the new token's
 * KV into its slot, then attends over the whole context, that token included;
 * P3 B.2: slot_mapping]
 *
 * k_new, v_new: [num_seqs, num_kv_heads, head_dim] in dtype (16-byte aligned),
 * the new token of sequence b in row b; slot_mapping[b]: its slot, which must be
 * the slot of position context_lens[b] - 1 (block_tables[b, (ctx - 1) /
 * block_size] * block_size + (ctx - 1) % block_size), or -1 for no write (the
 * only value allowed for an empty context). The other arguments, the result
 * and the workspace rules are those of pa_paged_attention_decode, and the
 * caches end as after pa_paged_kv_write.
 *
 * Where the tensor-core decode takes the call, it writes each token itself,
 * before it reads that token's block, instead of a separate scatter launch; a
 * slot other than that of position ctx - 1 then sets PA_DEVERR_SLOT and is not
 * written. The block holding a sequence's new token must not be read by another
 * sequence of the same call (copy-on-write guarantees it). Elsewhere the scatter
 * runs first, as its own launch.
 */
int pa_paged_attention_decode_append(void *out, const void *q, const void *k_new, const void *v_new,
                                     const int32_t *slot_mapping, void *key_cache, void *value_cache,
                                     const int32_t *block_tables, int max_blocks_per_seq,
                                     const int32_t *context_lens, int num_seqs, int num_heads, int num_kv_heads,
                                     int head_dim, int block_size, int64_t num_blocks, float scale,
                                     int max_context_len, int partition_size, void *workspace,
                                     size_t workspace_bytes, int dtype, void *stream);

/*
 * Decode attention that reads each shared prefix once for all sequences that
 * share it.
 * [P2 demo 3: forked samples share the prompt's blocks by reference count;
 *  P3 A.1/B.1: several block tables may point at the same physical blocks
 *  (prefix sharing)]
 *
 * Same result as pa_paged_attention_decode. group_members[g, 0..max_members)
 * lists the sequences of group g (-1 = empty slot, members first); a sequence
 * belongs to at most one group. prefix_lens[b] is the number of leading tokens
 * sequence b shares with its group (0 outside groups); all members of a group
 * must have the same prefix_lens and identical block-table entries for those
 * tokens (pa_prefix_groups derives such groups from the tables). The shared
 * tokens of a group are read once, through the first member's table, for all
 * members' queries together; each sequence's remaining tokens are read as in
 * pa_paged_attention_decode; the split-K merge combines both. max_prefix_len
 * is a host-side bound on prefix_lens. max_members * G' <= 128 (G' = group size
 * num_heads/num_kv_heads rounded up to a power of two).
 *
 * Supported: dtype f16/bf16, head_dim 128, num_heads/num_kv_heads <= 16,
 * block_size a power of two in [8, 128], scale > 0. workspace >=
 * pa_decode_shared_workspace_bytes(...) bytes (NULL: taken with cudaMallocAsync
 * on the stream and released after the merge). partition_size 0 = automatic
 * (pa_decode_shared_partition_size); the shared and the per-sequence tokens use
 * the same partition size.
 */
size_t pa_decode_shared_workspace_bytes(int num_seqs, int num_heads, int head_dim,
                                        int max_context_len, int partition_size);

/*
 * The partition size a sharing-aware decode call uses: partition_size itself
 * when it is not 0, else the multiple of 128 (at least 512, at most the longest
 * shared prefix rounded up) that minimises an estimate of the shared pass's time
 * on this device: ceil(items / SMs) x (128-key tiles per item + 1.4), items =
 * num_groups x num_kv_heads x ceil(max_prefix_len / partition); ties go to the
 * larger partition. When that holds each shared prefix in one partition, the
 * result grows to max_context_len rounded up to 128 if that is at most 8192 and
 * num_seqs x num_kv_heads >= 2 x SMs. With no groups or no shared tokens it is
 * 512. max_context_len: the call's bound (max_blocks_per_seq * block_size when the
 * call passes 0). A call whose partition is >= that bound (with at most 8 query
 * heads per kv head) runs no merge: the per-sequence pass joins the shared
 * partial itself. Workspace sized by
 * pa_decode_shared_workspace_bytes(..., 0) covers every automatic choice. Reads
 * the current device's SM count (152 when it cannot be read).
 */
int pa_decode_shared_partition_size(int num_seqs, int num_groups, int num_kv_heads, int max_prefix_len,
                                    int max_context_len, int partition_size);

int pa_paged_attention_decode_shared(void *out, const void *q, const void *key_cache,
                                     const void *value_cache, const int32_t *block_tables,
                                     int max_blocks_per_seq, const int32_t *context_lens,
                                     const int32_t *prefix_lens, const int32_t *group_members,
                                     int num_groups, int max_members, int max_prefix_len,
                                     int num_seqs, int num_heads, int num_kv_heads, int head_dim,
                                     int block_size, int64_t num_blocks, float scale,
                                     int max_context_len, int partition_size, void *workspace,
                                     size_t workspace_bytes, int dtype, void *stream);

/*
 * Chunked-prefill attention over the paged cache.
 * [P2 demo 1 and demo 2: a paged step writes the chunk's K/V into its blocks,
 *  then every position of the chunk attends to the positions up to its own;
 *  P3 B.2 and D.2: cu_seqlens_q (query_start_loc) packs the chunks of a batch]
 *
 * Sequence b owns query rows query_start_loc[b] .. query_start_loc[b+1]-1 of
 * q and out ([num_query_tokens, num_heads, head_dim]); q_len_b is their count.
 * Its context holds context_lens[b] tokens whose last q_len_b are the chunk
 * (already written, e.g. with pa_paged_kv_write). Row i sits at position
 * pos = context_lens[b] - q_len_b + i and
 *
 *   out[row, h, :] = sum_{t <= pos} softmax_t(scale * q[row, h, :] . K[b,t,h/G,:]) V[b,t,h/G,:].
 *
 * Accumulation is fp32 (probabilities rounded to the cache type for the
 * P.V product). max_query_len is a host-side bound on every q_len_b; it sizes
 * the grid. A sequence with q_len_b < 0, q_len_b > max_query_len,
 * q_len_b > context_lens[b], context_lens[b] > max_blocks_per_seq*block_size,
 * or rows outside [0, num_query_tokens) sets PA_DEVERR_CONTEXT and its rows are
 * left unwritten; a live table entry outside [0, num_blocks) sets
 * PA_DEVERR_BLOCK_ID and reads as zeros.
 *
 * Supported: dtype f16/bf16, head_dim 128, num_heads/num_kv_heads <= 16,
 * block_size a power of two in [8, 128]; else PA_ERR_UNSUPPORTED. scale must
 * be positive (PA_ERR_INVALID_ARG otherwise). Allocates nothing.
 */
int pa_paged_attention_prefill(void *out, const void *q, const void *key_cache,
                               const void *value_cache, const int32_t *block_tables,
                               int max_blocks_per_seq, const int32_t *context_lens,
                               const int32_t *query_start_loc, int num_seqs,
                               int64_t num_query_tokens, int max_query_len, int num_heads,
                               int num_kv_heads, int head_dim, int block_size,
                               int64_t num_blocks, float scale, int dtype, void *stream);

/*
 * Decode attention that allocates no device memory. The paper has no
 * counterpart to this entry point; it exists for callers, not for the method.
 *
 * Same computation, arguments and results as pa_paged_attention_decode, minus
 * the workspace. It is meant for callers that can neither allocate device
 * memory nor lend a buffer: for example a process whose device memory belongs to
 * a host runtime that forbids libraries to allocate, or a serving loop that
 * cannot afford an allocation on its critical path. The split-K scratch comes
 * from a fixed array of PA_NOALLOC_SCRATCH_BYTES inside this library, which every
 * GPU that loads the library holds until the process exits; no call allocates
 * or frees anything.
 *
 * Limit: when pa_decode_workspace_bytes(num_seqs, num_heads, head_dim,
 * max_context_len or max_blocks_per_seq*block_size, partition_size) exceeds
 * PA_NOALLOC_SCRATCH_BYTES the call returns PA_ERR_WORKSPACE and launches nothing.
 *
 * The first call on a device looks up the array's device address (with that
 * device current); make that first call before any stream capture. All calls on
 * a device share the array and it keeps the previous call's contents (nothing
 * in it needs to start at zero). Calls that overlap on the GPU race on it:
 * order them (one stream, or events between streams).
 */
#define PA_NOALLOC_SCRATCH_BYTES ((size_t)32 << 20)

int pa_paged_attention_decode_noalloc(void *out, const void *q, const void *key_cache,
                                      const void *value_cache, const int32_t *block_tables,
                                      int max_blocks_per_seq, const int32_t *context_lens,
                                      int num_seqs, int num_heads, int num_kv_heads, int head_dim,
                                      int block_size, int64_t num_blocks, float scale,
                                      int max_context_len, int partition_size, int dtype,
                                      void *stream);

/*
 * Whole-block copies for copy-on-write.
 * [P1 cow_write: a shared block is duplicated whole into a fresh block before
 *  the write; P2 demo 3]
 *
 * For each pair (src, dst): key_cache[dst] = key_cache[src] and
 * value_cache[dst] = value_cache[src] (all slots, heads and dims). Pairs with
 * an id outside [0, num_blocks) are skipped and set PA_DEVERR_COPY_PAIR.
 * Destinations must be distinct and must not appear as a source in the same
 * call (caller error otherwise; pa_alloc_append never produces that).
 */
int pa_copy_blocks(void *key_cache, void *value_cache, const int32_t *src_dst_pairs,
                   int64_t num_pairs, int64_t num_blocks, int block_size, int num_kv_heads,
                   int head_dim, int dtype, void *stream);

/*
 * ---- 8-bit (OCP FP8 E4M3) KV cache ------------------------------------------
 * Not on the pages [P1-P3]; an extension that halves the bytes a decode step
 * reads. Code format: OCP 8-bit Floating Point Specification, E4M3 (sign, 4
 * exponent bits with bias 7, 3 mantissa bits, no infinities, 0x7F/0xFF = NaN,
 * largest finite 448). The caches are uint8 arrays with the usual layout
 * [num_blocks, block_size, num_kv_heads, head_dim]; a K element stands for
 * decoded(code) * k_scale and a V element for decoded(code) * v_scale, with one
 * float32 scale for all of K and one for all of V (both finite and > 0).
 */

/*
 * Scatter with quantisation. [P1 write_kv; P3 B.2 for the slots, exactly as
 * pa_paged_kv_write]
 * Element x of k[t] is stored as the E4M3 code nearest to the float32 quotient
 * x / k_scale (IEEE division), ties to the even code, magnitudes >= 448 and
 * infinities saturating to +-448, NaN to a NaN code; v likewise with v_scale.
 * k, v: [num_tokens, num_kv_heads, head_dim] of src_dtype (PA_DTYPE_F32, _F16
 * or _BF16). Slot rules and errors as pa_paged_kv_write. Requires
 * num_kv_heads*head_dim to be a multiple of 16.
 */
int pa_paged_kv_write_fp8(const void *k, const void *v, const int32_t *slot_mapping,
                          int64_t num_tokens, void *key_cache, void *value_cache,
                          int64_t num_blocks, int block_size, int num_kv_heads, int head_dim,
                          float k_scale, float v_scale, int src_dtype, void *stream);

/*
 * Decode attention over E4M3 caches. [P2 demo 2, eq. 4, as
 * pa_paged_attention_decode]
 *
 *   out[b,h,:] = sum_t softmax_t(scale * q[b,h,:] . k_scale*K8[b,t,h/G,:])
 *                * v_scale*V8[b,t,h/G,:]
 *
 * q and out have dtype PA_DTYPE_BF16 or PA_DTYPE_F16. The codes are the
 * tensor-core operands as stored (E4M3 x E4M3 products, fp32 accumulation);
 * the query and the softmax weights enter those products as sums of two E4M3
 * terms: a query row scaled by a power of two is exact for bf16 (8 of an
 * f16's 11 significant bits), and a weight keeps about a bf16's precision.
 * Supported: head_dim 128, num_heads / num_kv_heads <= 16, block_size a power
 * of two in [8, 128]; PA_ERR_UNSUPPORTED otherwise. Partitions,
 * max_context_len, the workspace (size from pa_decode_workspace_bytes; NULL =
 * cudaMallocAsync on the stream) and the device error bits are those of
 * pa_paged_attention_decode. A NaN code inside a context makes the outputs of
 * its heads NaN (the write never stores one from a finite input); codes in
 * the slots past a context's end are never used, whatever they hold.
 */
int pa_paged_attention_decode_fp8(void *out, const void *q, const void *key_cache,
                                  const void *value_cache, const int32_t *block_tables,
                                  int max_blocks_per_seq, const int32_t *context_lens, int num_seqs,
                                  int num_heads, int num_kv_heads, int head_dim, int block_size,
                                  int64_t num_blocks, float scale, float k_scale, float v_scale,
                                  int max_context_len, int partition_size, void *workspace,
                                  size_t workspace_bytes, int dtype, void *stream);

/*
 * One decode step over E4M3 caches: pa_paged_kv_write_fp8 of each sequence's new
 * token, then pa_paged_attention_decode_fp8. [P2 demo 1: a decode step writes
 * the new token's KV into its slot, then attends over the whole context, that
 * token included; P3 B.2: slot_mapping]
 *
 * k_new, v_new: [num_seqs, num_kv_heads, head_dim] in dtype (the query's bf16 or
 * f16, 16-byte aligned), the new token of sequence b in row b; slot_mapping[b]:
 * its slot, which must be the slot of position context_lens[b] - 1, or -1 for
 * no write (the only value allowed for an empty context). The decode kernel
 * quantises and stores each token itself, with the scatter's encoding (the
 * nearest code of x / k_scale or x / v_scale), just before it reads the token's
 * block; a slot other than that of position ctx - 1 sets PA_DEVERR_SLOT and is
 * not written. The block holding a sequence's new token must not be read by
 * another sequence of the same call (copy-on-write guarantees it). The result,
 * the caches and the other arguments are those of pa_paged_kv_write_fp8
 * followed by pa_paged_attention_decode_fp8.
 */
int pa_paged_attention_decode_fp8_append(void *out, const void *q, const void *k_new, const void *v_new,
                                         const int32_t *slot_mapping, void *key_cache, void *value_cache,
                                         const int32_t *block_tables, int max_blocks_per_seq,
                                         const int32_t *context_lens, int num_seqs, int num_heads, int num_kv_heads,
                                         int head_dim, int block_size, int64_t num_blocks, float scale,
                                         float k_scale, float v_scale, int max_context_len, int partition_size,
                                         void *workspace, size_t workspace_bytes, int dtype, void *stream);

/*
 * Synchronise `stream`, then read and clear the current device's error word.
 * *bits receives the PA_DEVERR_* bits seen since the last call. Returns
 * PA_ERR_DEVICE_INDEX when any bit was set, PA_OK otherwise.
 */
int pa_get_device_error(void *stream, uint32_t *bits);

/*
 * Check of the failure path of the pipeline kernels' waits. The pages have no
 * counterpart; it tests this library's own failure detection.
 *
 * Every wait of the tensor-core kernels on an mbarrier is bounded: after a
 * limit of real time (1 s in those kernels) it gives up, the whole warp agrees
 * on that, and the kernel sets PA_DEVERR_WAIT, drains and returns instead of
 * hanging. This call runs that same wait code in a one-warp kernel on an
 * mbarrier phase that nothing completes, with nothing in flight, after first
 * completing and observing one phase itself. The wait gives up after limit_ns
 * nanoseconds (1000 <= limit_ns <= 1e9, else PA_ERR_INVALID_ARG) and the kernel
 * sets PA_DEVERR_WAIT in the device error word (read it with
 * pa_get_device_error). report, if not NULL, is device memory of 4 int64
 * (8-byte aligned): [0] 1 if the completed phase was seen, [1] how many of the
 * 32 lanes gave up on their own wait, [2] 1 if the warp agreed on the failure,
 * [3] nanoseconds lane 0 waited before giving up. Asynchronous on `stream`.
 */
int pa_check_bounded_wait(int64_t limit_ns, int64_t *report, void *stream);

/* ---- host block allocator ------------------------------------------------- */
/*
 * [P1 PagedKVManager: block pool whose free ids sit on a stack (initially
 *  0..N-1 pushed in order, allocation pops the top), reference counts,
 *  cow_write, free_sequence; P2 demo 1 (a new block only when a token starts
 *  one), demo 3 (forked samples share blocks; copy-on-write on a shared
 *  partial block)]
 * Host memory only; no CUDA calls. Not thread-safe: one caller at a time per
 * allocator object.
 */
typedef struct pa_allocator pa_allocator;

typedef struct pa_alloc_stats {
    int64_t num_blocks;
    int64_t num_free;
    int64_t num_used;
    int64_t peak_used;
    int64_t num_cow_copies;
    int64_t num_seqs;
} pa_alloc_stats;

/* Create a pool of num_blocks blocks of block_size tokens. */
int pa_alloc_create(int64_t num_blocks, int block_size, pa_allocator **out);
void pa_alloc_destroy(pa_allocator *a);

/* Register an empty sequence (PA_ERR_EXISTS if present). */
int pa_alloc_add_seq(pa_allocator *a, int64_t seq_id);

/* child shares every block of parent (each reference count + 1). */
int pa_alloc_fork(pa_allocator *a, int64_t parent, int64_t child);

/*
 * Append n_tokens positions to seq_id. slots_out[n_tokens] receives each new
 * position's slot. A position that starts a block takes a fresh block; a
 * position inside a block whose reference count is above 1 first copies it
 * (the (src, dst) pair is appended to cow_pairs_out, 2 ints per pair, at most
 * cow_cap pairs) and the table is repointed. *n_cow receives the pair count.
 * All-or-nothing: PA_ERR_OUT_OF_BLOCKS (or PA_ERR_INVALID_ARG when cow_cap is
 * too small) leaves the allocator unchanged.
 */
int pa_alloc_append(pa_allocator *a, int64_t seq_id, int64_t n_tokens, int32_t *slots_out,
                    int32_t *cow_pairs_out, int64_t cow_cap, int64_t *n_cow);

/* Drop the sequence; blocks whose count reaches 0 return to the free stack. */
int pa_alloc_free_seq(pa_allocator *a, int64_t seq_id);

/* Copy seq_id's table into out[cap]; *n receives its length (may exceed cap). */
int pa_alloc_block_table(const pa_allocator *a, int64_t seq_id, int32_t *out, int64_t cap,
                         int64_t *n);

/* Current length (tokens) of seq_id. */
int pa_alloc_seq_len(const pa_allocator *a, int64_t seq_id, int64_t *len);

/*
 * Export a decode batch: row i of tables[n_seqs, max_blocks_per_seq] gets
 * seq_ids[i]'s table padded with -1, context_lens[i] its length.
 * PA_ERR_INVALID_ARG when a table is longer than max_blocks_per_seq.
 */
int pa_alloc_export(const pa_allocator *a, const int64_t *seq_ids, int64_t n_seqs,
                    int32_t *tables, int max_blocks_per_seq, int32_t *context_lens);

/* Raw pool operations (take one block with count 1; drop one reference). */
int pa_alloc_block(pa_allocator *a, int32_t *block_out);
int pa_alloc_decref(pa_allocator *a, int32_t block);

/*
 * Host helper: group sequences whose block tables start with the same physical
 * blocks (the prefix sharing that fork() creates). Candidates need at least
 * min_shared_blocks full blocks and are keyed by their first block; each group
 * of 2..max_members sequences (larger sets are split in order) gets the longest
 * run of leading blocks that all members hold identically and completely.
 * Outputs prefix_lens[num_seqs] (shared tokens, 0 outside groups),
 * group_members[num_seqs * max_members] (num_groups rows used, -1 padded).
 * Host memory only.
 */
int pa_prefix_groups(const int32_t *block_tables, const int32_t *context_lens, int num_seqs,
                     int max_blocks_per_seq, int block_size, int max_members, int min_shared_blocks,
                     int32_t *prefix_lens, int32_t *group_members, int *num_groups);

/* Reference count of one block. */
int pa_alloc_refcount(const pa_allocator *a, int32_t block, int32_t *count);

int pa_alloc_get_stats(const pa_allocator *a, pa_alloc_stats *out);

/*
 * Checkpoint / resume of the allocator's whole state: free stack (order
 * included), reference counts, sequences with their lengths and tables, peak
 * and copy counters. Not on the pages; a serving process that restarts keeps
 * its device caches' block assignments.
 *
 * pa_alloc_snapshot writes an image of *a into buf (host memory, cap bytes) and
 * its size into *size. With buf NULL it only reports the size; with cap below
 * the size it writes nothing and returns PA_ERR_INVALID_ARG. The image is in
 * host byte order, tagged "PAALLOC1".
 *
 * pa_alloc_restore builds a new allocator (*out, owned by the caller, freed
 * with pa_alloc_destroy) from an image of exactly `size` bytes. It behaves as
 * the allocator the image was taken from: the same blocks, in the same order,
 * for every later call. The image is checked first. That means ids in range,
 * the free stack exactly the blocks with count 0 (each once), every table as
 * long as its length needs, every count at least the number of tables holding
 * the block, sequence ids increasing, and no trailing bytes. Any failure
 * returns PA_ERR_INVALID_ARG with *out = NULL.
 */
int pa_alloc_snapshot(const pa_allocator *a, void *buf, int64_t cap, int64_t *size);
int pa_alloc_restore(const void *buf, int64_t size, pa_allocator **out);

#ifdef __cplusplus
}
#endif

#endif /* PAGEDATTN_H */
