// Internal launch interface between the C-ABI layer (capi.cu) and the kernel
// translation units. Not part of the public ABI.
#pragma once

#include <cuda_runtime.h>
#include <stddef.h>
#include <stdint.h>

namespace pa {

// Everything a decode kernel needs; built and validated by the C-ABI layer.
struct DecodeParams {
    void *out;
    const void *q;
    const void *key_cache;
    const void *value_cache;
    const int32_t *block_tables;
    const int32_t *context_lens;
    float *ws_ml;              // [B][H][P][2] running max (log2 units) and sum
    float *ws_o;               // [B][H][P][D] unnormalised partial outputs
    unsigned int *err;         // device error word
    const int32_t *prefix_lens;  // optional [B]: leading tokens attended by the shared-prefix pass
    // optional decode-step write (tensor-core kernel): sequence b's new token, rows
    // app_k / app_v [B][Hk][128], goes to slot app_slots[b], which must be the slot of
    // position ctx_b - 1; the CTA reading that block writes it first
    const void *app_k;
    const void *app_v;
    const int32_t *app_slots;
    int64_t num_blocks;
    int max_blocks_per_seq;
    int num_seqs;
    int num_heads;
    int num_kv_heads;
    int group;                 // num_heads / num_kv_heads
    int head_dim;
    int block_size;
    int log2_block_size;
    int partition_size;        // tokens per partition (multiple of 128)
    int max_partitions;        // P: partitions per sequence the grid covers
    int context_limit;         // min(max_blocks_per_seq*bs, P*partition_size)
    float scale_log2;          // scale * log2(e)
    // Sharing-aware decode with one partition covering every whole context (each
    // sequence: at most one shared and one private partition): the tensor-core kernel's
    // item for a sequence's tokens after its shared prefix joins the shared pass's
    // partial (slot 0) with its own and writes the final row, so no merge runs; a
    // sequence whose whole context is shared gets an item with no tiles that only joins.
    int fold_shared;
    // Set with the tensor-core partition kernel: the one-warp-per-row merge lets the
    // next launch on the stream (the next call's partition kernel) start its set-up
    // while it runs. Not with the 8-bit kernel, whose two CTAs per SM, resident
    // early, slow that merge down more than their set-up gains.
    int chain_next;
};

// Chunked prefill: every query row of a packed chunk attends causally.
struct PrefillParams {
    void *out;                  // [num_query_tokens, num_heads, head_dim]
    const void *q;              // same layout
    const void *key_cache;
    const void *value_cache;
    const int32_t *block_tables;
    const int32_t *context_lens;
    const int32_t *query_start_loc;   // [num_seqs + 1]
    unsigned int *err;
    int64_t num_blocks;
    int64_t num_query_tokens;
    int max_blocks_per_seq;
    int num_seqs;
    int num_heads;
    int num_kv_heads;
    int group;                  // num_heads / num_kv_heads
    int group_pad;              // group rounded up to a power of two
    int rows_q;                 // query tokens per item: 128 / group_pad
    int qtiles;                 // ceil(max_query_len / rows_q)
    int sorted_items;           // set by the launcher: deal items largest first (see prefill_tc.cu)
    int head_dim;
    int block_size;
    int log2_block_size;
    int max_query_len;
    int context_limit;          // max_blocks_per_seq * block_size
    float scale_log2;
    // shared-prefix decode (group mode): rows are (member, head) pairs of a group
    const int32_t *prefix_lens;     // [num_seqs] shared leading tokens per sequence
    const int32_t *group_members;   // [num_groups, max_members], -1 = empty slot
    int num_groups;
    int max_members;
    int partition_size;
    int max_partitions;             // workspace stride P
    int shared_parts;               // partitions of the longest shared prefix
    float *ws_ml;
    float *ws_o;
};

bool prefill_tc_supported(const PrefillParams &p, int dtype);
int launch_prefill_tc(const PrefillParams &p, int dtype, cudaStream_t stream);
// Group mode of the same kernel: attention of every group member's query over
// the group's shared prefix, written as split-K partials (slots 0 .. shared-1).
int launch_shared_prefix_tc(const PrefillParams &p, int dtype, cudaStream_t stream);

int launch_kv_write(const void *k, const void *v, const int32_t *slot_mapping, int64_t num_tokens,
                    void *key_cache, void *value_cache, int64_t num_slots, int row_bytes,
                    unsigned int *err, cudaStream_t stream);

int launch_copy_blocks(void *key_cache, void *value_cache, const int32_t *pairs, int64_t num_pairs,
                       int64_t num_blocks, int64_t block_bytes, unsigned int *err,
                       cudaStream_t stream);

// SIMT partition kernel (any dtype); writes final rows for single-partition
// sequences and partials for the rest.
int launch_decode_simt(const DecodeParams &p, int dtype, cudaStream_t stream);

// Tensor-core partition kernel (bf16/f16, head_dim 128, group <= 16, block
// size 8..128). decode_tc_supported tells whether it covers a call.
bool decode_tc_supported(const DecodeParams &p, int dtype);

#ifdef __CUDACC__
// How a sequence's context splits between the shared-prefix pass and the
// per-sequence pass: tokens [0, ps) are covered by `shared` workspace slots
// written by the shared pass, tokens [ps, ctx) by `priv` partitions starting at
// slot `shared`. Without prefix_lens, ps = 0. ps is the given prefix length
// rounded down to whole blocks (both passes round alike), so every pass starts
// on a block boundary. `direct`: a single partition and nothing shared -- the
// partition kernel writes the final row itself.
struct SeqSplit {
    int ctx, ps, shared, priv;
    bool direct;
};

__device__ __forceinline__ SeqSplit seq_split(const DecodeParams &p, int b) {
    SeqSplit s;
    int ctx = p.context_lens[b];
    s.ctx = ctx < 0 ? 0 : (ctx > p.context_limit ? p.context_limit : ctx);
    int ps = p.prefix_lens ? p.prefix_lens[b] : 0;
    s.ps = (ps < 0 ? 0 : (ps > s.ctx ? s.ctx : ps)) & ~(p.block_size - 1);
    s.shared = (s.ps + p.partition_size - 1) / p.partition_size;
    s.priv = (s.ctx - s.ps + p.partition_size - 1) / p.partition_size;
    s.direct = s.ctx == 0 || (s.shared == 0 && s.priv <= 1);
    return s;
}
#endif
int launch_decode_tc(const DecodeParams &p, int dtype, cudaStream_t stream);

// Merge of the partials of sequences with more than one partition.
int launch_decode_reduce(const DecodeParams &p, int dtype, cudaStream_t stream);

// One warp waiting on an mbarrier phase that nothing completes, with the
// pipeline kernels' bounded wait (selftest.cu).
int launch_bounded_wait_check(unsigned long long limit_ns, int64_t *report, unsigned int *err,
                              cudaStream_t stream);

}  // namespace pa
