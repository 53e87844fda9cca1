// Scatter of new tokens into cache slots and whole-block copies.
//
// paged_kv_write follows "PagedAttention实现" (ainanfeng.cn), write_kv: a token
// at a position lands in page position / block_size at offset position %
// block_size; with the slot encoding of "04 - Paged Attention 实现进度" B.2
// (slot = block * block_size + offset) and the cache layout
// [num_blocks, block_size, num_kv_heads, head_dim], one token's K row (all
// kv heads) is a single contiguous run of num_kv_heads*head_dim elements in the
// cache, so the scatter is a row copy.
//
// copy_blocks follows the same page's cow_write: a shared block is duplicated
// whole (every slot, head and dim) into the fresh block; a block is one
// contiguous run of block_size*num_kv_heads*head_dim elements.
//
// Both are pure data movement, bound by HBM bandwidth: 16-byte vector loads and
// stores, several in flight per thread.
#include "common.cuh"
#include "kernels.h"

namespace pa {
namespace {

constexpr int kWriteWarps = 8;       // tokens per CTA (one warp per token)
constexpr int kWriteUnroll = 4;      // 16-byte vectors in flight per lane, per tensor

__global__ __launch_bounds__(kWriteWarps * 32) void kv_write_kernel(
    const uint4 *__restrict__ k, const uint4 *__restrict__ v, const int32_t *__restrict__ slots,
    int64_t num_tokens, uint4 *__restrict__ kc, uint4 *__restrict__ vc, int64_t num_slots,
    int row_vecs, unsigned int *err) {
    // a decode launched after this kernel may start its set-up now; it waits for
    // this grid to finish before reading the cache
    asm volatile("griddepcontrol.launch_dependents;");
    const int lane = threadIdx.x & 31;
    const int64_t t = (int64_t)blockIdx.x * kWriteWarps + (threadIdx.x >> 5);
    if (t >= num_tokens) return;
    const int64_t slot = slots[t];
    if (slot == -1) return;
    if (slot < 0 || slot >= num_slots) {
        if (lane == 0) raise_error(err, PA_DEVERR_SLOT);
        return;
    }
    const uint4 *ks = k + t * row_vecs;
    const uint4 *vs = v + t * row_vecs;
    uint4 *kd = kc + slot * row_vecs;
    uint4 *vd = vc + slot * row_vecs;
    for (int base = 0; base < row_vecs; base += 32 * kWriteUnroll) {
        uint4 a[kWriteUnroll], bv[kWriteUnroll];
#pragma unroll
        for (int u = 0; u < kWriteUnroll; ++u) {
            const int i = base + u * 32 + lane;
            if (i < row_vecs) {
                a[u] = __ldcs(ks + i);
                bv[u] = __ldcs(vs + i);
            }
        }
#pragma unroll
        for (int u = 0; u < kWriteUnroll; ++u) {
            const int i = base + u * 32 + lane;
            if (i < row_vecs) {
                kd[i] = a[u];
                vd[i] = bv[u];
            }
        }
    }
}

constexpr int kCopyThreads = 256;
constexpr int kCopyUnroll = 4;                            // vectors per thread per tensor
constexpr int kCopyChunk = kCopyThreads * kCopyUnroll;    // vectors per CTA (16 KiB)

__global__ __launch_bounds__(kCopyThreads) void copy_blocks_kernel(
    uint4 *__restrict__ kc, uint4 *__restrict__ vc, const int32_t *__restrict__ pairs,
    int64_t num_blocks, int64_t block_vecs, unsigned int *err) {
    const int64_t pair = blockIdx.x;
    const int64_t src = pairs[2 * pair];
    const int64_t dst = pairs[2 * pair + 1];
    if (src < 0 || src >= num_blocks || dst < 0 || dst >= num_blocks) {
        if (threadIdx.x == 0 && blockIdx.y == 0) raise_error(err, PA_DEVERR_COPY_PAIR);
        return;
    }
    const int64_t base = (int64_t)blockIdx.y * kCopyChunk;
    const uint4 *ks = kc + src * block_vecs;
    const uint4 *vs = vc + src * block_vecs;
    uint4 *kd = kc + dst * block_vecs;
    uint4 *vd = vc + dst * block_vecs;
    uint4 a[kCopyUnroll], b[kCopyUnroll];
#pragma unroll
    for (int u = 0; u < kCopyUnroll; ++u) {
        const int64_t i = base + u * kCopyThreads + threadIdx.x;
        if (i < block_vecs) {
            a[u] = __ldcs(ks + i);
            b[u] = __ldcs(vs + i);
        }
    }
#pragma unroll
    for (int u = 0; u < kCopyUnroll; ++u) {
        const int64_t i = base + u * kCopyThreads + threadIdx.x;
        if (i < block_vecs) {
            kd[i] = a[u];
            vd[i] = b[u];
        }
    }
}

}  // namespace

int launch_kv_write(const void *k, const void *v, const int32_t *slot_mapping, int64_t num_tokens,
                    void *key_cache, void *value_cache, int64_t num_slots, int row_bytes,
                    unsigned int *err, cudaStream_t stream) {
    if (num_tokens == 0) return 0;
    const int row_vecs = row_bytes / 16;
    const int64_t grid = (num_tokens + kWriteWarps - 1) / kWriteWarps;
    kv_write_kernel<<<(unsigned)grid, kWriteWarps * 32, 0, stream>>>(
        (const uint4 *)k, (const uint4 *)v, slot_mapping, num_tokens, (uint4 *)key_cache,
        (uint4 *)value_cache, num_slots, row_vecs, err);
    return cudaGetLastError() == cudaSuccess ? 0 : -1;
}

int launch_copy_blocks(void *key_cache, void *value_cache, const int32_t *pairs, int64_t num_pairs,
                       int64_t num_blocks, int64_t block_bytes, unsigned int *err,
                       cudaStream_t stream) {
    if (num_pairs == 0) return 0;
    const int64_t block_vecs = block_bytes / 16;
    const int64_t chunks = (block_vecs + kCopyChunk - 1) / kCopyChunk;
    dim3 grid((unsigned)num_pairs, (unsigned)chunks);
    copy_blocks_kernel<<<grid, kCopyThreads, 0, stream>>>((uint4 *)key_cache, (uint4 *)value_cache,
                                                          pairs, num_blocks, block_vecs, err);
    return cudaGetLastError() == cudaSuccess ? 0 : -1;
}

}  // namespace pa
