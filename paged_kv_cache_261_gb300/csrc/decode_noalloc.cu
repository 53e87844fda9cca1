// Decode attention for callers that must not allocate device memory.
//
// pa_paged_attention_decode needs split-K scratch (per-partition max, sum and
// partial output) whenever a context spans more than one partition. It takes
// that scratch from the caller, or, when the caller passes none, from
// cudaMallocAsync. Some callers can do neither: a host process whose device
// memory is owned by another runtime that forbids allocations by libraries, or
// a latency-bound serving loop where an allocation (and the synchronisation it
// can imply) is not acceptable, and that has no spare buffer of its own to lend.
//
// pa_paged_attention_decode_noalloc serves them with a fixed scratch array
// compiled into this library: kNoAllocScratchBytes of device memory on every GPU
// that loads the library, held from module load until the process exits. No call
// of this entry point allocates or frees device memory.
//
// All calls on a device share the one array, and it keeps whatever the previous
// call left in it. Nothing in it has to start at zero: every partial that the
// merge kernel reads is written by the same call first. Two calls that overlap
// on the GPU (different streams without ordering between them, or different
// host threads) race on the array and give undefined results; callers must
// order them.
#include <stdint.h>

#include "call_range.h"
#include "../../include/pagedattn.h"
#include "common.cuh"

namespace {

constexpr size_t kNoAllocScratchBytes = PA_NOALLOC_SCRATCH_BYTES;   // 32 MiB per GPU

static __device__ __align__(256) unsigned char g_noalloc_scratch[kNoAllocScratchBytes];

// Device address of g_noalloc_scratch on each device, looked up once per device
// on the first call made with that device current. (On the host the symbol
// names a host-side stand-in, not device memory, so only this address may be
// passed to kernels.)
void *g_scratch_addr[pa::kMaxDevices] = {};

int scratch_address(void **out) {
    int dev = 0;
    if (cudaGetDevice(&dev) != cudaSuccess || dev < 0 || dev >= pa::kMaxDevices) return PA_ERR_CUDA;
    if (!g_scratch_addr[dev]) {
        void *ptr = nullptr;
        if (cudaGetSymbolAddress(&ptr, g_noalloc_scratch) != cudaSuccess || !ptr) return PA_ERR_CUDA;
        g_scratch_addr[dev] = ptr;
    }
    *out = g_scratch_addr[dev];
    return PA_OK;
}

}  // namespace

extern "C" {

int pa_paged_attention_decode_noalloc(void *out, const void *q, const void *key_cache,
                                      const void *value_cache, const int32_t *block_tables,
                                      int max_blocks_per_seq, const int32_t *context_lens,
                                      int num_seqs, int num_heads, int num_kv_heads, int head_dim,
                                      int block_size, int64_t num_blocks, float scale,
                                      int max_context_len, int partition_size, int dtype,
                                      void *stream) {
    const pa::CallRange range(__func__);
    if (num_seqs < 0 || num_heads <= 0 || head_dim <= 0 || max_context_len < 0 || partition_size < 0 ||
        block_size <= 0 || max_blocks_per_seq <= 0)
        return PA_ERR_INVALID_ARG;
    const int64_t bound = max_context_len > 0 ? (int64_t)max_context_len
                                              : (int64_t)max_blocks_per_seq * block_size;
    if (bound > INT32_MAX) return PA_ERR_UNSUPPORTED;
    const size_t need = pa_decode_workspace_bytes(num_seqs, num_heads, head_dim, (int)bound, partition_size);
    if (need > kNoAllocScratchBytes) return PA_ERR_WORKSPACE;   // larger than the built-in scratch
    void *scratch = nullptr;
    if (int rc = scratch_address(&scratch)) return rc;
    return pa_paged_attention_decode(out, q, key_cache, value_cache, block_tables, max_blocks_per_seq,
                                     context_lens, num_seqs, num_heads, num_kv_heads, head_dim, block_size,
                                     num_blocks, scale, max_context_len, partition_size, scratch,
                                     kNoAllocScratchBytes, dtype, stream);
}

}  // extern "C"
