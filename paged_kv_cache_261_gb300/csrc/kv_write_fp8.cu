// Scatter of new tokens into an 8-bit (OCP FP8 E4M3) paged cache.
//
// The slot arithmetic is that of "PagedAttention实现" write_kv and "04 - Paged
// Attention 实现进度" B.2 (slot = block * block_size + offset; one token's row of
// all kv heads is contiguous in the [num_blocks, block_size, num_kv_heads,
// head_dim] cache). The 8-bit encoding is not on the pages: each element x is
// stored as the E4M3 code nearest to x / scale, the quotient taken in float32
// with IEEE division and rounded to the code by the hardware conversion
// (round to nearest even, saturating to +-448). One thread per 16-element run
// of one token's K or V row: it turns 16 source elements into one 16-byte run
// of codes, so even a batch of a few tokens spreads its divisions over the GPU.
#include "common.cuh"
#include "fp8_encode.cuh"
#include "kernels_fp8.h"

namespace pa {
namespace {

constexpr int kThreads = 256;

using fp8::encode16;
using fp8::load16;

template <typename TS>
__global__ __launch_bounds__(kThreads) void kv_write_fp8_kernel(
    const TS *__restrict__ k, const TS *__restrict__ v, const int32_t *__restrict__ slots, int64_t num_tokens,
    uint4 *__restrict__ kc, uint4 *__restrict__ vc, int64_t num_slots, int row_elems, float k_scale,
    float v_scale, unsigned int *err) {
    // a decode launched after this kernel may start its set-up now; it waits for
    // this grid to finish before reading the cache
    asm volatile("griddepcontrol.launch_dependents;");
    const int groups = row_elems / 16;              // 16-element runs per row
    const int64_t idx = (int64_t)blockIdx.x * kThreads + threadIdx.x;
    const int64_t t = idx / (2 * groups);           // token; then K runs, then V runs
    if (t >= num_tokens) return;
    const int r = (int)(idx - t * 2 * groups);
    const int64_t slot = slots[t];
    if (slot == -1) return;
    if (slot < 0 || slot >= num_slots) {
        if (r == 0) raise_error(err, PA_DEVERR_SLOT);
        return;
    }
    const bool is_v = r >= groups;
    const int g = is_v ? r - groups : r;
    float x[16];
    load16((is_v ? v : k) + t * row_elems + g * 16, x);
    (is_v ? vc : kc)[slot * groups + g] = encode16(x, is_v ? v_scale : k_scale);
}

template <typename TS>
int launch_t(const void *k, const void *v, const int32_t *slots, int64_t num_tokens, void *kc, void *vc,
             int64_t num_slots, int row_elems, float k_scale, float v_scale, unsigned int *err,
             cudaStream_t stream) {
    const int64_t threads = num_tokens * 2 * (row_elems / 16);
    const int64_t grid = (threads + kThreads - 1) / kThreads;
    if (grid > 0x7FFFFFFF) return -2;
    kv_write_fp8_kernel<TS><<<(unsigned)grid, kThreads, 0, stream>>>(
        static_cast<const TS *>(k), static_cast<const TS *>(v), slots, num_tokens, static_cast<uint4 *>(kc),
        static_cast<uint4 *>(vc), num_slots, row_elems, k_scale, v_scale, err);
    return cudaGetLastError() == cudaSuccess ? 0 : -1;
}

}  // namespace

int launch_kv_write_fp8(const void *k, const void *v, int src_dtype, const int32_t *slot_mapping,
                        int64_t num_tokens, void *key_cache, void *value_cache, int64_t num_slots,
                        int row_elems, float k_scale, float v_scale, unsigned int *err, cudaStream_t stream) {
    if (num_tokens == 0) return 0;
    switch (src_dtype) {
    case PA_DTYPE_F32:
        return launch_t<float>(k, v, slot_mapping, num_tokens, key_cache, value_cache, num_slots, row_elems,
                               k_scale, v_scale, err, stream);
    case PA_DTYPE_F16:
        return launch_t<__half>(k, v, slot_mapping, num_tokens, key_cache, value_cache, num_slots, row_elems,
                                k_scale, v_scale, err, stream);
    case PA_DTYPE_BF16:
        return launch_t<__nv_bfloat16>(k, v, slot_mapping, num_tokens, key_cache, value_cache, num_slots,
                                       row_elems, k_scale, v_scale, err, stream);
    default:
        return -2;
    }
}

}  // namespace pa
