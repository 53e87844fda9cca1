// C-ABI entry points of libpagedattn: host-side validation, kernel selection,
// split-K workspace handling and the device error word. The declarations and
// their contracts are in include/pagedattn.h.
#include <stdint.h>
#include <stdlib.h>
#include <string.h>

#include <algorithm>

#include "../../include/pagedattn.h"
#include "call_range.h"
#include "common.cuh"
#include "kernels.h"
#include "kernels_fp8.h"

namespace {

// Per-device error word. Kernels receive its address as an argument.
__device__ unsigned int g_device_error;

unsigned int *g_err_ptr[pa::kMaxDevices] = {};

int error_word(unsigned int **out) {
    int dev = 0;
    if (cudaGetDevice(&dev) != cudaSuccess || dev < 0 || dev >= pa::kMaxDevices) return PA_ERR_CUDA;
    if (!g_err_ptr[dev]) {
        void *p = nullptr;
        if (cudaGetSymbolAddress(&p, g_device_error) != cudaSuccess) return PA_ERR_CUDA;
        g_err_ptr[dev] = static_cast<unsigned int *>(p);
    }
    *out = g_err_ptr[dev];
    return PA_OK;
}

int elem_size(int dtype) {
    switch (dtype) {
    case PA_DTYPE_F32: return 4;
    case PA_DTYPE_F16: return 2;
    case PA_DTYPE_BF16: return 2;
    default: return 0;
    }
}

bool aligned16(const void *p) { return (reinterpret_cast<uintptr_t>(p) & 15u) == 0; }
bool pow2(int64_t x) { return x > 0 && (x & (x - 1)) == 0; }

int ilog2(int64_t x) {
    int r = 0;
    while ((int64_t(1) << r) < x) ++r;
    return r;
}

// Automatic partition size of the decode calls: 1024 tokens once the batch has
// enough of them (num_seqs x ceil(max_context_len / 1024) >= 64, so at least 64
// partitions per kv head in the worst case), else 512, which keeps small batches
// spread over the SMs. Measured on one GB300 with the current kernels (a call,
// 512 -> 1024): 8B-shaped batch 0.0993 -> 0.0972 ms, long context 0.3970 ->
// 0.3822 ms, mixed serving 0.3165 -> 0.3169 ms; over an 8-bit cache 0.0585 ->
// 0.0567, 0.2299 -> 0.2172, 0.1801 -> 0.1783 ms. Fewer, longer items cost less per
// item and leave fewer partials to merge; 2048 lost on the 8B-shaped and mixed
// batches.
constexpr int kSmallPartition = 512;
constexpr int kLargePartition = 1024;
constexpr int kSharedPartition = 512;           // sharing-aware decode: the smallest automatic choice

int auto_partition(int64_t num_seqs, int64_t max_ctx) {
    const int64_t parts = (max_ctx + kLargePartition - 1) / kLargePartition;
    return num_seqs * parts >= 64 ? kLargePartition : kSmallPartition;
}

int resolve_partition(int partition_size, int64_t num_seqs, int64_t max_ctx) {
    return partition_size == 0 ? auto_partition(num_seqs, max_ctx) : partition_size;
}

int64_t num_partitions(int64_t max_ctx, int part) {
    if (max_ctx <= 0) return 1;
    return (max_ctx + part - 1) / part;
}

int device_sm_count() {
    static int cached[64] = {};
    int dev = 0;
    if (cudaGetDevice(&dev) != cudaSuccess || dev < 0 || dev >= 64) return 152;
    if (cached[dev] == 0) {
        int n = 0;
        if (cudaDeviceGetAttribute(&n, cudaDevAttrMultiProcessorCount, dev) != cudaSuccess || n <= 0) return 152;
        cached[dev] = n;
    }
    return cached[dev];
}

// Partition of the sharing-aware decode when the caller names none. The shared pass
// has groups x kv heads x partitions items, which the persistent CTAs (one per SM)
// take in waves; an item costs its 128-key tiles plus about 1.4 tiles of fixed work
// (query rows into tensor memory, epilogue, pipeline fill). The estimate waves x
// (tiles + 1.4) is minimised over multiples of 128 from 512 up to the longest shared
// prefix, ties going to the larger partition (fewer partials to merge). Measured on
// the forked-sampling batch (32 prompts of 992 shared tokens, 8 samples each, G 4):
// 512 -> 0.0855 ms, 896 -> 0.0998 ms, 1024 -> 0.0803 ms, 2048 -> 0.0796 ms; the
// private pass uses the same partition. When the choice already holds each shared
// prefix in one partition, the partition grows to cover every whole context (the
// shared pass is unchanged) as long as that stays within kFoldMaxContext tokens and
// the private pass keeps two items per SM: then no merge runs (fold_shared).
constexpr int64_t kFoldMaxContext = 8192;

int shared_partition(int64_t num_groups, int64_t num_kv_heads, int64_t max_prefix, int sms) {
    if (num_groups <= 0 || num_kv_heads <= 0 || max_prefix <= 0 || sms <= 0) return kSharedPartition;
    const int64_t top = std::min<int64_t>((max_prefix + 127) / 128 * 128, 65536);
    int best = kSharedPartition;
    double best_cost = 0.0;
    for (int64_t part = kSharedPartition; part <= std::max<int64_t>(top, kSharedPartition); part += 128) {
        const int64_t items = num_groups * num_kv_heads * ((max_prefix + part - 1) / part);
        const int64_t waves = (items + sms - 1) / sms;
        const int64_t tiles = (std::min(part, max_prefix) + 127) / 128;
        const double cost = (double)waves * ((double)tiles + 1.4);
        if (part == kSharedPartition || cost <= best_cost) {
            best_cost = cost;
            best = (int)part;
        }
    }
    return best;
}

// Decode kernel choice: the tensor-core kernel where it applies, else SIMT.
// PA_DECODE_KERNEL=simt or =tc in the environment forces one (tests compare both).
enum class DecodeKernel { Auto, Simt, Tc };
DecodeKernel decode_kernel_choice() {
    const char *e = getenv("PA_DECODE_KERNEL");
    if (!e) return DecodeKernel::Auto;
    if (!strcmp(e, "simt")) return DecodeKernel::Simt;
    if (!strcmp(e, "tc")) return DecodeKernel::Tc;
    return DecodeKernel::Auto;
}

size_t align256(size_t x) { return (x + 255) & ~size_t(255); }

size_t workspace_bytes_for(int64_t B, int64_t H, int64_t D, int64_t P) {
    if (P <= 1) return 0;
    return align256((size_t)(B * H * P * 2 * 4)) + (size_t)(B * H * P * D * 4);
}

bool finite_positive(float x) { return x > 0.0f && x <= 3.4028234663852886e38f; }

constexpr int kNothingToDo = 1;

// Host-side validation and parameter set-up shared by the decode entry points
// (no CUDA call; p.err is left for the caller). Returns PA_OK, kNothingToDo (no
// sequences) or an error status. P receives the number of partitions per
// sequence the grid covers.
int decode_setup(pa::DecodeParams &p, int64_t &P, void *out, const void *q, const void *key_cache,
                 const void *value_cache, const int32_t *block_tables, int max_blocks_per_seq,
                 const int32_t *context_lens, int num_seqs, int num_heads, int num_kv_heads, int head_dim,
                 int block_size, int64_t num_blocks, float scale, int max_context_len, int partition_size) {
    if (num_seqs < 0 || num_heads <= 0 || num_kv_heads <= 0 || num_heads % num_kv_heads != 0 || head_dim <= 0 ||
        block_size <= 0 || num_blocks <= 0 || max_blocks_per_seq <= 0 || max_context_len < 0 || partition_size < 0)
        return PA_ERR_INVALID_ARG;
    if (!pow2(block_size) || block_size > 256) return PA_ERR_UNSUPPORTED;
    if (head_dim != 64 && head_dim != 128) return PA_ERR_UNSUPPORTED;
    if (num_heads / num_kv_heads > 16) return PA_ERR_UNSUPPORTED;
    if (partition_size != 0 && partition_size % 128 != 0) return PA_ERR_INVALID_ARG;
    if (num_seqs == 0) return kNothingToDo;
    if (num_seqs > 65535 || num_kv_heads > 65535) return PA_ERR_UNSUPPORTED;
    if (!out || !q || !key_cache || !value_cache || !block_tables || !context_lens) return PA_ERR_INVALID_ARG;
    if (!aligned16(out) || !aligned16(q) || !aligned16(key_cache) || !aligned16(value_cache))
        return PA_ERR_INVALID_ARG;
    if (!(scale == scale)) return PA_ERR_INVALID_ARG;

    const int64_t table_cap = (int64_t)max_blocks_per_seq * block_size;
    const int64_t max_ctx = max_context_len == 0 ? table_cap : max_context_len;
    if (max_ctx > INT32_MAX) return PA_ERR_UNSUPPORTED;
    const int part = resolve_partition(partition_size, num_seqs, max_ctx);
    P = num_partitions(max_ctx, part);
    if (P > INT32_MAX / part) return PA_ERR_UNSUPPORTED;
    int64_t limit = P * part < table_cap ? P * part : table_cap;
    if (limit > max_ctx) limit = max_ctx;

    p.out = out;
    p.q = q;
    p.key_cache = key_cache;
    p.value_cache = value_cache;
    p.block_tables = block_tables;
    p.context_lens = context_lens;
    p.num_blocks = num_blocks;
    p.max_blocks_per_seq = max_blocks_per_seq;
    p.num_seqs = num_seqs;
    p.num_heads = num_heads;
    p.num_kv_heads = num_kv_heads;
    p.group = num_heads / num_kv_heads;
    p.head_dim = head_dim;
    p.block_size = block_size;
    p.log2_block_size = ilog2(block_size);
    p.partition_size = part;
    p.max_partitions = (int)P;
    p.context_limit = (int)limit;
    p.scale_log2 = scale * pa::kLog2e;
    return PA_OK;
}

// Split-K workspace of a decode call: the caller's (checked) or, when none is
// given and one is needed, a cudaMallocAsync block returned in *owned for the
// caller to release after the merge.
int decode_workspace(pa::DecodeParams &p, int64_t P, void *workspace, size_t workspace_bytes, cudaStream_t s,
                     void **owned) {
    *owned = nullptr;
    const size_t need = workspace_bytes_for(p.num_seqs, p.num_heads, p.head_dim, P);
    if (need == 0) return PA_OK;
    void *ws = workspace;
    if (ws) {
        if (workspace_bytes < need) return PA_ERR_WORKSPACE;
        if (!aligned16(ws)) return PA_ERR_INVALID_ARG;
    } else {
        if (cudaMallocAsync(&ws, need, s) != cudaSuccess) return PA_ERR_CUDA;
        *owned = ws;
    }
    p.ws_ml = static_cast<float *>(ws);
    p.ws_o = reinterpret_cast<float *>(static_cast<char *>(ws) +
                                       align256((size_t)p.num_seqs * p.num_heads * P * 2 * 4));
    return PA_OK;
}

// The 8-bit decode, optionally with append (k_new, v_new and slot_mapping non-NULL:
// the kernel quantises and stores each sequence's new K/V row itself).
int decode_fp8_call(void *out, const void *q, const void *k_new, const void *v_new, const int32_t *slot_mapping,
                    const void *key_cache, const void *value_cache, const int32_t *block_tables,
                    int max_blocks_per_seq, const int32_t *context_lens, int num_seqs, int num_heads,
                    int num_kv_heads, int head_dim, int block_size, int64_t num_blocks, float scale, float k_scale,
                    float v_scale, int max_context_len, int partition_size, void *workspace, size_t workspace_bytes,
                    int dtype, void *stream) {
    if (dtype != PA_DTYPE_BF16 && dtype != PA_DTYPE_F16) return elem_size(dtype) ? PA_ERR_UNSUPPORTED
                                                                                  : PA_ERR_INVALID_ARG;
    if (!finite_positive(k_scale) || !finite_positive(v_scale)) return PA_ERR_INVALID_ARG;
    pa::DecodeParams p{};
    int64_t P = 0;
    int rc = decode_setup(p, P, out, q, key_cache, value_cache, block_tables, max_blocks_per_seq, context_lens,
                          num_seqs, num_heads, num_kv_heads, head_dim, block_size, num_blocks, scale,
                          max_context_len, partition_size);
    if (rc == kNothingToDo) return PA_OK;
    if (rc != PA_OK) return rc;
    if (!pa::decode_fp8_supported(p, dtype)) return PA_ERR_UNSUPPORTED;
    if ((rc = error_word(&p.err)) != PA_OK) return rc;
    p.scale_log2 = scale * k_scale * pa::kLog2e;                  // k_scale folded into the score scale
    p.app_k = k_new;
    p.app_v = v_new;
    p.app_slots = slot_mapping;
    cudaStream_t s = static_cast<cudaStream_t>(stream);
    void *owned = nullptr;
    if ((rc = decode_workspace(p, P, workspace, workspace_bytes, s, &owned)) != PA_OK) return rc;
    int krc = pa::launch_decode_fp8(p, v_scale, k_scale, dtype, s);
    if (krc == 0 && P > 1) krc = pa::launch_decode_reduce(p, dtype, s);
    if (owned) cudaFreeAsync(owned, s);
    if (krc == -2) return PA_ERR_UNSUPPORTED;
    return krc == 0 ? PA_OK : PA_ERR_CUDA;
}

}  // namespace

extern "C" {

const char *pa_status_string(int status) {
    switch (status) {
    case PA_OK: return "PA_OK";
    case PA_ERR_INVALID_ARG: return "PA_ERR_INVALID_ARG";
    case PA_ERR_UNSUPPORTED: return "PA_ERR_UNSUPPORTED";
    case PA_ERR_OUT_OF_BLOCKS: return "PA_ERR_OUT_OF_BLOCKS";
    case PA_ERR_CUDA: return "PA_ERR_CUDA";
    case PA_ERR_DEVICE_INDEX: return "PA_ERR_DEVICE_INDEX";
    case PA_ERR_UNKNOWN_SEQ: return "PA_ERR_UNKNOWN_SEQ";
    case PA_ERR_WORKSPACE: return "PA_ERR_WORKSPACE";
    case PA_ERR_EXISTS: return "PA_ERR_EXISTS";
    default: return "PA_ERR_UNKNOWN";
    }
}

int pa_version(void) { return 100; }

int pa_paged_kv_write(const void *k, const void *v, const int32_t *slot_mapping, int64_t num_tokens,
                      void *key_cache, void *value_cache, int64_t num_blocks, int block_size,
                      int num_kv_heads, int head_dim, int dtype, void *stream) {
    const pa::CallRange range(__func__);
    const int es = elem_size(dtype);
    if (es == 0 || num_tokens < 0 || num_blocks <= 0 || block_size <= 0 || num_kv_heads <= 0 ||
        head_dim <= 0)
        return PA_ERR_INVALID_ARG;
    const int64_t row_bytes = (int64_t)num_kv_heads * head_dim * es;
    if (row_bytes % 16 != 0 || row_bytes > (int64_t)1 << 30) return PA_ERR_UNSUPPORTED;
    if (num_tokens == 0) return PA_OK;
    if (!k || !v || !slot_mapping || !key_cache || !value_cache) return PA_ERR_INVALID_ARG;
    if (!aligned16(k) || !aligned16(v) || !aligned16(key_cache) || !aligned16(value_cache))
        return PA_ERR_INVALID_ARG;
    if (num_blocks > INT64_MAX / block_size) return PA_ERR_INVALID_ARG;
    if ((num_tokens + 7) / 8 > INT32_MAX) return PA_ERR_UNSUPPORTED;
    unsigned int *err = nullptr;
    if (int rc = error_word(&err)) return rc;
    if (pa::launch_kv_write(k, v, slot_mapping, num_tokens, key_cache, value_cache,
                            num_blocks * block_size, (int)row_bytes, err,
                            static_cast<cudaStream_t>(stream)) != 0)
        return PA_ERR_CUDA;
    return PA_OK;
}

size_t pa_decode_workspace_bytes(int num_seqs, int num_heads, int head_dim, int max_context_len,
                                 int partition_size) {
    if (num_seqs <= 0 || num_heads <= 0 || head_dim <= 0 || max_context_len < 0 || partition_size < 0)
        return 0;
    const int part = resolve_partition(partition_size, num_seqs, max_context_len);
    return workspace_bytes_for(num_seqs, num_heads, head_dim, num_partitions(max_context_len, part));
}

int pa_decode_partition_size(int num_seqs, int max_context_len, int partition_size) {
    if (num_seqs < 0 || max_context_len < 0 || partition_size < 0) return 0;
    return resolve_partition(partition_size, num_seqs, max_context_len);
}

int pa_paged_attention_decode(void *out, const void *q, const void *key_cache,
                              const void *value_cache, const int32_t *block_tables,
                              int max_blocks_per_seq, const int32_t *context_lens, int num_seqs,
                              int num_heads, int num_kv_heads, int head_dim, int block_size,
                              int64_t num_blocks, float scale, int max_context_len,
                              int partition_size, void *workspace, size_t workspace_bytes,
                              int dtype, void *stream) {
    const pa::CallRange range(__func__);
    if (elem_size(dtype) == 0) return PA_ERR_INVALID_ARG;
    pa::DecodeParams p{};
    int64_t P = 0;
    int rc = decode_setup(p, P, out, q, key_cache, value_cache, block_tables, max_blocks_per_seq, context_lens,
                          num_seqs, num_heads, num_kv_heads, head_dim, block_size, num_blocks, scale,
                          max_context_len, partition_size);
    if (rc == kNothingToDo) return PA_OK;
    if (rc != PA_OK) return rc;
    if ((rc = error_word(&p.err)) != PA_OK) return rc;
    cudaStream_t s = static_cast<cudaStream_t>(stream);
    void *owned = nullptr;
    if ((rc = decode_workspace(p, P, workspace, workspace_bytes, s, &owned)) != PA_OK) return rc;

    const DecodeKernel choice = decode_kernel_choice();
    int krc;
    if (choice == DecodeKernel::Tc || (choice == DecodeKernel::Auto && pa::decode_tc_supported(p, dtype))) {
        krc = pa::launch_decode_tc(p, dtype, s);
        p.chain_next = 1;
    } else {
        krc = pa::launch_decode_simt(p, dtype, s);
    }
    if (krc == 0 && P > 1) krc = pa::launch_decode_reduce(p, dtype, s);
    if (owned) cudaFreeAsync(owned, s);
    if (krc == -2) return PA_ERR_UNSUPPORTED;
    return krc == 0 ? PA_OK : PA_ERR_CUDA;
}

int pa_paged_attention_decode_append(void *out, const void *q, const void *k_new, const void *v_new,
                                     const int32_t *slot_mapping, void *key_cache, void *value_cache,
                                     const int32_t *block_tables, int max_blocks_per_seq,
                                     const int32_t *context_lens, int num_seqs, int num_heads, int num_kv_heads,
                                     int head_dim, int block_size, int64_t num_blocks, float scale,
                                     int max_context_len, int partition_size, void *workspace,
                                     size_t workspace_bytes, int dtype, void *stream) {
    const pa::CallRange range(__func__);
    if (elem_size(dtype) == 0) return PA_ERR_INVALID_ARG;
    pa::DecodeParams p{};
    int64_t P = 0;
    int rc = decode_setup(p, P, out, q, key_cache, value_cache, block_tables, max_blocks_per_seq, context_lens,
                          num_seqs, num_heads, num_kv_heads, head_dim, block_size, num_blocks, scale,
                          max_context_len, partition_size);
    if (rc == kNothingToDo) return PA_OK;
    if (rc != PA_OK) return rc;
    if (!k_new || !v_new || !slot_mapping || !aligned16(k_new) || !aligned16(v_new)) return PA_ERR_INVALID_ARG;
    if ((rc = error_word(&p.err)) != PA_OK) return rc;
    cudaStream_t s = static_cast<cudaStream_t>(stream);
    void *owned = nullptr;
    if ((rc = decode_workspace(p, P, workspace, workspace_bytes, s, &owned)) != PA_OK) return rc;

    const DecodeKernel choice = decode_kernel_choice();
    int krc;
    if (choice == DecodeKernel::Tc || (choice == DecodeKernel::Auto && pa::decode_tc_supported(p, dtype))) {
        // the tensor-core kernel writes each sequence's token itself, before reading its block
        p.app_k = k_new;
        p.app_v = v_new;
        p.app_slots = slot_mapping;
        krc = pa::launch_decode_tc(p, dtype, s);
        p.chain_next = 1;
    } else {
        // the scatter, then the decode (head_dim 64 or 128 keeps a row a multiple of
        // the scatter's 16-byte copies)
        const int64_t row_bytes = (int64_t)num_kv_heads * head_dim * elem_size(dtype);
        krc = row_bytes % 16 != 0 ? -2
                                  : pa::launch_kv_write(k_new, v_new, slot_mapping, num_seqs, key_cache,
                                                        value_cache, num_blocks * block_size, (int)row_bytes,
                                                        p.err, s);
        if (krc == 0) krc = pa::launch_decode_simt(p, dtype, s);
    }
    if (krc == 0 && P > 1) krc = pa::launch_decode_reduce(p, dtype, s);
    if (owned) cudaFreeAsync(owned, s);
    if (krc == -2) return PA_ERR_UNSUPPORTED;
    return krc == 0 ? PA_OK : PA_ERR_CUDA;
}

int pa_paged_kv_write_fp8(const void *k, const void *v, const int32_t *slot_mapping, int64_t num_tokens,
                          void *key_cache, void *value_cache, int64_t num_blocks, int block_size,
                          int num_kv_heads, int head_dim, float k_scale, float v_scale, int src_dtype,
                          void *stream) {
    const pa::CallRange range(__func__);
    if (elem_size(src_dtype) == 0 || num_tokens < 0 || num_blocks <= 0 || block_size <= 0 || num_kv_heads <= 0 ||
        head_dim <= 0)
        return PA_ERR_INVALID_ARG;
    if (!finite_positive(k_scale) || !finite_positive(v_scale)) return PA_ERR_INVALID_ARG;
    const int64_t row_elems = (int64_t)num_kv_heads * head_dim;
    if (row_elems % 16 != 0 || row_elems > (int64_t)1 << 28) return PA_ERR_UNSUPPORTED;
    if (num_tokens == 0) return PA_OK;
    if (!k || !v || !slot_mapping || !key_cache || !value_cache) return PA_ERR_INVALID_ARG;
    if (!aligned16(k) || !aligned16(v) || !aligned16(key_cache) || !aligned16(value_cache))
        return PA_ERR_INVALID_ARG;
    if (num_blocks > INT64_MAX / block_size) return PA_ERR_INVALID_ARG;
    const int64_t runs = 2 * (row_elems / 16);          // one thread per 16-element run of K or V
    if (num_tokens > INT64_MAX / runs || (num_tokens * runs + 255) / 256 > INT32_MAX) return PA_ERR_UNSUPPORTED;
    unsigned int *err = nullptr;
    if (int rc = error_word(&err)) return rc;
    if (pa::launch_kv_write_fp8(k, v, src_dtype, slot_mapping, num_tokens, key_cache, value_cache,
                                num_blocks * block_size, (int)row_elems, k_scale, v_scale, err,
                                static_cast<cudaStream_t>(stream)) != 0)
        return PA_ERR_CUDA;
    return PA_OK;
}

int pa_paged_attention_decode_fp8(void *out, const void *q, const void *key_cache, const void *value_cache,
                                  const int32_t *block_tables, int max_blocks_per_seq,
                                  const int32_t *context_lens, int num_seqs, int num_heads, int num_kv_heads,
                                  int head_dim, int block_size, int64_t num_blocks, float scale, float k_scale,
                                  float v_scale, int max_context_len, int partition_size, void *workspace,
                                  size_t workspace_bytes, int dtype, void *stream) {
    const pa::CallRange range(__func__);
    return decode_fp8_call(out, q, nullptr, nullptr, nullptr, key_cache, value_cache, block_tables,
                           max_blocks_per_seq, context_lens, num_seqs, num_heads, num_kv_heads, head_dim, block_size,
                           num_blocks, scale, k_scale, v_scale, max_context_len, partition_size, workspace,
                           workspace_bytes, dtype, stream);
}

int pa_paged_attention_decode_fp8_append(void *out, const void *q, const void *k_new, const void *v_new,
                                         const int32_t *slot_mapping, void *key_cache, void *value_cache,
                                         const int32_t *block_tables, int max_blocks_per_seq,
                                         const int32_t *context_lens, int num_seqs, int num_heads, int num_kv_heads,
                                         int head_dim, int block_size, int64_t num_blocks, float scale,
                                         float k_scale, float v_scale, int max_context_len, int partition_size,
                                         void *workspace, size_t workspace_bytes, int dtype, void *stream) {
    const pa::CallRange range(__func__);
    if (!k_new || !v_new || !slot_mapping || !aligned16(k_new) || !aligned16(v_new)) return PA_ERR_INVALID_ARG;
    return decode_fp8_call(out, q, k_new, v_new, slot_mapping, key_cache, value_cache, block_tables,
                           max_blocks_per_seq, context_lens, num_seqs, num_heads, num_kv_heads, head_dim, block_size,
                           num_blocks, scale, k_scale, v_scale, max_context_len, partition_size, workspace,
                           workspace_bytes, dtype, stream);
}

int shared_partition_for(int64_t num_seqs, int64_t num_groups, int64_t num_kv_heads, int64_t max_prefix,
                         int64_t max_ctx, int sms) {
    int part = shared_partition(num_groups, num_kv_heads, max_prefix, sms);
    const int64_t whole = (max_ctx + 127) / 128 * 128;
    if (num_groups > 0 && max_prefix > 0 && part >= max_prefix && whole > part && whole <= kFoldMaxContext &&
        num_seqs * num_kv_heads >= 2 * (int64_t)sms)
        part = (int)whole;
    return part;
}

int pa_decode_shared_partition_size(int num_seqs, int num_groups, int num_kv_heads, int max_prefix_len,
                                    int max_context_len, int partition_size) {
    if (partition_size != 0) return partition_size;
    return shared_partition_for(num_seqs, num_groups, num_kv_heads, max_prefix_len, max_context_len,
                                device_sm_count());
}

size_t pa_decode_shared_workspace_bytes(int num_seqs, int num_heads, int head_dim, int max_context_len,
                                        int partition_size) {
    if (num_seqs <= 0 || num_heads <= 0 || head_dim <= 0 || max_context_len < 0 || partition_size < 0) return 0;
    const int part = partition_size == 0 ? kSharedPartition : partition_size;
    const int64_t P = num_partitions(max_context_len, part) + 1;
    return align256((size_t)(num_seqs * (int64_t)num_heads * P * 2 * 4)) +
           (size_t)(num_seqs * (int64_t)num_heads * P * head_dim * 4);
}

int pa_paged_attention_decode_shared(void *out, const void *q, const void *key_cache, const void *value_cache,
                                     const int32_t *block_tables, int max_blocks_per_seq,
                                     const int32_t *context_lens, const int32_t *prefix_lens,
                                     const int32_t *group_members, int num_groups, int max_members,
                                     int max_prefix_len, int num_seqs, int num_heads, int num_kv_heads,
                                     int head_dim, int block_size, int64_t num_blocks, float scale,
                                     int max_context_len, int partition_size, void *workspace,
                                     size_t workspace_bytes, int dtype, void *stream) {
    const pa::CallRange range(__func__);
    if (elem_size(dtype) == 0 || num_seqs < 0 || num_heads <= 0 || num_kv_heads <= 0 ||
        num_heads % num_kv_heads != 0 || head_dim <= 0 || block_size <= 0 || num_blocks <= 0 ||
        max_blocks_per_seq <= 0 || max_context_len < 0 || partition_size < 0 || num_groups < 0 ||
        max_prefix_len < 0 || (num_groups > 0 && max_members < 1))
        return PA_ERR_INVALID_ARG;
    if (partition_size != 0 && partition_size % 128 != 0) return PA_ERR_INVALID_ARG;
    if (num_seqs == 0) return PA_OK;
    if (!out || !q || !key_cache || !value_cache || !block_tables || !context_lens || !prefix_lens ||
        (num_groups > 0 && !group_members))
        return PA_ERR_INVALID_ARG;
    if (!aligned16(out) || !aligned16(q) || !aligned16(key_cache) || !aligned16(value_cache))
        return PA_ERR_INVALID_ARG;
    if (!(scale > 0.f)) return PA_ERR_INVALID_ARG;
    const int64_t table_cap = (int64_t)max_blocks_per_seq * block_size;
    const int64_t max_ctx = max_context_len == 0 ? table_cap : max_context_len;
    if (max_ctx > INT32_MAX || num_seqs > 65535 || num_kv_heads > 65535) return PA_ERR_UNSUPPORTED;
    const int part = partition_size != 0 ? partition_size
                                         : shared_partition_for(num_seqs, num_groups, num_kv_heads,
                                                                std::min<int64_t>(max_prefix_len, max_ctx), max_ctx,
                                                                device_sm_count());
    const int64_t P = num_partitions(max_ctx, part) + 1;
    if (P > INT32_MAX / part) return PA_ERR_UNSUPPORTED;
    int64_t limit = (P - 1) * part < table_cap ? (P - 1) * part : table_cap;
    if (limit > max_ctx) limit = max_ctx;

    pa::DecodeParams d{};
    d.out = out;
    d.q = q;
    d.key_cache = key_cache;
    d.value_cache = value_cache;
    d.block_tables = block_tables;
    d.context_lens = context_lens;
    d.prefix_lens = prefix_lens;
    d.num_blocks = num_blocks;
    d.max_blocks_per_seq = max_blocks_per_seq;
    d.num_seqs = num_seqs;
    d.num_heads = num_heads;
    d.num_kv_heads = num_kv_heads;
    d.group = num_heads / num_kv_heads;
    d.head_dim = head_dim;
    d.block_size = block_size;
    d.log2_block_size = ilog2(block_size);
    d.partition_size = part;
    d.max_partitions = (int)P;
    d.context_limit = (int)limit;
    d.scale_log2 = scale * pa::kLog2e;
    // one partition covers every whole context: the private pass folds the shared
    // partials and writes the final rows, and no merge runs
    d.fold_shared = part >= max_ctx && d.group <= 8 ? 1 : 0;
    if (!pa::decode_tc_supported(d, dtype)) return PA_ERR_UNSUPPORTED;
    if (int rc = error_word(&d.err)) return rc;

    pa::PrefillParams g{};
    g.out = out;
    g.q = q;
    g.key_cache = key_cache;
    g.value_cache = value_cache;
    g.block_tables = block_tables;
    g.context_lens = context_lens;
    g.err = d.err;
    g.num_blocks = num_blocks;
    g.num_query_tokens = num_seqs;
    g.max_blocks_per_seq = max_blocks_per_seq;
    g.num_seqs = num_seqs;
    g.num_heads = num_heads;
    g.num_kv_heads = num_kv_heads;
    g.group = d.group;
    int gp = 1;
    while (gp < g.group) gp <<= 1;
    g.group_pad = gp;
    g.rows_q = 128 / gp;
    g.head_dim = head_dim;
    g.block_size = block_size;
    g.log2_block_size = d.log2_block_size;
    g.context_limit = (int)limit;
    g.scale_log2 = d.scale_log2;
    g.prefix_lens = prefix_lens;
    g.group_members = group_members;
    g.num_groups = num_groups;
    g.max_members = max_members;
    g.partition_size = part;
    g.max_partitions = (int)P;
    g.shared_parts = (int)num_partitions(max_prefix_len < limit ? max_prefix_len : limit, part);
    if (max_prefix_len == 0) g.shared_parts = 0;
    if (num_groups > 0 && (max_members > g.rows_q || !pa::prefill_tc_supported(g, dtype))) return PA_ERR_UNSUPPORTED;
    if ((int64_t)num_groups * num_kv_heads * (g.shared_parts + 1) > INT32_MAX) return PA_ERR_UNSUPPORTED;

    cudaStream_t s = static_cast<cudaStream_t>(stream);
    const size_t need = pa_decode_shared_workspace_bytes(num_seqs, num_heads, head_dim, (int)max_ctx, part);
    void *ws = workspace;
    bool owned = false;
    if (ws) {
        if (workspace_bytes < need) return PA_ERR_WORKSPACE;
        if (!aligned16(ws)) return PA_ERR_INVALID_ARG;
    } else {
        if (cudaMallocAsync(&ws, need, s) != cudaSuccess) return PA_ERR_CUDA;
        owned = true;
    }
    d.ws_ml = g.ws_ml = static_cast<float *>(ws);
    d.ws_o = g.ws_o = reinterpret_cast<float *>(static_cast<char *>(ws) +
                                                align256((size_t)num_seqs * num_heads * P * 2 * 4));
    int rc = 0;
    if (num_groups > 0 && g.shared_parts > 0) rc = pa::launch_shared_prefix_tc(g, dtype, s);
    if (rc == 0) rc = pa::launch_decode_tc(d, dtype, s);
    d.chain_next = 1;
    if (rc == 0 && !d.fold_shared) rc = pa::launch_decode_reduce(d, dtype, s);
    if (owned) cudaFreeAsync(ws, s);
    if (rc == -2) return PA_ERR_UNSUPPORTED;
    return rc == 0 ? PA_OK : PA_ERR_CUDA;
}

int pa_paged_attention_prefill(void *out, const void *q, const void *key_cache, const void *value_cache,
                               const int32_t *block_tables, int max_blocks_per_seq, const int32_t *context_lens,
                               const int32_t *query_start_loc, int num_seqs, int64_t num_query_tokens,
                               int max_query_len, int num_heads, int num_kv_heads, int head_dim, int block_size,
                               int64_t num_blocks, float scale, int dtype, void *stream) {
    const pa::CallRange range(__func__);
    if (elem_size(dtype) == 0 || num_seqs < 0 || num_query_tokens < 0 || max_query_len < 0 || num_heads <= 0 ||
        num_kv_heads <= 0 || num_heads % num_kv_heads != 0 || head_dim <= 0 || block_size <= 0 ||
        num_blocks <= 0 || max_blocks_per_seq <= 0)
        return PA_ERR_INVALID_ARG;
    if (dtype == PA_DTYPE_F32 || head_dim != 128 || num_heads / num_kv_heads > 16 || !pow2(block_size) ||
        block_size < 8 || block_size > 128)
        return PA_ERR_UNSUPPORTED;
    if (num_seqs == 0 || num_query_tokens == 0 || max_query_len == 0) return PA_OK;
    if (!out || !q || !key_cache || !value_cache || !block_tables || !context_lens || !query_start_loc)
        return PA_ERR_INVALID_ARG;
    if (!aligned16(out) || !aligned16(q) || !aligned16(key_cache) || !aligned16(value_cache))
        return PA_ERR_INVALID_ARG;
    if (!(scale > 0.f)) return PA_ERR_INVALID_ARG;     // the kernel takes the max of unscaled scores
    const int64_t table_cap = (int64_t)max_blocks_per_seq * block_size;
    if (table_cap > INT32_MAX || num_query_tokens > INT32_MAX) return PA_ERR_UNSUPPORTED;
    pa::PrefillParams p{};
    p.out = out;
    p.q = q;
    p.key_cache = key_cache;
    p.value_cache = value_cache;
    p.block_tables = block_tables;
    p.context_lens = context_lens;
    p.query_start_loc = query_start_loc;
    p.num_blocks = num_blocks;
    p.num_query_tokens = num_query_tokens;
    p.max_blocks_per_seq = max_blocks_per_seq;
    p.num_seqs = num_seqs;
    p.num_heads = num_heads;
    p.num_kv_heads = num_kv_heads;
    p.group = num_heads / num_kv_heads;
    int gp = 1;
    while (gp < p.group) gp <<= 1;
    p.group_pad = gp;
    p.rows_q = 128 / gp;
    p.qtiles = (max_query_len + p.rows_q - 1) / p.rows_q;
    p.head_dim = head_dim;
    p.block_size = block_size;
    p.log2_block_size = ilog2(block_size);
    p.max_query_len = max_query_len;
    p.context_limit = (int)table_cap;
    p.scale_log2 = scale * pa::kLog2e;
    if ((int64_t)num_seqs * num_kv_heads * p.qtiles > INT32_MAX) return PA_ERR_UNSUPPORTED;
    if (int rc = error_word(&p.err)) return rc;
    const int rc = pa::launch_prefill_tc(p, dtype, static_cast<cudaStream_t>(stream));
    if (rc == -2) return PA_ERR_UNSUPPORTED;
    return rc == 0 ? PA_OK : PA_ERR_CUDA;
}

int pa_copy_blocks(void *key_cache, void *value_cache, const int32_t *src_dst_pairs, int64_t num_pairs,
                   int64_t num_blocks, int block_size, int num_kv_heads, int head_dim, int dtype,
                   void *stream) {
    const pa::CallRange range(__func__);
    const int es = dtype == PA_DTYPE_E4M3 ? 1 : elem_size(dtype);
    if (es == 0 || num_pairs < 0 || num_blocks <= 0 || block_size <= 0 || num_kv_heads <= 0 ||
        head_dim <= 0)
        return PA_ERR_INVALID_ARG;
    const int64_t block_bytes = (int64_t)block_size * num_kv_heads * head_dim * es;
    if (block_bytes % 16 != 0) return PA_ERR_UNSUPPORTED;
    if (num_pairs == 0) return PA_OK;
    if (num_pairs > INT32_MAX) return PA_ERR_UNSUPPORTED;
    if (!key_cache || !value_cache || !src_dst_pairs) return PA_ERR_INVALID_ARG;
    if (!aligned16(key_cache) || !aligned16(value_cache)) return PA_ERR_INVALID_ARG;
    unsigned int *err = nullptr;
    if (int rc = error_word(&err)) return rc;
    if (pa::launch_copy_blocks(key_cache, value_cache, src_dst_pairs, num_pairs, num_blocks, block_bytes,
                               err, static_cast<cudaStream_t>(stream)) != 0)
        return PA_ERR_CUDA;
    return PA_OK;
}

int pa_check_bounded_wait(int64_t limit_ns, int64_t *report, void *stream) {
    const pa::CallRange range(__func__);
    if (limit_ns < 1000 || limit_ns > 1000000000) return PA_ERR_INVALID_ARG;
    if (report && (reinterpret_cast<uintptr_t>(report) & 7u) != 0) return PA_ERR_INVALID_ARG;
    unsigned int *err = nullptr;
    if (int rc = error_word(&err)) return rc;
    if (pa::launch_bounded_wait_check((unsigned long long)limit_ns, report, err,
                                      static_cast<cudaStream_t>(stream)) != 0)
        return PA_ERR_CUDA;
    return PA_OK;
}

int pa_get_device_error(void *stream, uint32_t *bits) {
    const pa::CallRange range(__func__);
    if (!bits) return PA_ERR_INVALID_ARG;
    *bits = 0;
    unsigned int *err = nullptr;
    if (int rc = error_word(&err)) return rc;
    cudaStream_t s = static_cast<cudaStream_t>(stream);
    unsigned int host = 0;
    if (cudaStreamSynchronize(s) != cudaSuccess) return PA_ERR_CUDA;
    if (cudaMemcpyAsync(&host, err, sizeof host, cudaMemcpyDeviceToHost, s) != cudaSuccess) return PA_ERR_CUDA;
    if (cudaMemsetAsync(err, 0, sizeof host, s) != cudaSuccess) return PA_ERR_CUDA;
    if (cudaStreamSynchronize(s) != cudaSuccess) return PA_ERR_CUDA;
    *bits = host;
    return host ? PA_ERR_DEVICE_INDEX : PA_OK;
}

}  // extern "C"
