// Internal launch interface of the 8-bit (OCP FP8 E4M3) cache path, between the
// C-ABI layer (capi.cu) and its kernel translation units. Not part of the
// public ABI.
#pragma once

#include <cuda_runtime.h>
#include <stdint.h>

#include "kernels.h"

namespace pa {

// Scatter with quantisation: element x of token t's K (V) row becomes the E4M3
// code nearest to the float32 quotient x / k_scale (x / v_scale), ties to even,
// saturating at 448. src_dtype: PA_DTYPE_F32, _F16 or _BF16. row_elems is
// num_kv_heads * head_dim, a multiple of 16.
int launch_kv_write_fp8(const void *k, const void *v, int src_dtype, const int32_t *slot_mapping,
                        int64_t num_tokens, void *key_cache, void *value_cache, int64_t num_slots,
                        int row_elems, float k_scale, float v_scale, unsigned int *err, cudaStream_t stream);

// Tensor-core decode over E4M3 caches (query/output bf16 or f16, head_dim 128,
// group <= 16, block size 8..128). p.scale_log2 must already include k_scale;
// v_scale multiplies the output. Partials for multi-partition sequences go to
// p.ws_ml / p.ws_o for launch_decode_reduce. With p.app_slots set (decode with
// append) the kernel also quantises and stores each sequence's new K/V row
// (p.app_k / p.app_v, in the query dtype) with k_scale / v_scale, as
// launch_kv_write_fp8 would, before it reads that row's block.
bool decode_fp8_supported(const DecodeParams &p, int dtype);
int launch_decode_fp8(const DecodeParams &p, float v_scale, float k_scale, int dtype, cudaStream_t stream);

}  // namespace pa
