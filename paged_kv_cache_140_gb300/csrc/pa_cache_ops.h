// Host-side interface between the C ABI (pa_api.cu) and the cache-op kernels
// (pa_cache_ops.cu): reshape_and_cache and whole-block copies.
#pragma once

#include <cuda_runtime.h>
#include <stdint.h>

namespace pa {

cudaError_t launch_reshape_and_cache(const void *key, const void *value, void *k_cache,
                                     void *v_cache, const int64_t *slot_mapping,
                                     int64_t num_tokens, int64_t num_slots, int64_t row_bytes,
                                     int *err_flag, cudaStream_t stream);

// One 16-bit row per sequence ([num_seqs, row_bytes]) written at the slot the
// block table gives position context_lens[s] - 1 (the decode step's append).
cudaError_t launch_append_rows(const void *key, const void *value, void *k_cache, void *v_cache,
                               const int32_t *block_tables, const int32_t *context_lens,
                               int max_blocks_per_seq, int max_context_len, int block_size,
                               int64_t num_blocks, int num_seqs, int64_t row_bytes, int *err_flag,
                               cudaStream_t stream);

// The same append into an e4m3 cache: 16-bit rows ([num_seqs, row_elems],
// bf16 if `bf16`) quantised as by launch_reshape_and_cache_fp8.
cudaError_t launch_append_rows_fp8(const void *key, const void *value, void *k_cache, void *v_cache,
                                   const int32_t *block_tables, const int32_t *context_lens,
                                   int max_blocks_per_seq, int max_context_len, int block_size,
                                   int64_t num_blocks, int num_seqs, int64_t row_elems, bool bf16,
                                   float k_scale, float v_scale, int *err_flag, cudaStream_t stream);

// Quantising variant: 16-bit rows (bf16 if `bf16`) -> e4m3 codes of
// x / scale; `row_elems` elements per token row (a multiple of 8).
cudaError_t launch_reshape_and_cache_fp8(const void *key, const void *value, void *k_cache,
                                         void *v_cache, const int64_t *slot_mapping,
                                         int64_t num_tokens, int64_t num_slots, int64_t row_elems,
                                         bool bf16, float k_scale, float v_scale, int *err_flag,
                                         cudaStream_t stream);

// Whole-block copies src -> dst (the same cache for copy_blocks), repeated for
// `layers` layers whose K/V caches lie `layer_bytes` apart (layers = 1,
// layer_bytes = 0 for a single layer).
cudaError_t launch_copy_blocks(const void *src_k, const void *src_v, void *dst_k, void *dst_v,
                               const int64_t *block_mapping, int64_t num_pairs, int64_t src_blocks,
                               int64_t dst_blocks, int64_t block_bytes, int *err_flag,
                               cudaStream_t stream, int layers = 1, int64_t layer_bytes = 0);

}  // namespace pa
