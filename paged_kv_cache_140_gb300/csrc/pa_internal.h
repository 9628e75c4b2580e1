// Host-side interface between the C ABI (pa_api.cu) and the decode kernel file.
#pragma once

#include <cuda.h>
#include <cuda_runtime.h>
#include <stdint.h>

namespace pa {

// Tokens per pipeline stage of the decode kernel: one stage brings 16 K rows
// and 16 V rows of one KV head into shared memory.
constexpr int kStageTokens = 16;
// Default ring depth (shared-memory slots) per warp and warps per CTA for
// 128-dim heads: 2 x 8 measured best on GB300 for every workload tried (13B,
// 7B, GQA, prefix sharing); deeper rings or more warps only add L2/HBM queueing.
constexpr int kDefaultStages = 2;
constexpr int kDefaultWarps128 = 8;
// e4m3 caches: a slot carries two 16-token stages (8 KB of K and V); 12
// warps fill shared memory (measured best: 8 warps 341 us, 11 293.5, 12 268.4
// on the 13B-shaped step).
constexpr int kDefaultWarpsFp8 = 12;

struct DecodeParams {
    void *out;
    int out_dtype;               // pa_dtype value
    const void *q;               // [B, Hq, D]
    const int32_t *block_tables; // [B, max_blocks_per_seq]
    const int32_t *context_lens; // [B]
    int max_blocks_per_seq;
    int max_context_len;
    int num_seqs;
    int num_heads;
    int num_kv_heads;
    int block_size;
    int64_t num_blocks;
    float scale_log2;            // softmax scale * log2(e) * k_scale (k_scale = 1 for 16-bit caches)
    float v_scale;               // e4m3 caches: V code scale (1 for 16-bit caches)
    int partition_size;          // tokens per partition, multiple of 16
    int max_partitions;          // partition slots per (seq, KV head) in the workspace
    float *ws_ml;                // [B * Hkv * max_partitions, G, 2]  (max, sum)
    float *ws_acc;               // [B * Hkv * max_partitions, G, D]
    int *err_flag;
    // Fused append (pa_decode_append): the step's new K/V rows, one per
    // sequence [B, Hkv, D] in the query's 16-bit type, written at position
    // context_lens[s] - 1 into the caches below; nullptr for plain decode.
    const void *new_k;
    const void *new_v;
    void *k_cache_w;
    void *v_cache_w;
    float k_scale_w;             // e4m3 caches: quantisation scales of the new rows
    float v_scale_w;
    int stages;                  // shared-memory slots per warp (ring depth)
    int interleave;              // 1: a CTA's warps take every nw-th item of the CTA's range
    int defer_wait;              // cooperative kernel: the previous kernel in the stream is the
                                 // step's append (it writes only the rows at positions ctx - 1),
                                 // so its completion is awaited only before those rows are read
};

// Shared memory the decode kernel needs for `warps` warps with `stages`
// slots each and `num_seqs` sequences (including alignment slack).
size_t decode_smem_bytes(int head_dim, int group, int elem_bytes, int warps, int stages,
                         int num_seqs);

// The CTA-cooperative decode kernel (pa_decode_coop.cu): 16-bit or e4m3
// caches (`es` 2 or 1 bytes per element), head dim 128, KV heads a multiple of
// 8, block size a multiple of 16; `tk`/`tv` map each cache as (dim, token,
// head) with {128 bytes, 16, 8} boxes.  `kv` as for launch_decode (0 f16,
// 1 bf16, 2/3 e4m3 with an f16/bf16 query).  Launches the merge kernel after
// it when sequences are split.
size_t decode_coop_smem_bytes(int group, int es, int stages, int num_seqs);
cudaError_t launch_decode_coop(const DecodeParams &p, int group, int kv, const CUtensorMap &tk,
                               const CUtensorMap &tv, int grid, size_t smem, cudaStream_t stream);

// The merge of split sequences' partial states (pa_decode.cu), chained with
// programmatic dependent launch; nothing is launched when no sequence splits.
cudaError_t launch_decode_merge(const DecodeParams &p, int head_dim, int group, cudaStream_t stream);


// kv: 0 = f16 cache/query, 1 = bf16, 2 = e4m3 cache + f16 query, 3 = e4m3 + bf16.
cudaError_t launch_decode(const DecodeParams &p, int head_dim, int group, int kv,
                          const CUtensorMap &tmap_k, const CUtensorMap &tmap_v, int grid,
                          int warps, size_t smem, cudaStream_t stream);

}  // namespace pa
