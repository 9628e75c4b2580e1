// Internal interface of the prefill kernel (causal attention of a chunk of
// new query tokens over a paged KV cache), shared by the C ABI in pa_api.cu
// and the kernel in pa_prefill.cu.
#pragma once

#include <cuda.h>
#include <cuda_runtime.h>
#include <stdint.h>

namespace pa {

constexpr int kPrefillTile = 128;       // rows of a query tile = KV tokens per stage
constexpr int kPrefillThreads = 352;    // 8 softmax warps, K/Q loader, MMA issuer, V loader
constexpr int kRankSeqs = 128;          // batches up to this many sequences run longest first

struct PrefillParams {
    const void *q;                  // [num_tokens, num_heads, head_dim]
    void *out;
    int out_dtype;                  // pa_dtype of out
    const int32_t *block_tables;    // [B, max_blocks_per_seq]
    const int32_t *context_lens;    // [B]
    const int32_t *cu_seqlens_q;    // [B + 1]
    int max_blocks_per_seq;
    int num_seqs;
    int64_t num_tokens;             // rows of query / out
    int num_heads;
    int num_kv_heads;
    int log2_group;                 // log2(num_heads / num_kv_heads)
    int block_size;
    int64_t num_blocks;
    int max_q_len;                  // host bound on every sequence's new-token count
    int tiles_per_seq;              // query tiles per sequence: ceil(max_q_len * group / 128)
    int pairs_per_seq;              // query-tile pairs per sequence: ceil(tiles_per_seq / 2)
    float scale_log2;               // softmax scale * log2(e)
    int *err_flag;
};

// Dynamic shared memory of one prefill CTA.
size_t prefill_smem_bytes(int head_dim);

// query [num_tokens, Hq, D] through `tq` (box 64 x G x 128/G); caches
// [NB * bs, Hkv, D] through `tk` / `tv` (box 64 x 1 x bs); the output through
// `to` (box 128 bytes x G x 128/G, written by full query tiles); all with
// 128-byte swizzle.
cudaError_t launch_prefill(const PrefillParams &p, int head_dim, bool bf16, const CUtensorMap &tq,
                           const CUtensorMap &tk, const CUtensorMap &tv, const CUtensorMap &to, size_t smem,
                           cudaStream_t stream);

}  // namespace pa
