/*
 * pa.h -- C ABI of the GB300 (sm_103a) paged decode-attention library.
 *
 * The library implements the data-parallel hot path of PagedAttention decode:
 * every running sequence's single new query token attends over a KV cache
 * that is split into fixed-size physical blocks reached through a per-sequence
 * block table.
 *
 *   Page A = "LLM推理优化：vLLM PagedAttention深度解析与工程实践"
 *   Page B = "vLLM 核心：PagedAttention 与 Continuous Batching"
 *   Page C = nano-vllm walkthrough, lqnn.cn/news/170268
 *   Page D = "优化大模型推理：PagedAttention 如何实现 GPU 显存高效管理"
 *
 * Conventions shared by every call
 * --------------------------------
 *  - All pointers except scalars are DEVICE pointers on the current CUDA
 *    device.  All tensors are dense, row-major (C order) and start on a 16-byte
 *    boundary.  The caller owns every buffer, the decode workspace included;
 *    the library allocates no memory.
 *  - KV cache layout (one layer, K and V in separate tensors):
 *        k_cache, v_cache : [num_blocks, block_size, num_kv_heads, head_dim]
 *    (Page A §4.1; Page C §2.2 gives the per-model form
 *    [layers, 2, blocks, block_size, heads, head_dim], of which these are
 *    one layer's K and V slices.)
 *  - A cache slot is  slot = physical_block * block_size + offset_in_block.
 *  - Element types: PA_F16 (IEEE binary16) or PA_BF16 for q/K/V; the decode
 *    output may also be PA_F32.  Arithmetic is fp32 (Page C §6: accumulating
 *    QK^T in half precision overflowed on long sequences).
 *  - FP8 KV cache (Page A §八 lists FP8 among vLLM's quantisation options):
 *    caches of PA_FP8_E4M3 hold one e4m3 code per element (bias 7, no
 *    infinities, largest value 448) with one scale per tensor: a K code c
 *    stands for value(c) * k_scale, V alike.  Writing quantises
 *    code = e4m3(fp32(x) / scale): the division in fp32 (IEEE), rounding to
 *    nearest-even, finite values saturating at +-448, NaN staying NaN.  The
 *    FP8 cache is supported for head_dim 128.
 *  - Supported shapes: head_dim 64 or 128; block_size 8 or a multiple of 16
 *    up to 256; num_heads a multiple of num_kv_heads with
 *    num_heads / num_kv_heads in {1, 2, 4, 8}.
 *  - `stream` is a cudaStream_t passed as void* (NULL = legacy default
 *    stream).  Every call only enqueues work and returns; host-side argument
 *    checks are synchronous and enqueue nothing when they fail.
 *  - `err_flag` (nullable, device int) collects problems found on the device.
 *    Kernels never trap and never spin without bound: a bad index is skipped
 *    and reported by atomically OR-ing a PA_FLAG_* bit into *err_flag.  The
 *    caller reads it after synchronising; any non-zero value means the
 *    affected outputs are not to be trusted (PA_ERR_DEVICE_BOUNDS).
 *    PA_FLAG_TIMEOUT means a bounded wait gave up: that call's outputs are
 *    undefined (a split sequence's merge may then read partial results that
 *    an earlier call left in the workspace).
 *  - Calls are not re-entrant on the same workspace: two pa_decode calls that
 *    may overlap on the GPU need two workspaces.
 *  - Tuning overrides.  The library chooses its kernels and their launch
 *    shapes itself; these environment variables, read once at the first
 *    decode call of the process, override that choice for tuning and testing.
 *    Under any setting the results stay within the documented tolerances and
 *    only the speed changes; leave them unset in deployment.
 *      PA_DECODE_COOP=0          run every decode on the per-warp kernel
 *                                (otherwise shapes with head_dim 128, KV heads
 *                                a multiple of 8 and block_size a multiple of
 *                                16 run on the CTA-cooperative kernel)
 *      PA_DECODE_COOP_STAGES=n   ring depth of the cooperative kernel (2..8)
 *      PA_DECODE_STAGES=n        ring depth per warp of the per-warp kernel (2..8)
 *      PA_DECODE_WARPS=n         warps per CTA of the per-warp kernel (1..16)
 *      PA_DECODE_INTERLEAVE=0    per-warp kernel: each warp takes a contiguous
 *                                run of its CTA's items instead of every n-th
 */
#ifndef PA_H_
#define PA_H_

#include <stddef.h>
#include <stdint.h>

#ifdef __cplusplus
extern "C" {
#endif

typedef enum {
    PA_OK = 0,
    PA_ERR_INVALID_ARG = 1,    /* null pointer, bad size, misaligned pointer */
    PA_ERR_UNSUPPORTED = 2,    /* valid request outside the supported shapes */
    PA_ERR_CUDA = 3,           /* a CUDA runtime/driver call failed */
    PA_ERR_WORKSPACE = 4,      /* decode workspace missing or too small */
    PA_ERR_DEVICE_BOUNDS = 5   /* returned by pa_check_err_flag for a non-zero flag */
} pa_status;

typedef enum { PA_F16 = 0, PA_BF16 = 1, PA_F32 = 2, PA_FP8_E4M3 = 3 } pa_dtype;

/* Bits OR-ed into *err_flag by the kernels. */
#define PA_FLAG_BAD_SLOT        0x1   /* slot_mapping entry >= num_blocks * block_size */
#define PA_FLAG_BAD_BLOCK_ID    0x2   /* block table entry outside [0, num_blocks) */
#define PA_FLAG_BAD_CONTEXT_LEN 0x4   /* context length < 0 or beyond the table/bound */
#define PA_FLAG_BAD_COPY_PAIR   0x8   /* copy pair id outside [0, num_blocks) */
#define PA_FLAG_TIMEOUT         0x10  /* a bounded wait on an async copy gave up */

/*
 * pa_reshape_and_cache -- write this step's new K/V rows into their slots.
 *
 * Defined by Page C §2.2 (a new token goes into the current physical block
 * while it has room, else a new block is taken and the table extended) and
 * §2.3 step 3 (write back and update the block's token count); Page A §二
 * (each step appends the new token's K and V to the cache).
 *
 *   key, value   : [num_tokens, num_kv_heads, head_dim], dtype (F16 or BF16)
 *   k_cache/v_cache : [num_blocks, block_size, num_kv_heads, head_dim],
 *                  cache_dtype (= dtype, or PA_FP8_E4M3)
 *   slot_mapping : [num_tokens] int64.  For token t with slot >= 0:
 *                    k_cache[slot / bs][slot % bs][h][:] = key[t][h][:]
 *                    v_cache[slot / bs][slot % bs][h][:] = value[t][h][:]
 *                  slot < 0 means "no write" (padding token).
 *   k_scale, v_scale : FP8 caches only (> 0): code = e4m3(x / scale).
 * A 16-bit copy is bit-exact.  Slots must be distinct (else the surviving row
 * is unspecified).  slot >= num_blocks * block_size: skipped,
 * PA_FLAG_BAD_SLOT.  num_tokens == 0 is a no-op.
 */
pa_status pa_reshape_and_cache(const void *key, const void *value,
                               void *k_cache, void *v_cache,
                               const int64_t *slot_mapping, int64_t num_tokens,
                               int64_t num_blocks, int block_size,
                               int num_kv_heads, int head_dim, pa_dtype dtype,
                               pa_dtype cache_dtype, float k_scale, float v_scale,
                               int *err_flag, void *stream);

/*
 * pa_decode_workspace_size -- bytes of workspace pa_decode needs.
 *
 * Returns 0 when no sequence can be split (max_context_len fits in one
 * partition).  The workspace holds the per-partition partial results of split
 * sequences (running max, sum of exponentials, unnormalised weighted V sum,
 * fp32).  It needs no initial contents: every partial is written before it is
 * read, within the same call.
 * `partition_size` is the same value later passed to pa_decode (0 = auto).
 * Returns (size_t)-1 for arguments pa_decode would reject.
 */
size_t pa_decode_workspace_size(int num_seqs, int num_heads, int num_kv_heads,
                                int head_dim, int block_size, int max_context_len,
                                int partition_size);

/* Zero-fill a decode workspace (stream-ordered memset); optional, since the
 * workspace needs no initial contents. */
pa_status pa_decode_workspace_init(void *workspace, size_t workspace_bytes, void *stream);

/* The partition length, in tokens, pa_decode uses for these arguments. */
int pa_decode_partition_size(int num_seqs, int num_heads, int num_kv_heads,
                             int head_dim, int block_size, int max_context_len,
                             int partition_size);

/*
 * pa_decode -- paged decode attention for one query token per sequence.
 *
 * For sequence s and query head h, with G = num_heads / num_kv_heads and the
 * KV head kvh = h / G (consecutive grouping; Page D's size formula counts
 * H_kv KV heads):
 *     x_p   = scale * <query[s][h][:], K_p>,  p = 0 .. context_lens[s]-1
 *     K_p   = k_cache[block_tables[s][p / bs]][p % bs][kvh][:]   (V_p alike)
 *     out[s][h][:] = sum_p softmax(x)_p * V_p
 * i.e. softmax(q K^T * scale) V (Page A §二) over the sequence's logical
 * context, gathered through its block table (Page A §3.1, §4.1; Page B §3;
 * Page C §2.3 steps 1-2).  Slots at positions >= context_lens[s] are never
 * read, so stale data there cannot leak in (Page C §6).
 *
 * Long contexts are cut into partitions of `partition_size` tokens (0 = auto)
 * whose partial results (max, sum, weighted V sum) are merged in partition
 * order -- the "partial accumulate, then merge" kernel of Page A §4.1.  The
 * result does not depend on the physical block ids or on the GPU schedule
 * and is bitwise reproducible run to run for a given partition size.
 *
 *   out          : [num_seqs, num_heads, head_dim], out_dtype (F16/BF16/F32)
 *   query        : [num_seqs, num_heads, head_dim], q_dtype (F16 or BF16)
 *   k_cache/v_cache : [num_blocks, block_size, num_kv_heads, head_dim], kv_dtype:
 *                  q_dtype, or PA_FP8_E4M3 with k_scale / v_scale (> 0;
 *                  ignored for 16-bit caches).  With an FP8 cache the
 *                  products run in binary16: e4m3 values are exact there and
 *                  a bfloat16 query is rounded to binary16 (exact for
 *                  |q| in [2^-14, 65504]).
 *   block_tables : [num_seqs, max_blocks_per_seq] int32; only the first
 *                  ceil(context_lens[s] / bs) entries of row s are read.
 *                  Sequences may share physical blocks.  Where neighbouring
 *                  rows start with the same block id, the blocks they share
 *                  must form a common prefix of both rows (as copy-on-write
 *                  sharing produces: once two rows differ, no later entry is
 *                  shared again).  With a 16-bit cache, head_dim 128, KV heads
 *                  a multiple of 8 and a group size of 1 or 2, such a run of
 *                  sequences is served from one copy of each shared block,
 *                  the shared length found by bisection on that property;
 *                  rows that share a block again after a differing one read
 *                  the first row's blocks in between.
 *   context_lens : [num_seqs] int32, each in [0, max_context_len]; 0 gives a
 *                  zero output row
 *   max_context_len : host-known upper bound of context_lens (sizes the
 *                  workspace); must be <= max_blocks_per_seq * block_size
 *   scale        : softmax scale, usually 1/sqrt(head_dim)
 *   partition_size : 0 (auto) or a multiple of 16 tokens, at most
 *                  32 * block_size
 *   workspace    : device buffer of pa_decode_workspace_size(...) bytes
 *                  (may be NULL if that size is 0)
 * Device-side problems: a block id outside [0, num_blocks) is not read, its
 * tokens are left out of the softmax and PA_FLAG_BAD_BLOCK_ID is set; a
 * context length outside [0, max_context_len] gives a zero row and
 * PA_FLAG_BAD_CONTEXT_LEN.
 */
pa_status pa_decode(void *out, pa_dtype out_dtype,
                    const void *query, pa_dtype q_dtype,
                    const void *k_cache, const void *v_cache, pa_dtype kv_dtype,
                    float k_scale, float v_scale,
                    const int32_t *block_tables, int max_blocks_per_seq,
                    const int32_t *context_lens, int max_context_len,
                    int num_seqs, int num_heads, int num_kv_heads, int head_dim,
                    int block_size, int64_t num_blocks, float scale,
                    int partition_size,
                    void *workspace, size_t workspace_bytes,
                    int *err_flag, void *stream);

/*
 * pa_decode_append -- reshape_and_cache of the step's new token fused with
 * pa_decode.
 *
 * For caches that pa_decode runs on its cooperative kernel (16-bit or e4m3,
 * head_dim 128, KV heads a multiple of 8, block size a multiple of 16), a
 * small kernel writes the new rows (quantised for e4m3) and the decode kernel,
 * chained to it by programmatic dependent launch, waits for it only before
 * the stages holding those rows; otherwise (other shapes) one decode kernel
 * does both.
 *
 * Each decode step appends one token per sequence and then attends over the
 * context including it (Page C §2.3 steps 1-3; Page A §二).  Here the new
 * token of sequence s is position context_lens[s] - 1: its K/V rows
 *   key, value : [num_seqs, num_kv_heads, head_dim], q_dtype
 * are written to the slot the block table gives for that position,
 *   block_tables[s][(ctx - 1) / bs] * bs + (ctx - 1) % bs,
 * (quantised as by pa_reshape_and_cache for an FP8 cache) and the attention
 * uses them; the result equals pa_reshape_and_cache with that slot mapping
 * followed by pa_decode, and the caches are bit-identical afterwards.  All
 * other arguments and rules are those of pa_decode; the caches are written.
 * A sequence with context length 0 appends nothing.  The last block of every
 * sequence must be private to it (copy shared blocks first, pa_copy_blocks).
 */
pa_status pa_decode_append(void *out, pa_dtype out_dtype,
                           const void *query, pa_dtype q_dtype,
                           const void *key, const void *value,
                           void *k_cache, void *v_cache, pa_dtype kv_dtype,
                           float k_scale, float v_scale,
                           const int32_t *block_tables, int max_blocks_per_seq,
                           const int32_t *context_lens, int max_context_len,
                           int num_seqs, int num_heads, int num_kv_heads, int head_dim,
                           int block_size, int64_t num_blocks, float scale,
                           int partition_size,
                           void *workspace, size_t workspace_bytes,
                           int *err_flag, void *stream);

/*
 * pa_decode_noalloc -- pa_decode for callers that cannot allocate device memory.
 *
 * The pages have no counterpart to this call; it exists for callers of this
 * library that cannot allocate, and so cannot supply pa_decode's workspace:
 * code running inside a host framework that owns all device memory and
 * forbids allocation while it executes (an inference engine plugin's execute
 * step, for example), or a deployment whose device-memory budget is fixed
 * when the library loads.
 *
 * Arguments and results are those of pa_decode without the workspace.  The
 * workspace is instead a scratch array of PA_NOALLOC_SCRATCH_BYTES inside the
 * library (a static __device__ array): every GPU that loads the library holds
 * that memory until the process exits.  The call allocates nothing - no
 * cudaMalloc, cudaFree or allocating library routine.
 *  - Arguments are checked exactly as pa_decode checks them; then, when
 *    pa_decode_workspace_size(...) for these arguments exceeds
 *    PA_NOALLOC_SCRATCH_BYTES, the call returns PA_ERR_WORKSPACE and enqueues
 *    nothing (use a larger partition_size, fewer sequences, or pa_decode with
 *    a workspace of your own).
 *  - The first call in each CUDA context - once per device with the runtime's
 *    primary contexts, again after cudaDeviceReset or under another context -
 *    looks up the array's device address (cudaGetSymbolAddress, with the
 *    device current) and caches it for that context; make that first call
 *    before any stream capture on the device.
 *  - Every call on a device shares the one array, which keeps the previous
 *    call's contents; nothing in it needs clearing between calls (every
 *    partial result is written before it is read within a call that completes
 *    without PA_FLAG_TIMEOUT).  Calls that may overlap on the GPU - different
 *    streams, threads or processes' shared contexts - race on the array and
 *    corrupt each other's results: order them (one stream, or events).
 */
#define PA_NOALLOC_SCRATCH_BYTES (32u * 1024u * 1024u)
pa_status pa_decode_noalloc(void *out, pa_dtype out_dtype,
                            const void *query, pa_dtype q_dtype,
                            const void *k_cache, const void *v_cache, pa_dtype kv_dtype,
                            float k_scale, float v_scale,
                            const int32_t *block_tables, int max_blocks_per_seq,
                            const int32_t *context_lens, int max_context_len,
                            int num_seqs, int num_heads, int num_kv_heads, int head_dim,
                            int block_size, int64_t num_blocks, float scale,
                            int partition_size, int *err_flag, void *stream);

/*
 * pa_prefill -- causal attention of each sequence's new tokens over its
 * paged context (prefill after a prefix-cache hit, or one chunk of a
 * chunked prefill).
 *
 * When a request's prefix is already cached, only its tail is computed: the
 * tail's query tokens attend to the cached prefix blocks and, causally, to
 * each other (Page C §3.4 with the block table and slot layout of §2.2;
 * Page A §二).  Sequence s owns query rows cu_seqlens_q[s] ..
 * cu_seqlens_q[s+1]-1, its q_len = cu_seqlens_q[s+1] - cu_seqlens_q[s] newest
 * tokens; with ctx = context_lens[s], its query token i sits at position
 * ctx - q_len + i, and for query head h (kvh = h / G):
 *     out[row][h][:] = sum_{p <= ctx - q_len + i} softmax(x)_p * V_p,
 *     x_p = scale * <query[row][h][:], K_p>,  row = cu_seqlens_q[s] + i,
 * K_p / V_p gathered through the block table as in pa_decode.  Each query
 * token's result is exactly pa_decode's for a context of (its position + 1)
 * tokens.  The K/V rows of the new tokens must already be in the cache
 * (pa_reshape_and_cache first).
 *
 *   out          : [num_tokens, num_heads, head_dim], out_dtype (F16/BF16/F32)
 *   query        : [num_tokens, num_heads, head_dim], kv_dtype
 *   k_cache/v_cache : [num_blocks, block_size, num_kv_heads, head_dim], F16 or
 *                  BF16 (the query's type; FP8 caches are not supported here)
 *   block_tables : [num_seqs, max_blocks_per_seq] int32
 *   context_lens : [num_seqs] int32, total tokens of each sequence including
 *                  its new ones; q_len <= ctx <= max_blocks_per_seq * bs
 *   cu_seqlens_q : [num_seqs + 1] int32 (device), cu_seqlens_q[0] = 0,
 *                  non-decreasing, cu_seqlens_q[num_seqs] <= num_tokens
 *   max_q_len    : host-known upper bound of every q_len (sizes the grid)
 *   scale        : softmax scale, > 0 (usually 1/sqrt(head_dim))
 * Supported: head_dim 64 or 128; block_size 8, 16, 32, 64 or 128;
 * num_heads / num_kv_heads a power of two up to 128.  Products run on the
 * tensor cores with fp32 accumulation; the softmax weights are rounded to
 * binary16, or for bfloat16 inputs split into two bfloat16 parts.
 * Device-side problems: an invalid cu_seqlens_q entry sets
 * PA_FLAG_BAD_CONTEXT_LEN and leaves that sequence's rows unwritten; a q_len
 * above max_q_len sets it too, and rows beyond the 128/G-token query tiles
 * the bound implies are left unwritten; a context length outside [q_len, max_blocks_per_seq * bs] gives
 * zero rows and PA_FLAG_BAD_CONTEXT_LEN; a block id outside [0, num_blocks)
 * is not read, sets PA_FLAG_BAD_BLOCK_ID and gives zero rows for the query
 * tiles that needed it.  No workspace; nothing is allocated.
 */
pa_status pa_prefill(void *out, pa_dtype out_dtype,
                     const void *query,
                     const void *k_cache, const void *v_cache, pa_dtype kv_dtype,
                     const int32_t *block_tables, int max_blocks_per_seq,
                     const int32_t *context_lens, const int32_t *cu_seqlens_q,
                     int num_seqs, int64_t num_tokens, int max_q_len,
                     int num_heads, int num_kv_heads, int head_dim,
                     int block_size, int64_t num_blocks, float scale,
                     int *err_flag, void *stream);

/*
 * pa_copy_blocks -- copy-on-write of shared blocks.
 *
 * A block referenced by several sequences is read-only; before one of them
 * writes into it, the block is copied to a fresh one (Page D, copy-on-write
 * section: parallel sampling of one prompt; Page A §3.1; Page B §3 prefix
 * sharing).  For every pair p:
 *     k_cache[dst_p] = k_cache[src_p],  v_cache[dst_p] = v_cache[src_p]
 * (whole blocks: block_size * num_kv_heads * head_dim elements each, of
 * `dtype`: F16, BF16 or FP8_E4M3), bit-exact.
 *
 *   block_mapping : [num_pairs, 2] int64 (src, dst), device memory
 * Destinations must be distinct and no destination may also be a source
 * (else the result depends on order and is unspecified).  A pair with an id
 * outside [0, num_blocks) is skipped and sets PA_FLAG_BAD_COPY_PAIR.
 * num_pairs == 0 is a no-op.
 */
pa_status pa_copy_blocks(void *k_cache, void *v_cache,
                         const int64_t *block_mapping, int64_t num_pairs,
                         int64_t num_blocks, int block_size, int num_kv_heads,
                         int head_dim, pa_dtype dtype, int *err_flag, void *stream);

/*
 * pa_copy_blocks_layers -- pa_copy_blocks for every layer of a model's cache
 * in one launch.
 *
 * The per-model cache is one tensor [layers, 2, blocks, block_size, heads,
 * head_dim] (Page C §2.2): layer l's K cache is kv_cache[l][0] and its V cache
 * kv_cache[l][1].  A sequence's physical blocks are the same in every layer,
 * so one (src, dst) pair list copies the block in all of them:
 *     kv_cache[l][0][dst_p] = kv_cache[l][0][src_p],
 *     kv_cache[l][1][dst_p] = kv_cache[l][1][src_p]   for every layer l,
 * bit-exact; rules and device-side checks as for pa_copy_blocks.
 *
 *   kv_cache      : [num_layers, 2, num_blocks, block_size, num_kv_heads,
 *                   head_dim] of `dtype` (F16, BF16 or FP8_E4M3), contiguous
 *   block_mapping : [num_pairs, 2] int64 (src, dst), device memory
 * num_layers == 0 or num_pairs == 0 is a no-op; at most 65535 layers.
 */
pa_status pa_copy_blocks_layers(void *kv_cache, int num_layers,
                                const int64_t *block_mapping, int64_t num_pairs,
                                int64_t num_blocks, int block_size, int num_kv_heads,
                                int head_dim, pa_dtype dtype, int *err_flag, void *stream);

/*
 * pa_swap_blocks -- copy whole blocks between two caches.
 *
 * Swap-mode preemption moves a preempted request's KV blocks from GPU memory
 * to CPU memory and back when it resumes (Page B §5, strategy 1: swapping);
 * the block table then names the blocks' new physical ids.  For every pair p:
 *     dst_k[dst_p] = src_k[src_p],  dst_v[dst_p] = src_v[src_p]
 * (whole blocks of block_size * num_kv_heads * head_dim elements of `dtype`),
 * bit-exact.  src and dst are [src_num_blocks, ...] and [dst_num_blocks, ...]
 * caches; either may live in page-locked host memory (cudaHostAlloc /
 * cudaHostRegister, which the GPU reads and writes directly over the
 * host link) and the other in device memory.  block_mapping [num_pairs, 2]
 * int64 (src, dst) may be device or page-locked host memory.  Every pointer is
 * checked with cudaPointerGetAttributes first: any other memory (e.g.
 * pageable host memory) gives PA_ERR_INVALID_ARG and nothing is launched.
 * Destinations must be distinct.  A pair with an id outside its cache is
 * skipped and sets PA_FLAG_BAD_COPY_PAIR.
 */
pa_status pa_swap_blocks(const void *src_k, const void *src_v, void *dst_k, void *dst_v,
                         const int64_t *block_mapping, int64_t num_pairs,
                         int64_t src_num_blocks, int64_t dst_num_blocks,
                         int block_size, int num_kv_heads, int head_dim, pa_dtype dtype,
                         int *err_flag, void *stream);

/* Host helper: synchronously read *err_flag (device), optionally clear it,
 * and map it to PA_OK / PA_ERR_DEVICE_BOUNDS.  `flag_out` (nullable, host)
 * receives the raw bits. */
pa_status pa_check_err_flag(int *err_flag, int clear, int *flag_out, void *stream);

/* A short, static description of a status code. */
const char *pa_status_string(pa_status status);

/* Library version as MAJOR * 10000 + MINOR * 100 + PATCH. */
int pa_version(void);

#ifdef __cplusplus
}
#endif

#endif /* PA_H_ */
