// reshape_and_cache and copy_blocks for sm_103a: bit-exact row and block
// copies with 16-byte vector accesses.
//
// reshape_and_cache writes each new token's K/V row ([Hkv, D], contiguous in
// both the source and the cache) into its slot, slot = block * bs + offset
// (nano-vllm walkthrough lqnn.cn/news/170268, §2.2 and §2.3 step 3).
// copy_blocks duplicates whole physical blocks for copy-on-write
// ("优化大模型推理：PagedAttention 如何实现 GPU 显存高效管理", copy-on-write
// section).  Both are pure data movement bound by HBM bandwidth; grids are
// sized in multiples of the SM count by the host.
#include "pa_cache_ops.h"
#include "pa_device.cuh"

namespace pa {

namespace {

// grid.x: tokens (grid-stride); a CTA moves a token's whole K and V row, each
// thread up to 8 + 8 16-byte chunks at a time with all loads issued before
// the stores, and with up to 16 CTAs per SM many tokens are in flight.  The
// kernel lets the next kernel in the stream (normally the decode, launched
// with programmatic dependent launch) start early; that kernel still waits
// for this one to complete before reading.
__global__ void __launch_bounds__(128)
    reshape_and_cache_kernel(const uint4 *__restrict__ key, const uint4 *__restrict__ value,
                             uint4 *__restrict__ k_cache, uint4 *__restrict__ v_cache,
                             const int64_t *__restrict__ slot_mapping, int64_t num_tokens,
                             int64_t num_slots, int64_t row16, int *err_flag) {
    pdl_launch_dependents();
    constexpr int kU = 8;
    for (int64_t t = blockIdx.x; t < num_tokens; t += gridDim.x) {
        const int64_t slot = slot_mapping[t];
        if (slot < 0) continue;
        if (slot >= num_slots) {
            if (threadIdx.x == 0) report(err_flag, 0x1 /* PA_FLAG_BAD_SLOT */);
            continue;
        }
        const uint4 *ks = key + t * row16;
        const uint4 *vs = value + t * row16;
        uint4 *kd = k_cache + slot * row16;
        uint4 *vd = v_cache + slot * row16;
        for (int64_t c0 = threadIdx.x; c0 < row16; c0 += kU * blockDim.x) {
            uint4 a[kU], b[kU];
#pragma unroll
            for (int u = 0; u < kU; ++u) {
                const int64_t c = c0 + u * blockDim.x;
                if (c < row16) {
                    a[u] = __ldg(ks + c);
                    b[u] = __ldg(vs + c);
                }
            }
#pragma unroll
            for (int u = 0; u < kU; ++u) {
                const int64_t c = c0 + u * blockDim.x;
                if (c < row16) {
                    kd[c] = a[u];
                    vd[c] = b[u];
                }
            }
        }
    }
}

// One new token per sequence, written where the sequence's block table puts
// position context_lens[s] - 1 (the decode step's append): the same bytes
// reshape_and_cache writes for that slot.  Sequences with no valid token
// (length <= 0 or above the bound) write nothing; a block id outside the pool
// is flagged and skipped.  Like reshape_and_cache it lets the next kernel (the
// decode, launched with programmatic dependent launch) start early.
__global__ void __launch_bounds__(128)
    append_rows_kernel(const uint4 *__restrict__ key, const uint4 *__restrict__ value,
                       uint4 *__restrict__ k_cache, uint4 *__restrict__ v_cache,
                       const int32_t *__restrict__ block_tables, const int32_t *__restrict__ context_lens,
                       int max_blocks_per_seq, int max_context_len, int block_size, int64_t num_blocks,
                       int num_seqs, int64_t row16, int *err_flag) {
    pdl_launch_dependents();
    constexpr int kU = 8;
    for (int s = blockIdx.x; s < num_seqs; s += gridDim.x) {
        const int c = context_lens[s];
        if (c <= 0 || c > max_context_len) continue;
        const int pos = c - 1;
        const int blk = block_tables[static_cast<int64_t>(s) * max_blocks_per_seq + pos / block_size];
        if (blk < 0 || static_cast<int64_t>(blk) >= num_blocks) {
            if (threadIdx.x == 0) report(err_flag, 0x2 /* PA_FLAG_BAD_BLOCK_ID */);
            continue;
        }
        const int64_t slot = static_cast<int64_t>(blk) * block_size + pos % block_size;
        const uint4 *ks = key + s * row16;
        const uint4 *vs = value + s * row16;
        uint4 *kd = k_cache + slot * row16;
        uint4 *vd = v_cache + slot * row16;
        for (int64_t c0 = threadIdx.x; c0 < row16; c0 += kU * blockDim.x) {
            uint4 a[kU], b[kU];
#pragma unroll
            for (int u = 0; u < kU; ++u) {
                const int64_t i = c0 + u * blockDim.x;
                if (i < row16) {
                    a[u] = __ldg(ks + i);
                    b[u] = __ldg(vs + i);
                }
            }
#pragma unroll
            for (int u = 0; u < kU; ++u) {
                const int64_t i = c0 + u * blockDim.x;
                if (i < row16) {
                    kd[i] = a[u];
                    vd[i] = b[u];
                }
            }
        }
    }
}

// 8 elements of a 16-bit row -> 8 e4m3 codes, code = e4m3(x / scale) with
// the division in fp32 (IEEE, round to nearest) and nearest-even rounding that
// saturates finite values at +-448.
template <bool BF16>
__device__ __forceinline__ uint2 quant8(uint4 w, float sc) {
    const uint32_t in[4] = {w.x, w.y, w.z, w.w};
    uint32_t code[4];
#pragma unroll
    for (int k = 0; k < 4; ++k) {
        const float2 f = Half2x<BF16>::to_float2(in[k]);
        code[k] = f32x2_to_e4m3x2(__fdiv_rn(f.x, sc), __fdiv_rn(f.y, sc));
    }
    return make_uint2(code[0] | (code[1] << 16), code[2] | (code[3] << 16));
}

// Quantising variant for an e4m3 cache: each thread turns 8 elements of a
// 16-bit row into 8 codes (quant8).
template <bool BF16>
__global__ void __launch_bounds__(128)
    reshape_and_cache_fp8_kernel(const uint4 *__restrict__ key, const uint4 *__restrict__ value,
                                 uint2 *__restrict__ k_cache, uint2 *__restrict__ v_cache,
                                 const int64_t *__restrict__ slot_mapping, int64_t num_tokens,
                                 int64_t num_slots, int64_t row8, float k_scale, float v_scale,
                                 int *err_flag) {
    pdl_launch_dependents();
    const int64_t i = static_cast<int64_t>(blockIdx.y) * blockDim.x + threadIdx.x;
    for (int64_t t = blockIdx.x; t < num_tokens; t += gridDim.x) {
        const int64_t slot = slot_mapping[t];
        if (slot < 0) continue;
        if (slot >= num_slots) {
            if (threadIdx.x == 0 && blockIdx.y == 0) report(err_flag, 0x1 /* PA_FLAG_BAD_SLOT */);
            continue;
        }
        for (int64_t c = i; c < row8; c += static_cast<int64_t>(gridDim.y) * blockDim.x) {
            const uint4 a = __ldg(key + t * row8 + c);
            const uint4 b = __ldg(value + t * row8 + c);
            k_cache[slot * row8 + c] = quant8<BF16>(a, k_scale);
            v_cache[slot * row8 + c] = quant8<BF16>(b, v_scale);
        }
    }
}

// The decode step's append into an e4m3 cache: append_rows_kernel's slot
// rule, the codes of reshape_and_cache_fp8_kernel.
template <bool BF16>
__global__ void __launch_bounds__(128)
    append_rows_fp8_kernel(const uint4 *__restrict__ key, const uint4 *__restrict__ value,
                           uint2 *__restrict__ k_cache, uint2 *__restrict__ v_cache,
                           const int32_t *__restrict__ block_tables, const int32_t *__restrict__ context_lens,
                           int max_blocks_per_seq, int max_context_len, int block_size, int64_t num_blocks,
                           int num_seqs, int64_t row8, float k_scale, float v_scale, int *err_flag) {
    pdl_launch_dependents();
    for (int s = blockIdx.x; s < num_seqs; s += gridDim.x) {
        const int c = context_lens[s];
        if (c <= 0 || c > max_context_len) continue;
        const int pos = c - 1;
        const int blk = block_tables[static_cast<int64_t>(s) * max_blocks_per_seq + pos / block_size];
        if (blk < 0 || static_cast<int64_t>(blk) >= num_blocks) {
            if (threadIdx.x == 0) report(err_flag, 0x2 /* PA_FLAG_BAD_BLOCK_ID */);
            continue;
        }
        const int64_t slot = static_cast<int64_t>(blk) * block_size + pos % block_size;
        for (int64_t i = threadIdx.x; i < row8; i += blockDim.x) {
            const uint4 a = __ldg(key + s * row8 + i);
            const uint4 b = __ldg(value + s * row8 + i);
            k_cache[slot * row8 + i] = quant8<BF16>(a, k_scale);
            v_cache[slot * row8 + i] = quant8<BF16>(b, v_scale);
        }
    }
}

// grid.x: copy pairs (grid-stride), grid.y: slices of the block, grid.z:
// layers (caches `layer16` 16-byte units apart); each thread moves 4 chunks
// of 16 bytes of K and of V per iteration.  Source and destination are
// separate caches (swap_blocks: e.g. GPU and pinned host memory) or the same
// one (copy_blocks; its pairs never overlap).
__global__ void __launch_bounds__(256)
    copy_blocks_kernel(const uint4 *src_k, const uint4 *src_v, uint4 *dst_k, uint4 *dst_v,
                       const int64_t *__restrict__ block_mapping, int64_t num_pairs,
                       int64_t src_blocks, int64_t dst_blocks, int64_t block16, int64_t layer16,
                       int *err_flag) {
    const int64_t lo = static_cast<int64_t>(blockIdx.z) * layer16;
    src_k += lo;
    src_v += lo;
    dst_k += lo;
    dst_v += lo;
    const int64_t slice = (block16 + gridDim.y - 1) / gridDim.y;
    const int64_t beg = blockIdx.y * slice;
    const int64_t end = min(block16, beg + slice);
    for (int64_t pr = blockIdx.x; pr < num_pairs; pr += gridDim.x) {
        const int64_t src = block_mapping[2 * pr];
        const int64_t dst = block_mapping[2 * pr + 1];
        if (src < 0 || src >= src_blocks || dst < 0 || dst >= dst_blocks) {
            if (threadIdx.x == 0 && blockIdx.y == 0 && blockIdx.z == 0) report(err_flag, 0x8 /* PA_FLAG_BAD_COPY_PAIR */);
            continue;
        }
        const uint4 *ks = src_k + src * block16;
        const uint4 *vs = src_v + src * block16;
        uint4 *kd = dst_k + dst * block16;
        uint4 *vd = dst_v + dst * block16;
        int64_t i = beg + threadIdx.x;
        const int64_t step = blockDim.x;
        for (; i + 3 * step < end; i += 4 * step) {
            uint4 a[4], b[4];
#pragma unroll
            for (int u = 0; u < 4; ++u) { a[u] = ks[i + u * step]; b[u] = vs[i + u * step]; }
#pragma unroll
            for (int u = 0; u < 4; ++u) { kd[i + u * step] = a[u]; vd[i + u * step] = b[u]; }
        }
        for (; i < end; i += step) {
            kd[i] = ks[i];
            vd[i] = vs[i];
        }
    }
}

int sm_count() {
    int dev = 0, n = 0;
    if (cudaGetDevice(&dev) != cudaSuccess) return 148;
    if (cudaDeviceGetAttribute(&n, cudaDevAttrMultiProcessorCount, dev) != cudaSuccess) return 148;
    return n > 0 ? n : 148;
}

}  // namespace

cudaError_t launch_reshape_and_cache(const void *key, const void *value, void *k_cache,
                                     void *v_cache, const int64_t *slot_mapping,
                                     int64_t num_tokens, int64_t num_slots, int64_t row_bytes,
                                     int *err_flag, cudaStream_t stream) {
    const int64_t row16 = row_bytes / 16;
    const int threads = 128;
    // Up to 16 CTAs (tokens) per SM at a time; long token lists grid-stride.
    const int64_t cap = static_cast<int64_t>(sm_count()) * 16;
    const int64_t gx = num_tokens < cap ? num_tokens : cap;
    reshape_and_cache_kernel<<<static_cast<unsigned>(gx), threads, 0, stream>>>(
        static_cast<const uint4 *>(key), static_cast<const uint4 *>(value),
        static_cast<uint4 *>(k_cache), static_cast<uint4 *>(v_cache), slot_mapping, num_tokens,
        num_slots, row16, err_flag);
    return cudaGetLastError();
}

cudaError_t launch_append_rows(const void *key, const void *value, void *k_cache, void *v_cache,
                               const int32_t *block_tables, const int32_t *context_lens,
                               int max_blocks_per_seq, int max_context_len, int block_size,
                               int64_t num_blocks, int num_seqs, int64_t row_bytes, int *err_flag,
                               cudaStream_t stream) {
    const int64_t cap = static_cast<int64_t>(sm_count()) * 16;
    const int64_t gx = num_seqs < cap ? num_seqs : cap;
    if (gx <= 0) return cudaSuccess;
    append_rows_kernel<<<static_cast<unsigned>(gx), 128, 0, stream>>>(
        static_cast<const uint4 *>(key), static_cast<const uint4 *>(value), static_cast<uint4 *>(k_cache),
        static_cast<uint4 *>(v_cache), block_tables, context_lens, max_blocks_per_seq, max_context_len, block_size,
        num_blocks, num_seqs, row_bytes / 16, err_flag);
    return cudaGetLastError();
}

cudaError_t launch_append_rows_fp8(const void *key, const void *value, void *k_cache, void *v_cache,
                                   const int32_t *block_tables, const int32_t *context_lens,
                                   int max_blocks_per_seq, int max_context_len, int block_size,
                                   int64_t num_blocks, int num_seqs, int64_t row_elems, bool bf16,
                                   float k_scale, float v_scale, int *err_flag, cudaStream_t stream) {
    const int64_t cap = static_cast<int64_t>(sm_count()) * 16;
    const int64_t gx = num_seqs < cap ? num_seqs : cap;
    if (gx <= 0) return cudaSuccess;
    auto kern = bf16 ? append_rows_fp8_kernel<true> : append_rows_fp8_kernel<false>;
    kern<<<static_cast<unsigned>(gx), 128, 0, stream>>>(
        static_cast<const uint4 *>(key), static_cast<const uint4 *>(value), static_cast<uint2 *>(k_cache),
        static_cast<uint2 *>(v_cache), block_tables, context_lens, max_blocks_per_seq, max_context_len, block_size,
        num_blocks, num_seqs, row_elems / 8, k_scale, v_scale, err_flag);
    return cudaGetLastError();
}

cudaError_t launch_reshape_and_cache_fp8(const void *key, const void *value, void *k_cache,
                                         void *v_cache, const int64_t *slot_mapping,
                                         int64_t num_tokens, int64_t num_slots, int64_t row_elems,
                                         bool bf16, float k_scale, float v_scale, int *err_flag,
                                         cudaStream_t stream) {
    const int64_t row8 = row_elems / 8;
    const int threads = 128;
    const int64_t slices = (row8 + threads - 1) / threads;
    const int64_t cap = (static_cast<int64_t>(sm_count()) * 32 + slices - 1) / slices;
    const int64_t gx = num_tokens < cap ? num_tokens : cap;
    dim3 grid(static_cast<unsigned>(gx), static_cast<unsigned>(slices < 65535 ? slices : 65535));
    auto kern = bf16 ? reshape_and_cache_fp8_kernel<true> : reshape_and_cache_fp8_kernel<false>;
    kern<<<grid, threads, 0, stream>>>(static_cast<const uint4 *>(key), static_cast<const uint4 *>(value),
                                       static_cast<uint2 *>(k_cache), static_cast<uint2 *>(v_cache),
                                       slot_mapping, num_tokens, num_slots, row8, k_scale, v_scale,
                                       err_flag);
    return cudaGetLastError();
}

cudaError_t launch_copy_blocks(const void *src_k, const void *src_v, void *dst_k, void *dst_v,
                               const int64_t *block_mapping, int64_t num_pairs, int64_t src_blocks,
                               int64_t dst_blocks, int64_t block_bytes, int *err_flag,
                               cudaStream_t stream, int layers, int64_t layer_bytes) {
    const int64_t block16 = block_bytes / 16;
    const int threads = 256;
    const int sms = sm_count();
    if (layers < 1 || layers > 65535) return cudaErrorInvalidValue;
    // Enough CTAs to cover the SMs a few times over, each slice >= 4 chunks/thread.
    int64_t slices = (block16 + 4 * threads - 1) / (4 * threads);
    const int64_t want = 4LL * sms;
    const int64_t units = num_pairs * layers;
    if (units * slices < want) {
        const int64_t more = (want + units - 1) / units;
        const int64_t maxs = (block16 + threads - 1) / threads;
        slices = more < maxs ? more : maxs;
    }
    if (slices < 1) slices = 1;
    if (slices > 65535) slices = 65535;
    const int64_t gx = num_pairs < 65535LL * 16 ? num_pairs : 65535LL * 16;
    dim3 grid(static_cast<unsigned>(gx), static_cast<unsigned>(slices), static_cast<unsigned>(layers));
    copy_blocks_kernel<<<grid, threads, 0, stream>>>(
        static_cast<const uint4 *>(src_k), static_cast<const uint4 *>(src_v), static_cast<uint4 *>(dst_k),
        static_cast<uint4 *>(dst_v), block_mapping, num_pairs, src_blocks, dst_blocks, block16, layer_bytes / 16,
        err_flag);
    return cudaGetLastError();
}

}  // namespace pa
