// The exported C ABI (declared in include/pa.h): argument validation,
// partition and workspace planning, TMA descriptor encoding and launches.
// The library allocates no memory and keeps no state between calls beyond
// cached device attributes (per device ordinal) and the driver entry point.
#include <cuda.h>
#include <cuda_runtime.h>
#include <stdint.h>

#include <stdlib.h>

#include <algorithm>
#include <atomic>
#include <mutex>

#include "pa.h"
#include "pa_cache_ops.h"
#include "pa_internal.h"
#include "pa_prefill.h"

#define PA_EXPORT extern "C" __attribute__((visibility("default")))

namespace {

using EncodeTiledFn = CUresult (*)(CUtensorMap *, CUtensorMapDataType, cuuint32_t, void *,
                                   const cuuint64_t *, const cuuint64_t *, const cuuint32_t *,
                                   const cuuint32_t *, CUtensorMapInterleave, CUtensorMapSwizzle,
                                   CUtensorMapL2promotion, CUtensorMapFloatOOBfill);

EncodeTiledFn encode_tiled() {
    static EncodeTiledFn fn = nullptr;
    static std::once_flag once;
    std::call_once(once, [] {
        void *p = nullptr;
        cudaDriverEntryPointQueryResult q;
        if (cudaGetDriverEntryPointByVersion("cuTensorMapEncodeTiled", &p, 12000,
                                             cudaEnableDefault, &q) == cudaSuccess &&
            q == cudaDriverEntryPointSuccess)
            fn = reinterpret_cast<EncodeTiledFn>(p);
    });
    return fn;
}

bool aligned16(const void *p) { return (reinterpret_cast<uintptr_t>(p) & 15u) == 0; }
bool half_dtype(pa_dtype d) { return d == PA_F16 || d == PA_BF16; }
bool cache_dtype_ok(pa_dtype d) { return half_dtype(d) || d == PA_FP8_E4M3; }
int elem_bytes(pa_dtype d) { return d == PA_FP8_E4M3 ? 1 : 2; }
bool scale_ok(float s) { return s > 0.f && s < 3.0e38f; }
bool supported_head_dim(int d) { return d == 64 || d == 128; }
bool supported_block_size(int bs) { return bs == 8 || (bs >= 16 && bs <= 256 && bs % 16 == 0); }
bool supported_group(int g) { return g == 1 || g == 2 || g == 4 || g == 8; }

int64_t round_up(int64_t x, int64_t m) { return (x + m - 1) / m * m; }

struct DeviceInfo {
    int sms = 0;
    int smem_optin = 0;
};

// Attributes of the current device, read once per device ordinal (they are
// properties of the hardware and do not change while the process runs).
constexpr int kMaxDevices = 64;

bool device_info(DeviceInfo &info) {
    static DeviceInfo cache[kMaxDevices];
    static std::atomic<bool> valid[kMaxDevices];
    static std::mutex mu;
    int dev = 0;
    if (cudaGetDevice(&dev) != cudaSuccess) return false;
    if (dev >= 0 && dev < kMaxDevices && valid[dev].load(std::memory_order_acquire)) {
        info = cache[dev];
        return true;
    }
    DeviceInfo d;
    if (cudaDeviceGetAttribute(&d.sms, cudaDevAttrMultiProcessorCount, dev) != cudaSuccess)
        return false;
    if (cudaDeviceGetAttribute(&d.smem_optin, cudaDevAttrMaxSharedMemoryPerBlockOptin, dev) !=
        cudaSuccess)
        return false;
    if (dev >= 0 && dev < kMaxDevices) {
        std::lock_guard<std::mutex> lock(mu);
        cache[dev] = d;
        valid[dev].store(true, std::memory_order_release);
    }
    info = d;
    return true;
}

// Tuning overrides read once from the environment (documented in pa.h):
// PA_DECODE_COOP=0 keeps every shape on the per-warp decode kernel;
// PA_DECODE_COOP_STAGES, PA_DECODE_STAGES and PA_DECODE_WARPS set ring depths
// and warps per CTA; PA_DECODE_INTERLEAVE=0 gives each per-warp pipeline a
// contiguous run of items.  Results stay within the documented tolerance under
// any setting; only speed changes.
struct Tuning {
    int stages = 0;  // 0: default
    int warps = 0;
    int interleave = 1;
    int coop = 1;            // 0: never use the CTA-cooperative decode kernel
    int coop_stages = 0;     // 0: default
};

int env_int(const char *name, int lo, int hi) {
    const char *v = getenv(name);
    if (v == nullptr) return 0;
    const int x = atoi(v);
    return (x >= lo && x <= hi) ? x : 0;
}

const Tuning &tuning() {
    static const Tuning t = [] {
        Tuning r;
        r.stages = env_int("PA_DECODE_STAGES", 2, 8);
        r.warps = env_int("PA_DECODE_WARPS", 1, 16);
        const char *il = getenv("PA_DECODE_INTERLEAVE");
        r.interleave = (il != nullptr && il[0] == '0') ? 0 : 1;
        const char *co = getenv("PA_DECODE_COOP");
        r.coop = (co != nullptr && co[0] == '0') ? 0 : 1;
        r.coop_stages = env_int("PA_DECODE_COOP_STAGES", 2, 8);
        return r;
    }();
    return t;
}

// Partition length in tokens for pa_decode; 0 when the request is invalid.
int resolve_partition(int max_context_len, int block_size, int requested) {
    const int cap = 32 * block_size;
    if (requested != 0) {
        if (requested < 16 || requested % 16 != 0 || requested > cap) return 0;
        return requested;
    }
    int P;
    if (max_context_len <= 256)
        P = static_cast<int>(std::max<int64_t>(16, round_up(max_context_len, 16)));
    else if (max_context_len <= 8192)
        P = 256;
    else
        P = 512;
    return std::min(P, cap);
}

struct WorkspacePlan {
    int partition = 0;
    int max_partitions = 1;
    size_t ml_off = 0, acc_off = 0, bytes = 0;
};

bool plan_workspace(int num_seqs, int num_heads, int num_kv_heads, int head_dim, int block_size,
                    int max_context_len, int partition_size, WorkspacePlan &w) {
    if (num_seqs < 0 || num_kv_heads <= 0 || num_heads <= 0 || num_heads % num_kv_heads != 0)
        return false;
    if (!supported_group(num_heads / num_kv_heads) || !supported_head_dim(head_dim) ||
        !supported_block_size(block_size) || max_context_len < 0)
        return false;
    w.partition = resolve_partition(max_context_len, block_size, partition_size);
    if (w.partition == 0) return false;
    w.max_partitions = std::max(1, (max_context_len + w.partition - 1) / w.partition);
    if (w.max_partitions <= 1) {
        w.bytes = 0;
        return true;
    }
    const int G = num_heads / num_kv_heads;
    const int64_t slots = static_cast<int64_t>(num_seqs) * num_kv_heads * w.max_partitions;
    w.ml_off = 0;
    w.acc_off = round_up(slots * G * 2 * 4, 256);
    w.bytes = w.acc_off + static_cast<size_t>(slots) * G * head_dim * 4;
    return true;
}

// Tensor map over a cache [NB * bs, Hkv, D] with 128-byte boxes of one KV
// head's row and min(bs, 16) rows, 128-byte swizzle.
bool encode_cache_map(CUtensorMap *map, const void *cache, int64_t num_blocks, int block_size,
                      int num_kv_heads, int head_dim, int es) {
    EncodeTiledFn fn = encode_tiled();
    if (fn == nullptr) return false;
    const cuuint64_t dims[3] = {static_cast<cuuint64_t>(head_dim),
                                static_cast<cuuint64_t>(num_kv_heads),
                                static_cast<cuuint64_t>(num_blocks) * block_size};
    const cuuint64_t strides[2] = {static_cast<cuuint64_t>(head_dim) * es,
                                   static_cast<cuuint64_t>(num_kv_heads) * head_dim * es};
    const cuuint32_t box[3] = {static_cast<cuuint32_t>(128 / es), 1u,
                               static_cast<cuuint32_t>(std::min(block_size, 16))};
    const cuuint32_t estr[3] = {1u, 1u, 1u};
    return fn(map, es == 1 ? CU_TENSOR_MAP_DATA_TYPE_UINT8 : CU_TENSOR_MAP_DATA_TYPE_UINT16, 3,
              const_cast<void *>(cache), dims, strides,
              box, estr, CU_TENSOR_MAP_INTERLEAVE_NONE, CU_TENSOR_MAP_SWIZZLE_128B,
              CU_TENSOR_MAP_L2_PROMOTION_L2_256B,
              CU_TENSOR_MAP_FLOAT_OOB_FILL_NONE) == CUDA_SUCCESS;
}

// Tensor map over a cache [NB * bs, Hkv, D] of `es`-byte elements with its
// dimensions taken in the order (dim, token, head): a box {128 / es, 16, 8}
// is one 128-byte column block of 16 token rows for 8 consecutive KV heads,
// landing as 8 per-head tiles of 16 rows x 128 bytes, 128-byte swizzle (the
// cooperative decode kernel).
bool encode_cache_map_heads8(CUtensorMap *map, const void *cache, int64_t num_blocks, int block_size,
                             int num_kv_heads, int head_dim, int es) {
    EncodeTiledFn fn = encode_tiled();
    if (fn == nullptr) return false;
    const cuuint64_t dims[3] = {static_cast<cuuint64_t>(head_dim),
                                static_cast<cuuint64_t>(num_blocks) * block_size,
                                static_cast<cuuint64_t>(num_kv_heads)};
    const cuuint64_t strides[2] = {static_cast<cuuint64_t>(num_kv_heads) * head_dim * es,
                                   static_cast<cuuint64_t>(head_dim) * es};
    const cuuint32_t box[3] = {static_cast<cuuint32_t>(128 / es), 16u, 8u};
    const cuuint32_t estr[3] = {1u, 1u, 1u};
    return fn(map, es == 1 ? CU_TENSOR_MAP_DATA_TYPE_UINT8 : CU_TENSOR_MAP_DATA_TYPE_UINT16, 3,
              const_cast<void *>(cache), dims, strides, box, estr,
              CU_TENSOR_MAP_INTERLEAVE_NONE, CU_TENSOR_MAP_SWIZZLE_128B, CU_TENSOR_MAP_L2_PROMOTION_L2_256B,
              CU_TENSOR_MAP_FLOAT_OOB_FILL_NONE) == CUDA_SUCCESS;
}

// The address a kernel on the current device may use for `p`: device or
// managed memory as is, page-locked host memory through its mapped device
// pointer.  False for anything else (e.g. pageable host memory), which the
// caller rejects before any launch.
bool device_address(const void *p, const void **out) {
    cudaPointerAttributes a;
    if (cudaPointerGetAttributes(&a, p) != cudaSuccess) {
        cudaGetLastError();
        return false;
    }
    if (a.type == cudaMemoryTypeDevice || a.type == cudaMemoryTypeManaged) {
        *out = p;
        return true;
    }
    if (a.type == cudaMemoryTypeHost && a.devicePointer != nullptr) {
        *out = a.devicePointer;
        return true;
    }
    return false;
}

}  // namespace

PA_EXPORT const char *pa_status_string(pa_status s) {
    switch (s) {
        case PA_OK: return "ok";
        case PA_ERR_INVALID_ARG: return "invalid argument";
        case PA_ERR_UNSUPPORTED: return "unsupported shape or dtype";
        case PA_ERR_CUDA: return "CUDA error";
        case PA_ERR_WORKSPACE: return "decode workspace missing or too small";
        case PA_ERR_DEVICE_BOUNDS: return "device-side index out of bounds (see err_flag bits)";
    }
    return "unknown status";
}

PA_EXPORT int pa_version(void) { return 100; }

PA_EXPORT pa_status pa_reshape_and_cache(const void *key, const void *value, void *k_cache,
                                         void *v_cache, const int64_t *slot_mapping,
                                         int64_t num_tokens, int64_t num_blocks, int block_size,
                                         int num_kv_heads, int head_dim, pa_dtype dtype,
                                         pa_dtype cache_dtype, float k_scale, float v_scale,
                                         int *err_flag, void *stream) {
    if (num_tokens < 0 || num_blocks <= 0 || block_size <= 0 || num_kv_heads <= 0 ||
        head_dim <= 0 || !half_dtype(dtype) || !cache_dtype_ok(cache_dtype))
        return PA_ERR_INVALID_ARG;
    const bool fp8 = cache_dtype == PA_FP8_E4M3;
    if (!fp8 && cache_dtype != dtype) return PA_ERR_UNSUPPORTED;
    if (fp8 && (!scale_ok(k_scale) || !scale_ok(v_scale))) return PA_ERR_INVALID_ARG;
    const int64_t row_elems = static_cast<int64_t>(num_kv_heads) * head_dim;
    if ((row_elems * 2) % 16 != 0 || row_elems % 8 != 0) return PA_ERR_UNSUPPORTED;
    if (num_tokens == 0) return PA_OK;
    if (!key || !value || !k_cache || !v_cache || !slot_mapping) return PA_ERR_INVALID_ARG;
    if (!aligned16(key) || !aligned16(value) || !aligned16(k_cache) || !aligned16(v_cache))
        return PA_ERR_INVALID_ARG;
    cudaError_t e;
    if (fp8)
        e = pa::launch_reshape_and_cache_fp8(key, value, k_cache, v_cache, slot_mapping, num_tokens,
                                             num_blocks * block_size, row_elems, dtype == PA_BF16,
                                             k_scale, v_scale, err_flag,
                                             static_cast<cudaStream_t>(stream));
    else
        e = pa::launch_reshape_and_cache(key, value, k_cache, v_cache, slot_mapping, num_tokens,
                                         num_blocks * block_size, row_elems * 2, err_flag,
                                         static_cast<cudaStream_t>(stream));
    return e == cudaSuccess ? PA_OK : PA_ERR_CUDA;
}

PA_EXPORT pa_status pa_copy_blocks(void *k_cache, void *v_cache, const int64_t *block_mapping,
                                   int64_t num_pairs, int64_t num_blocks, int block_size,
                                   int num_kv_heads, int head_dim, pa_dtype dtype, int *err_flag,
                                   void *stream) {
    if (num_pairs < 0 || num_blocks <= 0 || block_size <= 0 || num_kv_heads <= 0 ||
        head_dim <= 0 || !cache_dtype_ok(dtype))
        return PA_ERR_INVALID_ARG;
    const int64_t block_bytes =
        static_cast<int64_t>(block_size) * num_kv_heads * head_dim * elem_bytes(dtype);
    if (block_bytes % 16 != 0) return PA_ERR_UNSUPPORTED;
    if (num_pairs == 0) return PA_OK;
    if (!k_cache || !v_cache || !block_mapping) return PA_ERR_INVALID_ARG;
    if (!aligned16(k_cache) || !aligned16(v_cache)) return PA_ERR_INVALID_ARG;
    cudaError_t e = pa::launch_copy_blocks(k_cache, v_cache, k_cache, v_cache, block_mapping, num_pairs,
                                           num_blocks, num_blocks, block_bytes, err_flag,
                                           static_cast<cudaStream_t>(stream));
    return e == cudaSuccess ? PA_OK : PA_ERR_CUDA;
}

PA_EXPORT pa_status pa_copy_blocks_layers(void *kv_cache, int num_layers, const int64_t *block_mapping,
                                          int64_t num_pairs, int64_t num_blocks, int block_size,
                                          int num_kv_heads, int head_dim, pa_dtype dtype, int *err_flag,
                                          void *stream) {
    if (num_layers < 0 || num_pairs < 0 || num_blocks <= 0 || block_size <= 0 || num_kv_heads <= 0 ||
        head_dim <= 0 || !cache_dtype_ok(dtype))
        return PA_ERR_INVALID_ARG;
    if (num_layers > 65535) return PA_ERR_UNSUPPORTED;
    const int64_t block_bytes =
        static_cast<int64_t>(block_size) * num_kv_heads * head_dim * elem_bytes(dtype);
    if (block_bytes % 16 != 0) return PA_ERR_UNSUPPORTED;
    if (num_pairs == 0 || num_layers == 0) return PA_OK;
    if (!kv_cache || !block_mapping || !aligned16(kv_cache)) return PA_ERR_INVALID_ARG;
    // [layers, 2, num_blocks, ...]: layer l's K at l * 2 * NB blocks, its V right after.
    uint8_t *base = static_cast<uint8_t *>(kv_cache);
    const int64_t cache_bytes = num_blocks * block_bytes;
    cudaError_t e = pa::launch_copy_blocks(base, base + cache_bytes, base, base + cache_bytes, block_mapping,
                                           num_pairs, num_blocks, num_blocks, block_bytes, err_flag,
                                           static_cast<cudaStream_t>(stream), num_layers, 2 * cache_bytes);
    return e == cudaSuccess ? PA_OK : PA_ERR_CUDA;
}

PA_EXPORT pa_status pa_swap_blocks(const void *src_k, const void *src_v, void *dst_k, void *dst_v,
                                   const int64_t *block_mapping, int64_t num_pairs,
                                   int64_t src_num_blocks, int64_t dst_num_blocks, int block_size,
                                   int num_kv_heads, int head_dim, pa_dtype dtype, int *err_flag,
                                   void *stream) {
    if (num_pairs < 0 || src_num_blocks <= 0 || dst_num_blocks <= 0 || block_size <= 0 ||
        num_kv_heads <= 0 || head_dim <= 0 || !cache_dtype_ok(dtype))
        return PA_ERR_INVALID_ARG;
    const int64_t block_bytes =
        static_cast<int64_t>(block_size) * num_kv_heads * head_dim * elem_bytes(dtype);
    if (block_bytes % 16 != 0) return PA_ERR_UNSUPPORTED;
    if (num_pairs == 0) return PA_OK;
    if (!src_k || !src_v || !dst_k || !dst_v || !block_mapping) return PA_ERR_INVALID_ARG;
    if (!aligned16(src_k) || !aligned16(src_v) || !aligned16(dst_k) || !aligned16(dst_v))
        return PA_ERR_INVALID_ARG;
    const void *sk, *sv, *dk, *dv, *bm;
    if (!device_address(src_k, &sk) || !device_address(src_v, &sv) || !device_address(dst_k, &dk) ||
        !device_address(dst_v, &dv) || !device_address(block_mapping, &bm))
        return PA_ERR_INVALID_ARG;
    cudaError_t e = pa::launch_copy_blocks(sk, sv, const_cast<void *>(dk), const_cast<void *>(dv),
                                           static_cast<const int64_t *>(bm), num_pairs, src_num_blocks,
                                           dst_num_blocks, block_bytes, err_flag,
                                           static_cast<cudaStream_t>(stream));
    return e == cudaSuccess ? PA_OK : PA_ERR_CUDA;
}

PA_EXPORT size_t pa_decode_workspace_size(int num_seqs, int num_heads, int num_kv_heads,
                                          int head_dim, int block_size, int max_context_len,
                                          int partition_size) {
    WorkspacePlan w;
    if (!plan_workspace(num_seqs, num_heads, num_kv_heads, head_dim, block_size, max_context_len,
                        partition_size, w))
        return static_cast<size_t>(-1);
    return w.bytes;
}

PA_EXPORT int pa_decode_partition_size(int num_seqs, int num_heads, int num_kv_heads,
                                       int head_dim, int block_size, int max_context_len,
                                       int partition_size) {
    WorkspacePlan w;
    if (!plan_workspace(num_seqs, num_heads, num_kv_heads, head_dim, block_size, max_context_len,
                        partition_size, w))
        return 0;
    return w.partition;
}

PA_EXPORT pa_status pa_decode_workspace_init(void *workspace, size_t workspace_bytes,
                                             void *stream) {
    if (workspace_bytes == 0) return PA_OK;
    if (workspace == nullptr) return PA_ERR_INVALID_ARG;
    return cudaMemsetAsync(workspace, 0, workspace_bytes, static_cast<cudaStream_t>(stream)) ==
                   cudaSuccess
               ? PA_OK
               : PA_ERR_CUDA;
}

namespace {

// pa_decode and pa_decode_append share everything but the new rows.
pa_status decode_impl(void *out, pa_dtype out_dtype, const void *query, pa_dtype q_dtype,
                      const void *new_k, const void *new_v,
                      const void *k_cache, const void *v_cache, pa_dtype kv_dtype,
                      float k_scale, float v_scale,
                              const int32_t *block_tables, int max_blocks_per_seq,
                              const int32_t *context_lens, int max_context_len, int num_seqs,
                              int num_heads, int num_kv_heads, int head_dim, int block_size,
                              int64_t num_blocks, float scale, int partition_size,
                              void *workspace, size_t workspace_bytes, int *err_flag,
                              void *stream) {
    if (num_seqs < 0 || num_heads <= 0 || num_kv_heads <= 0 || head_dim <= 0 ||
        block_size <= 0 || num_blocks <= 0 || max_blocks_per_seq <= 0 || max_context_len < 0)
        return PA_ERR_INVALID_ARG;
    if (!half_dtype(q_dtype) || !cache_dtype_ok(kv_dtype) ||
        (out_dtype != PA_F16 && out_dtype != PA_BF16 && out_dtype != PA_F32))
        return PA_ERR_INVALID_ARG;
    const bool fp8 = kv_dtype == PA_FP8_E4M3;
    if (fp8 && (!scale_ok(k_scale) || !scale_ok(v_scale))) return PA_ERR_INVALID_ARG;
    if (!fp8 && kv_dtype != q_dtype) return PA_ERR_UNSUPPORTED;     // 16-bit caches: same type as q
    if (fp8 && head_dim != 128) return PA_ERR_UNSUPPORTED;
    if (num_heads % num_kv_heads != 0) return PA_ERR_INVALID_ARG;
    if (!supported_group(num_heads / num_kv_heads) || !supported_head_dim(head_dim) ||
        !supported_block_size(block_size))
        return PA_ERR_UNSUPPORTED;
    if (static_cast<int64_t>(max_context_len) > static_cast<int64_t>(max_blocks_per_seq) * block_size)
        return PA_ERR_INVALID_ARG;
    if (num_blocks * block_size > INT32_MAX) return PA_ERR_UNSUPPORTED;
    if (!(scale == scale)) return PA_ERR_INVALID_ARG;
    WorkspacePlan w;
    if (!plan_workspace(num_seqs, num_heads, num_kv_heads, head_dim, block_size, max_context_len,
                        partition_size, w))
        return PA_ERR_INVALID_ARG;
    // Work is counted in 16-token stages in 32-bit arithmetic on the device.
    const int64_t max_units = static_cast<int64_t>(num_seqs) * num_kv_heads *
                              std::max<int64_t>(1, (max_context_len + 15) / 16);
    if (max_units >= (int64_t{1} << 31)) return PA_ERR_UNSUPPORTED;
    if (num_seqs == 0) return PA_OK;
    if (!out || !query || !k_cache || !v_cache || !block_tables || !context_lens)
        return PA_ERR_INVALID_ARG;
    if ((new_k == nullptr) != (new_v == nullptr)) return PA_ERR_INVALID_ARG;
    if (new_k && (!aligned16(new_k) || !aligned16(new_v))) return PA_ERR_INVALID_ARG;
    if (!aligned16(out) || !aligned16(query) || !aligned16(k_cache) || !aligned16(v_cache))
        return PA_ERR_INVALID_ARG;
    if (w.bytes > 0 && (workspace == nullptr || workspace_bytes < w.bytes || !aligned16(workspace)))
        return PA_ERR_WORKSPACE;

    DeviceInfo dev;
    if (!device_info(dev)) return PA_ERR_CUDA;
    const int G = num_heads / num_kv_heads;
    // Ring depth and warps per CTA (PA_DECODE_STAGES / PA_DECODE_WARPS override
    // the defaults for tuning); fewer warps are used if shared memory is short.
    const Tuning &tune = tuning();
    const int stages = tune.stages > 0 ? tune.stages : pa::kDefaultStages;
    const int max_warps = head_dim == 128 ? 12 : 16;
    const int def_warps = head_dim == 128 ? (fp8 ? pa::kDefaultWarpsFp8 : pa::kDefaultWarps128) : 16;
    int warps = tune.warps > 0 ? std::min(tune.warps, max_warps) : def_warps;
    const int es = elem_bytes(kv_dtype);
    while (warps > 1 && pa::decode_smem_bytes(head_dim, G, es, warps, stages, num_seqs) >
                            static_cast<size_t>(dev.smem_optin))
        --warps;
    const size_t smem_used = pa::decode_smem_bytes(head_dim, G, es, warps, stages, num_seqs);
    if (smem_used > static_cast<size_t>(dev.smem_optin)) return PA_ERR_UNSUPPORTED;

    pa::DecodeParams p{};
    p.out = out;
    p.out_dtype = static_cast<int>(out_dtype);
    p.q = query;
    p.block_tables = block_tables;
    p.context_lens = context_lens;
    p.max_blocks_per_seq = max_blocks_per_seq;
    p.max_context_len = max_context_len;
    p.num_seqs = num_seqs;
    p.num_heads = num_heads;
    p.num_kv_heads = num_kv_heads;
    p.block_size = block_size;
    p.num_blocks = num_blocks;
    p.scale_log2 = scale * 1.4426950408889634f * (fp8 ? k_scale : 1.0f);
    p.v_scale = fp8 ? v_scale : 1.0f;
    p.partition_size = w.partition;
    p.max_partitions = w.max_partitions;
    uint8_t *ws = static_cast<uint8_t *>(workspace);
    p.ws_ml = w.bytes ? reinterpret_cast<float *>(ws + w.ml_off) : nullptr;
    p.ws_acc = w.bytes ? reinterpret_cast<float *>(ws + w.acc_off) : nullptr;
    p.err_flag = err_flag;
    p.stages = stages;
    p.new_k = new_k;
    p.new_v = new_v;
    p.k_cache_w = const_cast<void *>(k_cache);
    p.v_cache_w = const_cast<void *>(v_cache);
    p.k_scale_w = k_scale;
    p.v_scale_w = v_scale;
    p.interleave = tune.interleave;

    const int kv = fp8 ? (q_dtype == PA_F16 ? 2 : 3) : (kv_dtype == PA_BF16 ? 1 : 0);
    // Caches whose KV heads come in groups of 8 run the CTA-cooperative
    // kernel (8-head TMA boxes); everything else the per-warp kernel.  With
    // new rows to append, an append kernel writes them first (quantised for
    // an e4m3 cache) and the cooperative kernel, chained by programmatic
    // dependent launch, waits for it only before the stages that hold them.
    if (tune.coop && head_dim == 128 && num_kv_heads % 8 == 0 && block_size % 16 == 0) {
        // a slot holds one 16-token stage of a 16-bit cache or two of an e4m3
        // cache: 64 KB either way
        int cst = tune.coop_stages > 0 ? tune.coop_stages : 3;
        while (cst > 2 && pa::decode_coop_smem_bytes(G, es, cst, num_seqs) > static_cast<size_t>(dev.smem_optin))
            --cst;
        const size_t csmem = pa::decode_coop_smem_bytes(G, es, cst, num_seqs);
        CUtensorMap ck, cv;
        if (csmem > 0 && csmem <= static_cast<size_t>(dev.smem_optin) &&
            encode_cache_map_heads8(&ck, k_cache, num_blocks, block_size, num_kv_heads, head_dim, es) &&
            encode_cache_map_heads8(&cv, v_cache, num_blocks, block_size, num_kv_heads, head_dim, es)) {
            p.stages = cst;
            if (new_k != nullptr) {
                const int64_t row = static_cast<int64_t>(num_kv_heads) * head_dim;
                const cudaError_t ea =
                    fp8 ? pa::launch_append_rows_fp8(new_k, new_v, const_cast<void *>(k_cache),
                                                     const_cast<void *>(v_cache), block_tables, context_lens,
                                                     max_blocks_per_seq, max_context_len, block_size, num_blocks,
                                                     num_seqs, row, q_dtype == PA_BF16, k_scale, v_scale, err_flag,
                                                     static_cast<cudaStream_t>(stream))
                        : pa::launch_append_rows(new_k, new_v, const_cast<void *>(k_cache),
                                                 const_cast<void *>(v_cache), block_tables, context_lens,
                                                 max_blocks_per_seq, max_context_len, block_size, num_blocks,
                                                 num_seqs, row * 2, err_flag, static_cast<cudaStream_t>(stream));
                if (ea != cudaSuccess) return PA_ERR_CUDA;
                p.new_k = p.new_v = nullptr;
                p.defer_wait = 1;
            }
            const cudaError_t e = pa::launch_decode_coop(p, G, kv, ck, cv, dev.sms, csmem,
                                                         static_cast<cudaStream_t>(stream));
            return e == cudaSuccess ? PA_OK : PA_ERR_CUDA;
        }
    }
    CUtensorMap tk, tv;
    if (!encode_cache_map(&tk, k_cache, num_blocks, block_size, num_kv_heads, head_dim, es) ||
        !encode_cache_map(&tv, v_cache, num_blocks, block_size, num_kv_heads, head_dim, es))
        return PA_ERR_CUDA;
    cudaError_t e = pa::launch_decode(p, head_dim, G, kv, tk, tv, dev.sms, warps,
                                      smem_used, static_cast<cudaStream_t>(stream));
    return e == cudaSuccess ? PA_OK : PA_ERR_CUDA;
}

}  // namespace

PA_EXPORT pa_status pa_decode(void *out, pa_dtype out_dtype, const void *query, pa_dtype q_dtype,
                              const void *k_cache, const void *v_cache, pa_dtype kv_dtype,
                              float k_scale, float v_scale, const int32_t *block_tables,
                              int max_blocks_per_seq, const int32_t *context_lens,
                              int max_context_len, int num_seqs, int num_heads, int num_kv_heads,
                              int head_dim, int block_size, int64_t num_blocks, float scale,
                              int partition_size, void *workspace, size_t workspace_bytes,
                              int *err_flag, void *stream) {
    return decode_impl(out, out_dtype, query, q_dtype, nullptr, nullptr, k_cache, v_cache, kv_dtype,
                       k_scale, v_scale, block_tables, max_blocks_per_seq, context_lens,
                       max_context_len, num_seqs, num_heads, num_kv_heads, head_dim, block_size,
                       num_blocks, scale, partition_size, workspace, workspace_bytes, err_flag,
                       stream);
}

PA_EXPORT pa_status pa_decode_append(void *out, pa_dtype out_dtype, const void *query,
                                     pa_dtype q_dtype, const void *key, const void *value,
                                     void *k_cache, void *v_cache, pa_dtype kv_dtype, float k_scale,
                                     float v_scale, const int32_t *block_tables,
                                     int max_blocks_per_seq, const int32_t *context_lens,
                                     int max_context_len, int num_seqs, int num_heads,
                                     int num_kv_heads, int head_dim, int block_size,
                                     int64_t num_blocks, float scale, int partition_size,
                                     void *workspace, size_t workspace_bytes, int *err_flag,
                                     void *stream) {
    if (num_seqs > 0 && (key == nullptr || value == nullptr)) return PA_ERR_INVALID_ARG;
    return decode_impl(out, out_dtype, query, q_dtype, key, value, k_cache, v_cache, kv_dtype,
                       k_scale, v_scale, block_tables, max_blocks_per_seq, context_lens,
                       max_context_len, num_seqs, num_heads, num_kv_heads, head_dim, block_size,
                       num_blocks, scale, partition_size, workspace, workspace_bytes, err_flag,
                       stream);
}

namespace {

// Tensor map over a dense 3-D array [d2][d1][d0] of `es`-byte elements with
// a (128 / es, box1, box2) box (128 bytes wide) and 128-byte swizzle.
bool encode_map_128b(CUtensorMap *map, const void *ptr, int es, int64_t d0, int64_t d1, int64_t d2, int box1,
                     int box2) {
    EncodeTiledFn fn = encode_tiled();
    if (fn == nullptr) return false;
    const cuuint64_t dims[3] = {static_cast<cuuint64_t>(d0), static_cast<cuuint64_t>(d1),
                                static_cast<cuuint64_t>(d2)};
    const cuuint64_t strides[2] = {static_cast<cuuint64_t>(d0) * es, static_cast<cuuint64_t>(d0 * d1) * es};
    const cuuint32_t box[3] = {static_cast<cuuint32_t>(128 / es), static_cast<cuuint32_t>(box1),
                               static_cast<cuuint32_t>(box2)};
    const cuuint32_t estr[3] = {1u, 1u, 1u};
    return fn(map, es == 4 ? CU_TENSOR_MAP_DATA_TYPE_UINT32 : CU_TENSOR_MAP_DATA_TYPE_UINT16, 3,
              const_cast<void *>(ptr), dims, strides, box, estr, CU_TENSOR_MAP_INTERLEAVE_NONE,
              CU_TENSOR_MAP_SWIZZLE_128B, CU_TENSOR_MAP_L2_PROMOTION_L2_256B,
              CU_TENSOR_MAP_FLOAT_OOB_FILL_NONE) == CUDA_SUCCESS;
}

}  // namespace

PA_EXPORT pa_status pa_prefill(void *out, pa_dtype out_dtype, const void *query,
                               const void *k_cache, const void *v_cache, pa_dtype kv_dtype,
                               const int32_t *block_tables, int max_blocks_per_seq,
                               const int32_t *context_lens, const int32_t *cu_seqlens_q,
                               int num_seqs, int64_t num_tokens, int max_q_len, int num_heads,
                               int num_kv_heads, int head_dim, int block_size, int64_t num_blocks,
                               float scale, int *err_flag, void *stream) {
    if (num_seqs < 0 || num_tokens < 0 || max_q_len < 0 || num_heads <= 0 || num_kv_heads <= 0 ||
        head_dim <= 0 || block_size <= 0 || num_blocks <= 0 || max_blocks_per_seq <= 0)
        return PA_ERR_INVALID_ARG;
    if (!half_dtype(kv_dtype) || (out_dtype != PA_F16 && out_dtype != PA_BF16 && out_dtype != PA_F32))
        return PA_ERR_INVALID_ARG;
    if (num_heads % num_kv_heads != 0) return PA_ERR_INVALID_ARG;
    const int G = num_heads / num_kv_heads;
    if (G > pa::kPrefillTile || (G & (G - 1)) != 0) return PA_ERR_UNSUPPORTED;
    if (!supported_head_dim(head_dim)) return PA_ERR_UNSUPPORTED;
    if (block_size < 8 || block_size > pa::kPrefillTile || (block_size & (block_size - 1)) != 0)
        return PA_ERR_UNSUPPORTED;
    if (num_blocks * block_size > INT32_MAX || num_tokens > INT32_MAX) return PA_ERR_UNSUPPORTED;
    if (!(scale > 0.f) || scale > 3.0e38f) return PA_ERR_INVALID_ARG;
    int lg = 0;
    while ((1 << lg) < G) ++lg;
    const int tokens_per_tile = pa::kPrefillTile / G;
    const int64_t tiles = (static_cast<int64_t>(max_q_len) + tokens_per_tile - 1) / tokens_per_tile;
    const int64_t grid = static_cast<int64_t>(num_seqs) * num_kv_heads * ((tiles + 1) / 2);
    if (grid >= (int64_t{1} << 31)) return PA_ERR_UNSUPPORTED;
    if (grid == 0 || num_tokens == 0) return PA_OK;
    if (!out || !query || !k_cache || !v_cache || !block_tables || !context_lens || !cu_seqlens_q)
        return PA_ERR_INVALID_ARG;
    if (!aligned16(out) || !aligned16(query) || !aligned16(k_cache) || !aligned16(v_cache))
        return PA_ERR_INVALID_ARG;

    DeviceInfo dev;
    if (!device_info(dev)) return PA_ERR_CUDA;
    const size_t smem = pa::prefill_smem_bytes(head_dim);
    // + the kernel's static shared memory (barriers, the sequence order), under 8 KB
    if (smem + 8192 > static_cast<size_t>(dev.smem_optin)) return PA_ERR_UNSUPPORTED;

    CUtensorMap tq, tk, tv, to;
    const int out_es = out_dtype == PA_F32 ? 4 : 2;
    if (!encode_map_128b(&tq, query, 2, head_dim, num_heads, num_tokens, G, tokens_per_tile) ||
        !encode_map_128b(&tk, k_cache, 2, head_dim, num_kv_heads, num_blocks * block_size, 1, block_size) ||
        !encode_map_128b(&tv, v_cache, 2, head_dim, num_kv_heads, num_blocks * block_size, 1, block_size) ||
        !encode_map_128b(&to, out, out_es, head_dim, num_heads, num_tokens, G, tokens_per_tile))
        return PA_ERR_CUDA;

    pa::PrefillParams p{};
    p.q = query;
    p.out = out;
    p.out_dtype = static_cast<int>(out_dtype);
    p.block_tables = block_tables;
    p.context_lens = context_lens;
    p.cu_seqlens_q = cu_seqlens_q;
    p.max_blocks_per_seq = max_blocks_per_seq;
    p.num_seqs = num_seqs;
    p.num_tokens = num_tokens;
    p.num_heads = num_heads;
    p.num_kv_heads = num_kv_heads;
    p.log2_group = lg;
    p.block_size = block_size;
    p.num_blocks = num_blocks;
    p.max_q_len = max_q_len;
    p.tiles_per_seq = static_cast<int>(tiles);
    p.pairs_per_seq = static_cast<int>((tiles + 1) / 2);
    p.scale_log2 = scale * 1.4426950408889634f;
    p.err_flag = err_flag;
    cudaError_t e = pa::launch_prefill(p, head_dim, kv_dtype == PA_BF16, tq, tk, tv, to, smem,
                                       static_cast<cudaStream_t>(stream));
    return e == cudaSuccess ? PA_OK : PA_ERR_CUDA;
}

PA_EXPORT pa_status pa_check_err_flag(int *err_flag, int clear, int *flag_out, void *stream) {
    if (err_flag == nullptr) return PA_ERR_INVALID_ARG;
    cudaStream_t s = static_cast<cudaStream_t>(stream);
    int host = 0;
    if (cudaMemcpyAsync(&host, err_flag, sizeof(int), cudaMemcpyDeviceToHost, s) != cudaSuccess)
        return PA_ERR_CUDA;
    if (cudaStreamSynchronize(s) != cudaSuccess) return PA_ERR_CUDA;
    if (clear && cudaMemsetAsync(err_flag, 0, sizeof(int), s) != cudaSuccess) return PA_ERR_CUDA;
    if (flag_out) *flag_out = host;
    return host == 0 ? PA_OK : PA_ERR_DEVICE_BOUNDS;
}
