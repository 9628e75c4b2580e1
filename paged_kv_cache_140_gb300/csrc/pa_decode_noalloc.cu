// pa_decode_noalloc: paged decode attention for callers that cannot allocate
// device memory.
//
// pa_decode needs a caller-provided workspace for the partial results of
// split sequences.  Some callers cannot obtain one while they run: code that
// executes inside a host framework owning all device memory (an inference
// engine's plugin that must not allocate during its execute step), or a
// deployment whose device-memory budget is fixed when the library loads.
// This entry point gives them decode without any allocation: the workspace is
// a fixed-size array that lives in the library itself.
//
// The array is a file-scope static __device__ variable, so every GPU that
// loads this library holds PA_NOALLOC_SCRATCH_BYTES of device memory for it
// until the process exits.  Host code cannot use the array's name as a device
// address (on the host it names a stand-in object); the device address is
// looked up once per device with cudaGetSymbolAddress and passed to the
// kernel like any other workspace pointer.
#include <cuda_runtime.h>
#include <stdint.h>

#include <mutex>

#include "pa.h"

#define PA_EXPORT extern "C" __attribute__((visibility("default")))

namespace {

static __device__ __align__(256) unsigned char g_decode_scratch[PA_NOALLOC_SCRATCH_BYTES];

constexpr int kMaxDevices = 256;
std::mutex g_scratch_mutex;
void *g_scratch_ptr[kMaxDevices] = {};

// Device address of g_decode_scratch on the current device (looked up on the
// first call per device, with that device current).  nullptr on failure.
void *scratch_on_current_device() {
    int dev = 0;
    if (cudaGetDevice(&dev) != cudaSuccess || dev < 0 || dev >= kMaxDevices) return nullptr;
    std::lock_guard<std::mutex> lock(g_scratch_mutex);
    if (g_scratch_ptr[dev] == nullptr) {
        void *p = nullptr;
        if (cudaGetSymbolAddress(&p, g_decode_scratch) != cudaSuccess) return nullptr;
        g_scratch_ptr[dev] = p;
    }
    return g_scratch_ptr[dev];
}

}  // namespace

PA_EXPORT pa_status pa_decode_noalloc(void *out, pa_dtype out_dtype, const void *query,
                                      pa_dtype q_dtype, const void *k_cache, const void *v_cache,
                                      pa_dtype kv_dtype, float k_scale, float v_scale,
                                      const int32_t *block_tables, int max_blocks_per_seq,
                                      const int32_t *context_lens, int max_context_len,
                                      int num_seqs, int num_heads, int num_kv_heads, int head_dim,
                                      int block_size, int64_t num_blocks, float scale,
                                      int partition_size, int *err_flag, void *stream) {
    const size_t need = pa_decode_workspace_size(num_seqs, num_heads, num_kv_heads, head_dim,
                                                 block_size, max_context_len, partition_size);
    if (need == static_cast<size_t>(-1) || need == 0) {
        // Rejected arguments, or nothing to split: pa_decode needs no
        // workspace (and reports the exact argument error).
        return pa_decode(out, out_dtype, query, q_dtype, k_cache, v_cache, kv_dtype, k_scale, v_scale, block_tables,
                         max_blocks_per_seq, context_lens, max_context_len, num_seqs, num_heads,
                         num_kv_heads, head_dim, block_size, num_blocks, scale, partition_size,
                         nullptr, 0, err_flag, stream);
    }
    if (need > static_cast<size_t>(PA_NOALLOC_SCRATCH_BYTES)) return PA_ERR_WORKSPACE;
    if (num_seqs == 0) return PA_OK;
    void *scratch = scratch_on_current_device();
    if (scratch == nullptr) return PA_ERR_CUDA;
    // The array keeps the previous call's contents; nothing in the decode
    // workspace needs an initial value (every partial state is written before
    // the merge kernel reads it), so no clearing is needed.
    return pa_decode(out, out_dtype, query, q_dtype, k_cache, v_cache, kv_dtype, k_scale, v_scale, block_tables,
                     max_blocks_per_seq, context_lens, max_context_len, num_seqs, num_heads,
                     num_kv_heads, head_dim, block_size, num_blocks, scale, partition_size, scratch,
                     static_cast<size_t>(PA_NOALLOC_SCRATCH_BYTES), err_flag, stream);
}
