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
// looked up with cudaGetSymbolAddress, with the device current, and passed to
// the kernel like any other workspace pointer.  The address belongs to the CUDA
// context that loaded the module, so it is cached per context (by the
// context's unique id, which is never reused within a process): the first call
// in each context - normally once per device, again after a device reset or
// under another context - looks it up.
#include <cuda.h>
#include <cuda_runtime.h>
#include <stdint.h>

#include <mutex>

#include "pa.h"

#define PA_EXPORT extern "C" __attribute__((visibility("default")))

namespace {

static __device__ __align__(256) unsigned char g_decode_scratch[PA_NOALLOC_SCRATCH_BYTES];

using CtxGetCurrentFn = CUresult (*)(CUcontext *);
using CtxGetIdFn = CUresult (*)(CUcontext, unsigned long long *);

struct DriverFns {
    CtxGetCurrentFn get_current = nullptr;
    CtxGetIdFn get_id = nullptr;
};

const DriverFns &driver_fns() {
    static DriverFns fns;
    static std::once_flag once;
    std::call_once(once, [] {
        void *p = nullptr;
        cudaDriverEntryPointQueryResult q;
        if (cudaGetDriverEntryPointByVersion("cuCtxGetCurrent", &p, 12000, cudaEnableDefault, &q) ==
                cudaSuccess && q == cudaDriverEntryPointSuccess)
            fns.get_current = reinterpret_cast<CtxGetCurrentFn>(p);
        p = nullptr;
        if (cudaGetDriverEntryPointByVersion("cuCtxGetId", &p, 12000, cudaEnableDefault, &q) ==
                cudaSuccess && q == cudaDriverEntryPointSuccess)
            fns.get_id = reinterpret_cast<CtxGetIdFn>(p);
    });
    return fns;
}

// Unique id of the current context; false if there is none (yet) or the
// driver cannot say.
bool current_context_id(unsigned long long *id) {
    const DriverFns &d = driver_fns();
    if (d.get_current == nullptr || d.get_id == nullptr) return false;
    CUcontext ctx = nullptr;
    if (d.get_current(&ctx) != CUDA_SUCCESS || ctx == nullptr) return false;
    return d.get_id(ctx, id) == CUDA_SUCCESS;
}

constexpr int kCacheEntries = 64;
struct ScratchEntry {
    unsigned long long ctx_id;
    void *ptr;
};
std::mutex g_scratch_mutex;
ScratchEntry g_scratch[kCacheEntries] = {};
int g_scratch_next = 0;

// Device address of g_decode_scratch in the current context: looked up with
// cudaGetSymbolAddress on the first call in each context, cached after that.
// nullptr on failure.
void *scratch_in_current_context() {
    unsigned long long id = 0;
    const bool have_id = current_context_id(&id);
    if (have_id) {
        std::lock_guard<std::mutex> lock(g_scratch_mutex);
        for (const ScratchEntry &e : g_scratch)
            if (e.ptr != nullptr && e.ctx_id == id) return e.ptr;
    }
    // The lookup also makes the runtime's context current on this thread if
    // no runtime call has done so yet.
    void *p = nullptr;
    if (cudaGetSymbolAddress(&p, g_decode_scratch) != cudaSuccess) return nullptr;
    if (have_id || current_context_id(&id)) {
        std::lock_guard<std::mutex> lock(g_scratch_mutex);
        g_scratch[g_scratch_next] = ScratchEntry{id, p};
        g_scratch_next = (g_scratch_next + 1) % kCacheEntries;
    }
    return p;
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
    if (need == static_cast<size_t>(-1) || need == 0 || need > static_cast<size_t>(PA_NOALLOC_SCRATCH_BYTES)) {
        // Rejected arguments, nothing to split (no workspace needed), or more
        // than the array holds: pa_decode without a workspace checks every
        // argument first and then answers PA_ERR_WORKSPACE (enqueuing nothing)
        // where one would be needed.
        return pa_decode(out, out_dtype, query, q_dtype, k_cache, v_cache, kv_dtype, k_scale, v_scale, block_tables,
                         max_blocks_per_seq, context_lens, max_context_len, num_seqs, num_heads,
                         num_kv_heads, head_dim, block_size, num_blocks, scale, partition_size,
                         nullptr, 0, err_flag, stream);
    }
    void *scratch = scratch_in_current_context();
    if (scratch == nullptr) return PA_ERR_CUDA;
    // The array keeps the previous call's contents; nothing in the decode
    // workspace needs an initial value (every partial state is written before
    // the merge kernel reads it), so no clearing is needed.
    return pa_decode(out, out_dtype, query, q_dtype, k_cache, v_cache, kv_dtype, k_scale, v_scale, block_tables,
                     max_blocks_per_seq, context_lens, max_context_len, num_seqs, num_heads,
                     num_kv_heads, head_dim, block_size, num_blocks, scale, partition_size, scratch,
                     static_cast<size_t>(PA_NOALLOC_SCRATCH_BYTES), err_flag, stream);
}
