// Helpers shared by the two paged decode kernels (pa_decode.cu: per-warp
// pipelines; pa_decode_coop.cu: CTA-cooperative): the work weight of a
// sequence, a warp-wide float maximum, the output-row store and the launch
// with programmatic dependent launch.
#pragma once

#include "pa_device.cuh"
#include "pa_internal.h"

namespace pa {
namespace decode_common {

constexpr uint32_t kFull = 0xffffffffu;

// Work weight of a sequence, in 16-token stages summed over its KV heads.
// A sequence with no valid tokens still costs one stage per KV head (it
// writes a zero row).
__device__ __forceinline__ uint32_t seq_weight(int ctx, int hkv) {
    int st = ctx > 0 ? (ctx + kStageTokens - 1) / kStageTokens : 1;
    return static_cast<uint32_t>(st) * static_cast<uint32_t>(hkv);
}

// Maximum over the warp of a float, via an order-preserving integer image.
__device__ __forceinline__ float warp_max(float x) {
    int k = __float_as_int(x);
    k = k >= 0 ? k : k ^ 0x7fffffff;
    k = __reduce_max_sync(kFull, k);
    return __int_as_float(k >= 0 ? k : k ^ 0x7fffffff);
}

// Store D/32 consecutive floats of a row (this lane's slice) as f32, bf16 or
// f16 (pa_dtype codes 2, 1, 0), rounding to nearest even.
template <int D>
__device__ __forceinline__ void store_row(void *base, int dtype, int64_t off, const float *o) {
    constexpr int DPL = D / 32;
    if (dtype == 2) {
        float *dst = static_cast<float *>(base) + off;
        if constexpr (DPL == 4)
            *reinterpret_cast<float4 *>(dst) = make_float4(o[0], o[1], o[2], o[3]);
        else
            *reinterpret_cast<float2 *>(dst) = make_float2(o[0], o[1]);
    } else {
        uint16_t h[DPL];
#pragma unroll
        for (int i = 0; i < DPL; ++i) h[i] = dtype == 1 ? float_to_bf16_bits(o[i]) : float_to_f16_bits(o[i]);
        uint16_t *dst = static_cast<uint16_t *>(base) + off;
        if constexpr (DPL == 4)
            *reinterpret_cast<uint2 *>(dst) =
                make_uint2(h[0] | (uint32_t(h[1]) << 16), h[2] | (uint32_t(h[3]) << 16));
        else
            *reinterpret_cast<uint32_t *>(dst) = h[0] | (uint32_t(h[1]) << 16);
    }
}

// Launch `kern` with programmatic stream serialization: it may start while
// the previous kernel in the stream finishes, and waits (griddepcontrol.wait)
// before reading anything that kernel wrote.
template <typename Kern, typename... Args>
cudaError_t launch_pdl(Kern kern, dim3 grid, dim3 block, size_t smem, cudaStream_t stream,
                       Args... args) {
    cudaLaunchConfig_t cfg = {};
    cfg.gridDim = grid;
    cfg.blockDim = block;
    cfg.dynamicSmemBytes = smem;
    cfg.stream = stream;
    cudaLaunchAttribute attr[1];
    attr[0].id = cudaLaunchAttributeProgrammaticStreamSerialization;
    attr[0].val.programmaticStreamSerializationAllowed = 1;
    cfg.attrs = attr;
    cfg.numAttrs = 1;
    return cudaLaunchKernelEx(&cfg, kern, args...);
}

}  // namespace decode_common
}  // namespace pa
