// Paged decode attention for sm_103a (GB300).
//
// What it computes: for each sequence s and query head h (KV head h / G),
// softmax(q K^T * scale) V over the sequence's first context_lens[s] cached
// tokens, whose K/V rows live in fixed-size physical blocks reached through
// the sequence's block table ("LLM推理优化：vLLM PagedAttention深度解析与工程
// 实践", §二 formula, §3.1 block table, §4.1 paged layout; nano-vllm
// walkthrough lqnn.cn/news/170268, §2.3 steps 1-2).  Long contexts are cut into
// partitions whose partial softmax states are merged in partition order (the
// "partial accumulate, then merge" v2 kernel of the same page, §4.1).
//
// How (GB300 design, not the pages' A100 kernels):
//  * Persistent grid, one CTA per SM, every warp an independent pipeline.
//    Work items are (sequence, partition, KV head); the item list is split
//    into contiguous ranges of equal token weight, one per warp, so a
//    long-tailed length mix cannot leave SMs idle at the end.
//  * Each warp owns a ring of kStages shared-memory slots.  A slot holds one
//    16-token stage: the K and V rows of one KV head, brought in by TMA
//    (3-D tensor map over [blocks*block_size, Hkv, D], 64-element boxes with
//    128-byte swizzle) straight from the physical block the table names,
//    plus the item's query rows (bulk copy) on its first stage.  Loads for
//    the next stages - across item boundaries - are in flight while the warp
//    computes on the current one.
//  * QK: lane (t, half) dots token t's half row with the fp32 query held in
//    shared memory (broadcast reads; the swizzle makes the 16 row reads
//    conflict-free); one shuffle joins the halves.  Online softmax in base 2
//    with fp32 state (nano-vllm §6: fp32 accumulation).  PV: each lane owns
//    D/32 output dims and walks the stage's tokens.
//  * Positions at or beyond the context length are masked by select, never
//    multiplied, so NaN in stale slots cannot leak (nano-vllm §6).
//  * Partial states of split sequences go to a caller-owned workspace; the
//    last warp to finish a (sequence, KV head) - found with an atomic ticket
//    - merges them in partition order and resets the ticket.  No warp ever
//    waits on another.
#include "pa_device.cuh"
#include "pa_internal.h"

namespace pa {

namespace {

constexpr uint32_t kFull = 0xffffffffu;
constexpr int kRowBytes = 128;                        // one swizzled 64-element half row
constexpr int kRegionBytes = kStageTokens * kRowBytes;  // 16 rows x 128 B = 2 KB

template <int D, int G>
struct Layout {
    static constexpr int kHalves = D / 64;                 // swizzled regions per K (or V) tile
    static constexpr int kTileBytes = kHalves * kRegionBytes;
    static constexpr int kVOffset = kTileBytes;
    static constexpr int kQOffset = 2 * kTileBytes;
    static constexpr int kQBytes = G * D * 2;
    static constexpr int kSlotBytes = ((2 * kTileBytes + kQBytes + 1023) / 1024) * 1024;
    static constexpr int kQStride = D + 8;                 // floats per fp32 query row
    static constexpr int kQ32Bytes = G * kQStride * 4;
    static constexpr int kChunksPerLane = D / 16;          // 16-byte K chunks per lane in QK
    static constexpr int kDimsPerLane = D / 32;            // output dims per lane in PV
};

struct StageMeta {
    int s, kvh, part, j;
    int nst, nparts, mask, pad;
};

constexpr int kMetaBytes = sizeof(StageMeta);

// Work weight of a sequence, in 16-token stages summed over its KV heads.
// A sequence with no valid tokens still costs one stage per KV head (it
// writes a zero row).
__device__ __forceinline__ uint32_t seq_weight(int ctx, int hkv) {
    int st = ctx > 0 ? (ctx + kStageTokens - 1) / kStageTokens : 1;
    return static_cast<uint32_t>(st) * static_cast<uint32_t>(hkv);
}

// Cursor over the ordered work items (s, part, kvh) of one warp.
struct Cursor {
    int s, part, kvh;
    int ctx, nparts, ntok, nst;
    uint32_t start;  // global stage index of the item's first stage

    __device__ __forceinline__ void set_seq(int s_, const int *ctx_s, int P) {
        s = s_;
        ctx = ctx_s[s_];
        nparts = ctx > 0 ? (ctx + P - 1) / P : 1;
    }
    __device__ __forceinline__ void set_part(int part_, int P) {
        part = part_;
        ntok = ctx > 0 ? min(P, ctx - part_ * P) : 0;
        nst = ntok > 0 ? (ntok + kStageTokens - 1) / kStageTokens : 1;
    }
    __device__ __forceinline__ void advance(const int *ctx_s, const uint32_t *prefix, int hkv,
                                            int P, int B) {
        start += nst;
        if (++kvh < hkv) return;
        kvh = 0;
        if (part + 1 < nparts) {
            set_part(part + 1, P);
            return;
        }
        if (s + 1 < B) {
            set_seq(s + 1, ctx_s, P);
            set_part(0, P);
            start = prefix[s];
        }
    }
};

// 128-dim heads run at most 8 warps per CTA (the slot ring fills shared
// memory), so they get 255 registers per thread; 64-dim heads run up to 16.
template <int D>
constexpr int kMaxThreads = D == 128 ? 256 : 512;

template <int D, int G, bool BF16>
__global__ void __launch_bounds__(kMaxThreads<D>, 1)
    paged_decode_kernel(const __grid_constant__ DecodeParams p,
                        const __grid_constant__ CUtensorMap tmap_k,
                        const __grid_constant__ CUtensorMap tmap_v) {
    using L = Layout<D, G>;
    using Cvt = Half2x<BF16>;
    extern __shared__ uint8_t smem_raw[];
    uint8_t *smem = reinterpret_cast<uint8_t *>(
        (reinterpret_cast<uintptr_t>(smem_raw) + 1023) & ~static_cast<uintptr_t>(1023));

    const int lane = threadIdx.x & 31;
    const int warp = threadIdx.x >> 5;
    const int nw = blockDim.x >> 5;
    const int B = p.num_seqs;
    const int Hkv = p.num_kv_heads;
    const int P = p.partition_size;

    uint8_t *slots = smem + static_cast<size_t>(warp) * kStages * L::kSlotBytes;
    uint8_t *misc = smem + static_cast<size_t>(nw) * kStages * L::kSlotBytes;
    float *q32 = reinterpret_cast<float *>(misc + warp * L::kQ32Bytes);
    misc += nw * L::kQ32Bytes;
    StageMeta *meta = reinterpret_cast<StageMeta *>(misc) + warp * kStages;
    misc += nw * kStages * kMetaBytes;
    uint64_t *bars = reinterpret_cast<uint64_t *>(misc) + warp * kStages;
    misc += nw * kStages * 8;
    uint32_t *warp_tot = reinterpret_cast<uint32_t *>(misc);
    misc += 32 * 4;
    int *ctx_s = reinterpret_cast<int *>(misc);
    uint32_t *prefix = reinterpret_cast<uint32_t *>(misc + 4 * B);

    // ---- CTA prologue: validated context lengths and the work prefix ----
    for (int i = threadIdx.x; i < B; i += blockDim.x) {
        int c = p.context_lens[i];
        if (c < 0 || c > p.max_context_len) {
            if (blockIdx.x == 0) report(p.err_flag, 0x4 /* PA_FLAG_BAD_CONTEXT_LEN */);
            c = 0;
        }
        ctx_s[i] = c;
    }
    if (lane == 0) {
        for (int i = 0; i < kStages; ++i) mbar_init(&bars[i], 1);
        fence_barrier_init();
    }
    if (threadIdx.x == 0) {
        prefetch_tensormap(&tmap_k);
        prefetch_tensormap(&tmap_v);
    }
    __syncthreads();
    {
        const int nthr = blockDim.x;
        const int per = (B + nthr - 1) / nthr;
        const int beg = min(B, threadIdx.x * per);
        const int end = min(B, beg + per);
        uint32_t local = 0;
        for (int i = beg; i < end; ++i) local += seq_weight(ctx_s[i], Hkv);
        uint32_t incl = local;
#pragma unroll
        for (int o = 1; o < 32; o <<= 1) {
            uint32_t v = __shfl_up_sync(kFull, incl, o);
            if (lane >= o) incl += v;
        }
        if (lane == 31) warp_tot[warp] = incl;
        __syncthreads();
        uint32_t base = 0;
        for (int w = 0; w < warp; ++w) base += warp_tot[w];
        uint32_t run = base + incl - local;
        for (int i = beg; i < end; ++i) {
            prefix[i] = run;
            run += seq_weight(ctx_s[i], Hkv);
        }
        if (threadIdx.x == 0) {
            uint32_t tot = 0;
            for (int w = 0; w < nw; ++w) tot += warp_tot[w];
            prefix[B] = tot;
        }
        __syncthreads();
    }

    // ---- this warp's range of work [lo, hi) in stage units ----
    const uint32_t total = prefix[B];
    const uint64_t nwarps = static_cast<uint64_t>(gridDim.x) * nw;
    const uint64_t gw = static_cast<uint64_t>(blockIdx.x) * nw + warp;
    const uint32_t lo = static_cast<uint32_t>(static_cast<uint64_t>(total) * gw / nwarps);
    const uint32_t hi = static_cast<uint32_t>(static_cast<uint64_t>(total) * (gw + 1) / nwarps);
    if (lo >= hi) return;

    // First item whose first stage is >= lo.
    Cursor ic;
    {
        int a = 0, b = B;  // largest s with prefix[s] <= lo
        while (b - a > 1) {
            int m = (a + b) >> 1;
            if (prefix[m] <= lo) a = m; else b = m;
        }
        ic.set_seq(a, ctx_s, P);
        const uint32_t off = lo - prefix[a];
        const uint32_t P16 = static_cast<uint32_t>(P / kStageTokens);
        int part = static_cast<int>(off / (static_cast<uint32_t>(Hkv) * P16));
        if (part > ic.nparts - 1) part = ic.nparts - 1;
        ic.set_part(part, P);
        const uint32_t pstart = prefix[a] + static_cast<uint32_t>(part) * Hkv * P16;
        const uint32_t rem = off - (pstart - prefix[a]);
        int kvh = static_cast<int>((rem + ic.nst - 1) / ic.nst);
        ic.kvh = kvh;
        ic.start = pstart + static_cast<uint32_t>(kvh) * ic.nst;
        if (kvh >= Hkv) {  // step to the next partition or sequence
            ic.kvh = Hkv - 1;
            ic.start = pstart + static_cast<uint32_t>(Hkv - 1) * ic.nst;
            ic.advance(ctx_s, prefix, Hkv, P, B);
        }
    }
    if (ic.start >= hi) return;

    const uint64_t policy = l2_policy_evict_first();
    const int bs = p.block_size;
    const int Hq = p.num_heads;

    // ---- issuer state ----
    int ij = 0;                  // stage within the issuer's current item
    int32_t bid = -1;            // lane i: block id i of the issuer's item
    int fb = 0;                  // first logical block of the issuer's item
    bool more = true;
    uint32_t issued = 0;

    auto issue = [&]() {
        const int slot = static_cast<int>(issued % kStages);
        uint8_t *sp = slots + slot * L::kSlotBytes;
        if (ij == 0 && ic.ntok > 0) {
            fb = (ic.part * P) / bs;
            const int lb = (ic.part * P + ic.ntok - 1) / bs;
            bid = (lane <= lb - fb)
                      ? p.block_tables[static_cast<int64_t>(ic.s) * p.max_blocks_per_seq + fb + lane]
                      : -1;
        }
        const int tok0 = ic.part * P + ij * kStageTokens;
        const int n = ic.ntok > 0 ? min(kStageTokens, ic.ntok - ij * kStageTokens) : 0;
        int mask = n > 0 ? static_cast<int>((1u << n) - 1u) : 0;
        // Physical blocks of this stage: one when block_size >= 16, two when 8.
        const int nsub = bs >= kStageTokens ? 1 : kStageTokens / bs;
        int ids[2] = {-1, -1};
        uint32_t bytes = 0;
#pragma unroll
        for (int b = 0; b < 2; ++b) {
            if (b < nsub) {
                const int first = tok0 + b * bs;
                const bool used = n > b * bs;
                const int idx = used ? first / bs - fb : 0;
                const int id = __shfl_sync(kFull, bid, idx & 31);
                if (used) {
                    if (id < 0 || static_cast<int64_t>(id) >= p.num_blocks) {
                        const int rows = min(bs, kStageTokens);
                        mask &= ~(((1 << rows) - 1) << (b * bs));
                        if (lane == 0) report(p.err_flag, 0x2 /* PA_FLAG_BAD_BLOCK_ID */);
                    } else {
                        ids[b] = id;
                        bytes += 2u * L::kHalves * min(bs, kStageTokens) * kRowBytes;
                    }
                }
            }
        }
        const bool with_q = (ij == 0 && ic.ntok > 0);
        if (with_q) bytes += L::kQBytes;
        if (lane == 0) {
            StageMeta m;
            m.s = ic.s; m.kvh = ic.kvh; m.part = ic.part; m.j = ij;
            m.nst = ic.nst; m.nparts = ic.nparts; m.mask = mask; m.pad = 0;
            meta[slot] = m;
            mbar_arrive_expect_tx(&bars[slot], bytes);
            const int rows = min(bs, kStageTokens);
#pragma unroll
            for (int b = 0; b < 2; ++b) {
                if (ids[b] >= 0) {
                    const int z = ids[b] * bs + ((tok0 + b * bs) % bs);
#pragma unroll
                    for (int h = 0; h < L::kHalves; ++h) {
                        tma_load_3d(sp + h * kRegionBytes + b * rows * kRowBytes, &tmap_k,
                                    &bars[slot], h * 64, ic.kvh, z, policy);
                        tma_load_3d(sp + L::kVOffset + h * kRegionBytes + b * rows * kRowBytes,
                                    &tmap_v, &bars[slot], h * 64, ic.kvh, z, policy);
                    }
                }
            }
            if (with_q) {
                const uint16_t *qsrc = static_cast<const uint16_t *>(p.q) +
                                       (static_cast<int64_t>(ic.s) * Hq + ic.kvh * G) * D;
                bulk_load(sp + L::kQOffset, qsrc, L::kQBytes, &bars[slot]);
            }
        }
        ++issued;
        if (++ij == ic.nst) {
            ij = 0;
            ic.advance(ctx_s, prefix, Hkv, P, B);
            more = ic.start < hi;
        }
    };

    // ---- consumer state ----
    const int t = lane & 15;      // QK: token of this lane
    const int hh = lane >> 4;     // QK: which half of the dims
    float m_run[G], l_lane[G], acc[G][L::kDimsPerLane];

    for (int k = 0; k < kStages && more; ++k) issue();

    uint32_t consumed = 0;
    while (consumed < issued) {
        const int slot = static_cast<int>(consumed % kStages);
        const uint8_t *sp = slots + slot * L::kSlotBytes;
        if (!mbar_wait_bounded(&bars[slot], (consumed / kStages) & 1u)) {
            if (lane == 0) report(p.err_flag, 0x10 /* PA_FLAG_TIMEOUT */);
            return;
        }
        const StageMeta m = meta[slot];

        if (m.j == 0) {
            // New item: widen the query to fp32, pre-scaled into the log2 domain.
            const uint16_t *qh = reinterpret_cast<const uint16_t *>(sp + L::kQOffset);
#pragma unroll
            for (int k = 0; k < G * D / 64; ++k) {
                const int e = 2 * (lane + 32 * k);  // element pair (e, e+1)
                const int g = e / D, d = e % D;
                const float2 f = Cvt::to_float2(*reinterpret_cast<const uint32_t *>(qh + e));
                float *dst = q32 + g * L::kQStride + d + (d >= 64 ? 4 : 0);
                dst[0] = f.x * p.scale_log2;
                dst[1] = f.y * p.scale_log2;
            }
#pragma unroll
            for (int g = 0; g < G; ++g) {
                m_run[g] = -INFINITY;
                l_lane[g] = 0.f;
#pragma unroll
                for (int i = 0; i < L::kDimsPerLane; ++i) acc[g][i] = 0.f;
            }
            __syncwarp();
        }

        // ---- QK^T for the stage's 16 tokens ----
        float x[G];
#pragma unroll
        for (int g = 0; g < G; ++g) x[g] = 0.f;
#pragma unroll
        for (int i = 0; i < L::kChunksPerLane; ++i) {
            const int c = hh * L::kChunksPerLane + i;
            const int hr = c >> 3, cc = c & 7;
            const uint4 kw = *reinterpret_cast<const uint4 *>(sp + hr * kRegionBytes + t * kRowBytes +
                                                              ((cc ^ (t & 7)) << 4));
            const float2 k0 = Cvt::to_float2(kw.x), k1 = Cvt::to_float2(kw.y);
            const float2 k2 = Cvt::to_float2(kw.z), k3 = Cvt::to_float2(kw.w);
#pragma unroll
            for (int g = 0; g < G; ++g) {
                const float *qp = q32 + g * L::kQStride + c * 8 + (hr ? 4 : 0);
                const float4 qa = *reinterpret_cast<const float4 *>(qp);
                const float4 qb = *reinterpret_cast<const float4 *>(qp + 4);
                float a = x[g];
                a = fmaf(qa.x, k0.x, a); a = fmaf(qa.y, k0.y, a);
                a = fmaf(qa.z, k1.x, a); a = fmaf(qa.w, k1.y, a);
                a = fmaf(qb.x, k2.x, a); a = fmaf(qb.y, k2.y, a);
                a = fmaf(qb.z, k3.x, a); a = fmaf(qb.w, k3.y, a);
                x[g] = a;
            }
        }
        const bool valid = (m.mask >> t) & 1;
        float pr[G];
#pragma unroll
        for (int g = 0; g < G; ++g) {
            if (L::kHalves * 8 > L::kChunksPerLane) x[g] += __shfl_xor_sync(kFull, x[g], 16);
            const float xv = valid ? x[g] : -INFINITY;
            float mt = xv;
#pragma unroll
            for (int o = 1; o < 16; o <<= 1) mt = fmaxf(mt, __shfl_xor_sync(kFull, mt, o));
            const float m_new = fmaxf(m_run[g], mt);
            const float m_use = (m_new == -INFINITY) ? 0.f : m_new;
            const float alpha = fast_exp2(m_run[g] - m_use);
            pr[g] = fast_exp2(xv - m_use);
            l_lane[g] = l_lane[g] * alpha + pr[g];
#pragma unroll
            for (int i = 0; i < L::kDimsPerLane; ++i) acc[g][i] *= alpha;
            m_run[g] = m_new;
        }

        // ---- PV: lane owns kDimsPerLane consecutive output dims ----
        const uint8_t *vt = sp + L::kVOffset;
#pragma unroll
        for (int tt = 0; tt < kStageTokens; ++tt) {
            if (!((m.mask >> tt) & 1)) continue;
            float pt[G];
#pragma unroll
            for (int g = 0; g < G; ++g) pt[g] = __shfl_sync(kFull, pr[g], tt);
            if constexpr (D == 128) {
                const int hr = lane >> 4, cc = (lane & 15) >> 1, sub = (lane & 1) * 8;
                const uint2 vw = *reinterpret_cast<const uint2 *>(
                    vt + hr * kRegionBytes + tt * kRowBytes + ((cc ^ (tt & 7)) << 4) + sub);
                const float2 v0 = Cvt::to_float2(vw.x), v1 = Cvt::to_float2(vw.y);
#pragma unroll
                for (int g = 0; g < G; ++g) {
                    acc[g][0] = fmaf(pt[g], v0.x, acc[g][0]);
                    acc[g][1] = fmaf(pt[g], v0.y, acc[g][1]);
                    acc[g][2] = fmaf(pt[g], v1.x, acc[g][2]);
                    acc[g][3] = fmaf(pt[g], v1.y, acc[g][3]);
                }
            } else {
                const int cc = lane >> 2, sub = (lane & 3) * 4;
                const uint32_t vw = *reinterpret_cast<const uint32_t *>(
                    vt + tt * kRowBytes + ((cc ^ (tt & 7)) << 4) + sub);
                const float2 v0 = Cvt::to_float2(vw);
#pragma unroll
                for (int g = 0; g < G; ++g) {
                    acc[g][0] = fmaf(pt[g], v0.x, acc[g][0]);
                    acc[g][1] = fmaf(pt[g], v0.y, acc[g][1]);
                }
            }
        }

        // ---- item end: write the output or the partial state ----
        if (m.j == m.nst - 1) {
            float l_tot[G];
#pragma unroll
            for (int g = 0; g < G; ++g) {
                float v = l_lane[g];
#pragma unroll
                for (int o = 1; o < 16; o <<= 1) v += __shfl_xor_sync(kFull, v, o);
                l_tot[g] = v;
            }
            const int d0 = lane * L::kDimsPerLane;
            const int64_t orow0 = static_cast<int64_t>(m.s) * Hq + m.kvh * G;
            auto store_out = [&](int g, const float *o) {
                const int64_t off = (orow0 + g) * D + d0;
                if (p.out_dtype == 2) {
                    float *dst = static_cast<float *>(p.out) + off;
                    if constexpr (L::kDimsPerLane == 4)
                        *reinterpret_cast<float4 *>(dst) = make_float4(o[0], o[1], o[2], o[3]);
                    else
                        *reinterpret_cast<float2 *>(dst) = make_float2(o[0], o[1]);
                } else {
                    uint16_t h[L::kDimsPerLane];
#pragma unroll
                    for (int i = 0; i < L::kDimsPerLane; ++i)
                        h[i] = p.out_dtype == 1 ? float_to_bf16_bits(o[i]) : float_to_f16_bits(o[i]);
                    uint16_t *dst = static_cast<uint16_t *>(p.out) + off;
                    if constexpr (L::kDimsPerLane == 4)
                        *reinterpret_cast<uint2 *>(dst) =
                            make_uint2(h[0] | (uint32_t(h[1]) << 16), h[2] | (uint32_t(h[3]) << 16));
                    else
                        *reinterpret_cast<uint32_t *>(dst) = h[0] | (uint32_t(h[1]) << 16);
                }
            };
            if (m.nparts == 1) {
#pragma unroll
                for (int g = 0; g < G; ++g) {
                    const float inv = l_tot[g] > 0.f ? 1.f / l_tot[g] : 0.f;
                    float o[L::kDimsPerLane];
#pragma unroll
                    for (int i = 0; i < L::kDimsPerLane; ++i) o[i] = acc[g][i] * inv;
                    store_out(g, o);
                }
            } else {
                const int64_t pair = static_cast<int64_t>(m.s) * Hkv + m.kvh;
                const int64_t base = pair * p.max_partitions;
#pragma unroll
                for (int g = 0; g < G; ++g) {
                    float *a = p.ws_acc + ((base + m.part) * G + g) * D + d0;
                    if constexpr (L::kDimsPerLane == 4)
                        *reinterpret_cast<float4 *>(a) =
                            make_float4(acc[g][0], acc[g][1], acc[g][2], acc[g][3]);
                    else
                        *reinterpret_cast<float2 *>(a) = make_float2(acc[g][0], acc[g][1]);
                    if (lane == 0)
                        *reinterpret_cast<float2 *>(p.ws_ml + ((base + m.part) * G + g) * 2) =
                            make_float2(m_run[g], l_tot[g]);
                }
                __threadfence();
                __syncwarp();
                uint32_t ticket = 0;
                if (lane == 0) ticket = atomicAdd(p.counters + pair, 1u);
                ticket = __shfl_sync(kFull, ticket, 0);
                if (ticket == static_cast<uint32_t>(m.nparts - 1)) {
                    // Last partition to finish: merge all of them in order.
                    if (lane == 0) p.counters[pair] = 0u;
                    __threadfence();
#pragma unroll
                    for (int g = 0; g < G; ++g) {
                        float M = -INFINITY;
                        for (int j = 0; j < m.nparts; ++j) {
                            const float2 ml = __ldcg(reinterpret_cast<const float2 *>(
                                p.ws_ml + ((base + j) * G + g) * 2));
                            M = fmaxf(M, ml.x);
                        }
                        float Lsum = 0.f, o[L::kDimsPerLane];
#pragma unroll
                        for (int i = 0; i < L::kDimsPerLane; ++i) o[i] = 0.f;
                        for (int j = 0; j < m.nparts; ++j) {
                            const float2 ml = __ldcg(reinterpret_cast<const float2 *>(
                                p.ws_ml + ((base + j) * G + g) * 2));
                            const float w = (ml.x == -INFINITY) ? 0.f : fast_exp2(ml.x - M);
                            Lsum = fmaf(ml.y, w, Lsum);
                            const float *a = p.ws_acc + ((base + j) * G + g) * D + d0;
                            if constexpr (L::kDimsPerLane == 4) {
                                const float4 v = __ldcg(reinterpret_cast<const float4 *>(a));
                                o[0] = fmaf(v.x, w, o[0]); o[1] = fmaf(v.y, w, o[1]);
                                o[2] = fmaf(v.z, w, o[2]); o[3] = fmaf(v.w, w, o[3]);
                            } else {
                                const float2 v = __ldcg(reinterpret_cast<const float2 *>(a));
                                o[0] = fmaf(v.x, w, o[0]); o[1] = fmaf(v.y, w, o[1]);
                            }
                        }
                        const float inv = Lsum > 0.f ? 1.f / Lsum : 0.f;
#pragma unroll
                        for (int i = 0; i < L::kDimsPerLane; ++i) o[i] *= inv;
                        store_out(g, o);
                    }
                }
            }
        }

        ++consumed;
        if (more) {
            fence_proxy_async_smem();
            __syncwarp();
            issue();
        } else {
            __syncwarp();
        }
    }
}

template <int D, int G>
size_t smem_for(int warps, int num_seqs) {
    using L = Layout<D, G>;
    size_t per_warp = static_cast<size_t>(kStages) * L::kSlotBytes + L::kQ32Bytes +
                      kStages * kMetaBytes + kStages * 8;
    return 1024 + per_warp * warps + 32 * 4 + 4 * static_cast<size_t>(num_seqs) +
           4 * (static_cast<size_t>(num_seqs) + 1);
}

template <int D, int G, bool BF16>
cudaError_t launch_t(const DecodeParams &p, const CUtensorMap &tk, const CUtensorMap &tv,
                     int grid, int warps, size_t smem, cudaStream_t stream) {
    auto kern = paged_decode_kernel<D, G, BF16>;
    cudaError_t e = cudaFuncSetAttribute(kern, cudaFuncAttributeMaxDynamicSharedMemorySize,
                                         static_cast<int>(smem));
    if (e != cudaSuccess) return e;
    kern<<<grid, warps * 32, smem, stream>>>(p, tk, tv);
    return cudaGetLastError();
}

template <int D, int G>
cudaError_t launch_dt(const DecodeParams &p, bool bf16, const CUtensorMap &tk,
                      const CUtensorMap &tv, int grid, int warps, size_t smem,
                      cudaStream_t stream) {
    return bf16 ? launch_t<D, G, true>(p, tk, tv, grid, warps, smem, stream)
                : launch_t<D, G, false>(p, tk, tv, grid, warps, smem, stream);
}

template <int D>
cudaError_t launch_g(const DecodeParams &p, int group, bool bf16, const CUtensorMap &tk,
                     const CUtensorMap &tv, int grid, int warps, size_t smem,
                     cudaStream_t stream) {
    switch (group) {
        case 1: return launch_dt<D, 1>(p, bf16, tk, tv, grid, warps, smem, stream);
        case 2: return launch_dt<D, 2>(p, bf16, tk, tv, grid, warps, smem, stream);
        case 4: return launch_dt<D, 4>(p, bf16, tk, tv, grid, warps, smem, stream);
        case 8: return launch_dt<D, 8>(p, bf16, tk, tv, grid, warps, smem, stream);
        default: return cudaErrorInvalidValue;
    }
}

template <int D>
size_t smem_g(int group, int warps, int num_seqs) {
    switch (group) {
        case 1: return smem_for<D, 1>(warps, num_seqs);
        case 2: return smem_for<D, 2>(warps, num_seqs);
        case 4: return smem_for<D, 4>(warps, num_seqs);
        case 8: return smem_for<D, 8>(warps, num_seqs);
        default: return 0;
    }
}

}  // namespace

size_t decode_smem_bytes(int head_dim, int group, int warps, int num_seqs) {
    return head_dim == 64 ? smem_g<64>(group, warps, num_seqs)
                          : smem_g<128>(group, warps, num_seqs);
}

cudaError_t launch_decode(const DecodeParams &p, int head_dim, int group, bool bf16,
                          const CUtensorMap &tk, const CUtensorMap &tv, int grid, int warps,
                          size_t smem, cudaStream_t stream) {
    if (head_dim == 64) return launch_g<64>(p, group, bf16, tk, tv, grid, warps, smem, stream);
    if (head_dim == 128) return launch_g<128>(p, group, bf16, tk, tv, grid, warps, smem, stream);
    return cudaErrorInvalidValue;
}

}  // namespace pa
