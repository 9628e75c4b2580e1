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
// This per-warp kernel serves head_dim 64, block size 8 and KV-head counts
// that are not a multiple of 8 (16-bit or e4m3 caches, with or without the
// fused append); caches with KV heads in groups of 8 run the CTA-cooperative
// kernel of pa_decode_coop.cu (8-head TMA boxes), which shares this file's
// merge kernel.
//
// How (GB300 design, not the pages' A100 kernels):
//  * Persistent grid, one CTA per SM, every warp an independent pipeline.
//    Work items are (sequence, partition, KV head); the item list is split
//    into contiguous ranges of equal token weight, one per warp, so a
//    long-tailed length mix cannot leave SMs idle at the end.
//  * Each warp owns a ring of shared-memory slots.  A slot holds one 16-token
//    stage (two for an e4m3 cache, 8 KB of K and V either way): the K and V
//    rows of one KV head, brought in by TMA (3-D tensor map over
//    [blocks*block_size, Hkv, D], 128-byte boxes with 128-byte swizzle)
//    straight from the physical block the table names, plus the item's query
//    rows (bulk copy) on its first stage.  The stages of a slot are processed
//    jointly: QK of each, one softmax update over all their tokens, PV of
//    each.  Loads for the next slots - across item boundaries - are in flight
//    while the warp computes on the current one; the block-table slice of the
//    next item is prefetched into registers.
//  * QK and PV run on warp-level tensor-core MMA (m16n8k16, fp32 accumulate):
//    the query heads of one KV group are the N = 8 columns (a dense tile for
//    G = 8, padded for smaller groups).  Decode is bound by reading K/V; the
//    MMA is there to keep each warp's instruction count per byte low enough
//    that 8 warps per SM keep HBM busy.  ldmatrix reads the swizzled tiles
//    conflict-free.  The softmax weights enter PV as a 16-bit high part plus
//    a 16-bit residual, keeping ~16 significant bits.
//  * Online softmax in base 2 with fp32 state (nano-vllm §6: fp32
//    accumulation) and lazy rescaling (the reference max only moves when a
//    logit exceeds it by more than 2^8).
//  * Positions at or beyond the context length are masked by select, and
//    their V rows are zeroed in shared memory before PV, so NaN in stale slots
//    cannot leak (nano-vllm §6).
//  * Split sequences write their partial states (max, sum, weighted V sum) to
//    a caller-owned workspace; a small merge kernel, chained with
//    programmatic dependent launch, combines them in partition order.  No
//    warp ever waits on another.
#include "pa_decode_common.cuh"
#include "pa_device.cuh"
#include "pa_internal.h"

namespace pa {

namespace {

using namespace decode_common;

constexpr int kRowBytes = 128;                          // one swizzled 64-element half row
constexpr int kRegionBytes = kStageTokens * kRowBytes;  // 16 rows x 128 B = 2 KB

// Slots of an e4m3 cache carry two consecutive 16-token stages (8 KB of K
// and V, like one 16-bit stage), so that the per-slot work (barrier wait,
// loads, bookkeeping) is paid once per 8 KB; 16-bit caches one stage.
template <int ES>
constexpr int kSub = ES == 1 ? 2 : 1;

// ES = bytes per cache element (2: f16/bf16, 1: e4m3).  A slot holds SUB
// stages: K of stage h at h * kHalfBytes, V of stage h at kVOffset + the same.
template <int D, int G, int ES, int SUB = kSub<ES>>
struct Layout {
    static constexpr int kBoxes = D * ES / 128;            // 128-byte TMA boxes per K (or V) row
    static constexpr int kBoxElems = 128 / ES;             // elements per box row
    static constexpr int kHalfBytes = kBoxes * kRegionBytes;   // one stage's K (or V) rows
    static constexpr int kTileBytes = SUB * kHalfBytes;
    static constexpr int kVOffset = kTileBytes;
    static constexpr int kQOffset = 2 * kTileBytes;
    static constexpr int kQBytes = G * D * 2;              // the query stays 16-bit
    static constexpr int kSlotBytes = ((2 * kTileBytes + kQBytes + 1023) / 1024) * 1024;
    static constexpr int kOStride = D + 4;                 // floats per staged output row
    static constexpr int kOBytes = G * kOStride * 4;       // per-warp output staging
    static constexpr int kSteps = D / 16;                  // MMA steps over the head dim
    static constexpr int kDimsPerLane = D / 32;            // output dims per lane in the store
};

struct StageMeta {
    int s, kvh, part, j;
    int nst, nparts, mask, pad;
};

constexpr int kMetaBytes = sizeof(StageMeta);

__device__ __forceinline__ float warp_sum(float x) {
#pragma unroll
    for (int o = 16; o > 0; o >>= 1) x += __shfl_xor_sync(kFull, x, o);
    return x;
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

// Block ids of one item's partition, one per lane (lane i: logical block
// first + i), or -1 past the item's last block.
__device__ __forceinline__ int32_t load_item_blocks(const DecodeParams &p, const Cursor &c,
                                                    int P, int lane) {
    if (c.ntok <= 0) return -1;
    const int fb = (c.part * P) / p.block_size;
    const int lb = (c.part * P + c.ntok - 1) / p.block_size;
    return lane <= lb - fb
               ? __ldg(p.block_tables + static_cast<int64_t>(c.s) * p.max_blocks_per_seq + fb + lane)
               : -1;
}

// 128-dim heads run at most 12 warps per CTA (the slot ring fills shared
// memory); 64-dim heads run up to 16.
template <int D, int KV>
constexpr int kMaxThreads = D == 128 ? 384 : 512;

// KV: 0 = f16 cache and query, 1 = bf16 cache and query, 2 / 3 = e4m3 cache
// with an f16 / bf16 query (run as f16 MMAs; e4m3 values are exact in f16,
// bf16 queries are rounded to f16).
template <int D, int G, int KV>
__global__ void __launch_bounds__((kMaxThreads<D, KV>), 1)
    paged_decode_kernel(const __grid_constant__ DecodeParams p,
                        const __grid_constant__ CUtensorMap tmap_k,
                        const __grid_constant__ CUtensorMap tmap_v) {
    constexpr bool kFp8 = KV >= 2;
    constexpr bool kQBf16 = KV == 1 || KV == 3;
    constexpr bool BF16 = KV == 1;     // MMA operand type
    static_assert(!kFp8 || D == 128, "the e4m3 cache path is built for head_dim 128");
    using L = Layout<D, G, kFp8 ? 1 : 2>;
    constexpr int SUB = kSub<kFp8 ? 1 : 2>;    // stages per slot
    using Cvt = Half2x<BF16>;
    constexpr int KS = L::kSteps;   // QK steps over the head dim
    constexpr int MT = L::kSteps;   // PV tiles over the head dim
    constexpr int DPL = L::kDimsPerLane;
    extern __shared__ uint8_t smem_raw[];
    uint8_t *smem = reinterpret_cast<uint8_t *>(
        (reinterpret_cast<uintptr_t>(smem_raw) + 1023) & ~static_cast<uintptr_t>(1023));

    const int lane = threadIdx.x & 31;
    const int warp = threadIdx.x >> 5;
    const int nw = blockDim.x >> 5;
    const int S = p.stages;
    const int B = p.num_seqs;
    const int Hkv = p.num_kv_heads;
    const int P = p.partition_size;

    uint8_t *slots = smem + static_cast<size_t>(warp) * S * L::kSlotBytes;
    uint8_t *misc = smem + static_cast<size_t>(nw) * S * L::kSlotBytes;
    float *obuf = reinterpret_cast<float *>(misc + warp * L::kOBytes);
    misc += nw * L::kOBytes;
    StageMeta *meta = reinterpret_cast<StageMeta *>(misc) + warp * S;
    misc += nw * S * kMetaBytes;
    uint64_t *bars = reinterpret_cast<uint64_t *>(misc) + warp * S;
    misc += nw * S * 8;
    uint32_t *warp_tot = reinterpret_cast<uint32_t *>(misc);
    misc += 32 * 4;
    int *ctx_s = reinterpret_cast<int *>(misc);
    uint32_t *prefix = reinterpret_cast<uint32_t *>(misc + 4 * B);

    // ---- CTA prologue: validated context lengths and the work prefix ----
    if (lane == 0) {
        for (int i = 0; i < S; ++i) mbar_init(&bars[i], 1);
        fence_barrier_init();
    }
    if (threadIdx.x == 0) {
        prefetch_tensormap(&tmap_k);
        prefetch_tensormap(&tmap_v);
    }
    // Launched with programmatic dependent launch: wait for the previous
    // kernel in the stream (e.g. reshape_and_cache writing this step's rows)
    // before reading any input.
    pdl_wait();
    for (int i = threadIdx.x; i < B; i += blockDim.x) {
        int c = p.context_lens[i];
        if (c < 0 || c > p.max_context_len) {
            if (blockIdx.x == 0) report(p.err_flag, 0x4 /* PA_FLAG_BAD_CONTEXT_LEN */);
            c = 0;
        }
        ctx_s[i] = c;
    }
    // The merge kernel (if launched) may start launching now; it waits for
    // this grid's completion before reading any partial state.
    pdl_launch_dependents();
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

    // ---- the range of work [lo, hi) in stage units ----
    // Interleaved (default): the CTA owns a contiguous range and its warps take
    // every nw-th item of it, so at any moment they read neighbouring KV heads
    // of the same token rows (DRAM locality).  Otherwise each warp owns a
    // contiguous range of its own.
    const uint32_t total = prefix[B];
    const bool inter = p.interleave != 0;
    const uint64_t nranges = inter ? gridDim.x : static_cast<uint64_t>(gridDim.x) * nw;
    const uint64_t rid = inter ? blockIdx.x : static_cast<uint64_t>(blockIdx.x) * nw + warp;
    const int step = inter ? nw : 1;
    const uint32_t lo = static_cast<uint32_t>(static_cast<uint64_t>(total) * rid / nranges);
    const uint32_t hi = static_cast<uint32_t>(static_cast<uint64_t>(total) * (rid + 1) / nranges);
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
    if (inter)
        for (int k = 0; k < warp; ++k) ic.advance(ctx_s, prefix, Hkv, P, B);
    if (ic.start >= hi) return;

    const uint64_t policy = l2_policy_evict_first();
    const uint64_t keep = l2_policy_evict_last();
    const int bs = p.block_size;
    const int Hq = p.num_heads;
    const int rows = min(bs, kStageTokens);          // rows per TMA box
    const int nsub = bs >= kStageTokens ? 1 : kStageTokens / bs;  // blocks per stage

    // ---- issuer state ----
    int ij = 0;                                       // stage within the issuer's item
    int32_t bid = load_item_blocks(p, ic, P, lane);   // block ids of the issuer's item
    int32_t bid_next = -1;                            // prefetched ids of the following item
    bool next_ready = false;
    int fb = 0;                                       // first logical block of the issuer's item
    bool more = true;
    int islot = 0;

    auto issue = [&]() {
        const int slot = islot;
        islot = (islot + 1 == S) ? 0 : islot + 1;
        uint8_t *sp = slots + slot * L::kSlotBytes;
        if (ij == 0) {
            if (next_ready) bid = bid_next;
            next_ready = false;
            fb = (ic.part * P) / bs;
            // Prefetch the next item's block ids; they are used one item later.
            Cursor nx = ic;
            for (int k = 0; k < step; ++k) nx.advance(ctx_s, prefix, Hkv, P, B);
            if (nx.start < hi) {
                bid_next = load_item_blocks(p, nx, P, lane);
                next_ready = true;
            }
        }
        int tok0[SUB], ids[SUB][2];
        uint32_t mask_all = 0, bytes = 0;
#pragma unroll
        for (int hs = 0; hs < SUB; ++hs) {
            const int js = ij + hs;   // stage of the item
            tok0[hs] = ic.part * P + js * kStageTokens;
            const int n = (ic.ntok > 0 && js < ic.nst) ? min(kStageTokens, ic.ntok - js * kStageTokens) : 0;
            int mask = n > 0 ? static_cast<int>((1u << n) - 1u) : 0;
#pragma unroll
            for (int b = 0; b < 2; ++b) {
                ids[hs][b] = -1;
                if (b < nsub) {
                    const bool used = n > b * bs;
                    const int idx = used ? (tok0[hs] + b * bs) / bs - fb : 0;
                    const int id = __shfl_sync(kFull, bid, idx & 31);
                    if (used) {
                        if (id < 0 || static_cast<int64_t>(id) >= p.num_blocks) {
                            mask &= ~(((1 << rows) - 1) << (b * bs));
                            if (lane == 0) report(p.err_flag, 0x2 /* PA_FLAG_BAD_BLOCK_ID */);
                        } else {
                            ids[hs][b] = id;
                            bytes += 2u * L::kBoxes * rows * kRowBytes;
                        }
                    }
                }
            }
            mask_all |= static_cast<uint32_t>(mask) << (kStageTokens * hs);
        }
        const bool with_q = (ij == 0 && ic.ntok > 0);
        if (with_q) bytes += L::kQBytes;
        if (lane == 0) {
            StageMeta m;
            m.s = ic.s; m.kvh = ic.kvh; m.part = ic.part; m.j = ij;
            m.nst = ic.nst; m.nparts = ic.nparts; m.mask = static_cast<int>(mask_all); m.pad = 0;
            meta[slot] = m;
            mbar_arrive_expect_tx(&bars[slot], bytes);
#pragma unroll
            for (int hs = 0; hs < SUB; ++hs) {
#pragma unroll
                for (int b = 0; b < 2; ++b) {
                    if (ids[hs][b] >= 0) {
                        const int z = ids[hs][b] * bs + ((tok0[hs] + b * bs) % bs);
                        uint8_t *kd = sp + hs * L::kHalfBytes + b * rows * kRowBytes;
#pragma unroll
                        for (int h = 0; h < L::kBoxes; ++h) {
                            tma_load_3d(kd + h * kRegionBytes, &tmap_k, &bars[slot], h * L::kBoxElems, ic.kvh, z,
                                        policy);
                            tma_load_3d(kd + L::kVOffset + h * kRegionBytes, &tmap_v, &bars[slot],
                                        h * L::kBoxElems, ic.kvh, z, policy);
                        }
                    }
                }
            }
            if (with_q) {
                const uint16_t *qsrc = static_cast<const uint16_t *>(p.q) +
                                       (static_cast<int64_t>(ic.s) * Hq + ic.kvh * G) * D;
                bulk_load(sp + L::kQOffset, qsrc, L::kQBytes, &bars[slot]);
            }
        }
        ij += SUB;
        if (ij >= ic.nst) {
            ij = 0;
            for (int k = 0; k < step; ++k) ic.advance(ctx_s, prefix, Hkv, P, B);
            more = ic.start < hi;
        }
    };

    // ---- consumer state (mma.sync fragments; g = lane / 4, t = lane % 4) ----
    // QK:  C[token][head] = K[token][:] . q[head][:]   (M = 16 tokens, N = 8 heads,
    //      K = 16 dims per step); lane holds tokens g, g+8 of heads 2t, 2t+1.
    // PV:  O^T[dim][head] += V^T[dim][token] p[token][head] (M = 16 dims per tile,
    //      N = 8 heads, K = 16 tokens); lane holds dims g, g+8 of heads 2t, 2t+1.
    // Heads >= G are padding: their query fragments are zero and their logits
    // are masked, so they never contribute.
    const int g = lane >> 2, t = lane & 3;
    const uint32_t sm_base = smem_addr(slots);
    uint32_t qf[KS][2];          // query B fragments for the item
    float acc[MT][4];            // O^T accumulators
    float m_run[2], l_run[2];    // running max (log2 domain) and sum, heads 2t, 2t+1
    // Fused append (p.new_k != nullptr): the item that holds a sequence's last
    // position (this step's token) patches that row into its shared-memory
    // tile and writes it to the cache.  nj: the stage holding it (-1: none).
    const bool append = p.new_k != nullptr;
    int nj = -1, nrow = 0, npos = 0;
    int32_t nid = -1;       // block id of the new token (loaded at item start, used later)
    uint2 nk = make_uint2(0u, 0u), nv = make_uint2(0u, 0u);   // this lane's 4 elements

    int inflight = 0;
    for (int k = 0; k < S && more; ++k) {
        issue();
        ++inflight;
    }

    int cslot = 0;
    uint32_t cphase = 0;
    while (inflight > 0) {
        const int slot = cslot;
        uint8_t *sp = slots + slot * L::kSlotBytes;
        const uint32_t sa = sm_base + slot * L::kSlotBytes;
        if (!mbar_try_wait(&bars[slot], cphase) && !mbar_wait_bounded(&bars[slot], cphase)) {
            if (lane == 0) report(p.err_flag, 0x10 /* PA_FLAG_TIMEOUT */);
            return;
        }
        if (++cslot == S) {
            cslot = 0;
            cphase ^= 1u;
        }
        const StageMeta m = meta[slot];

        if (m.j == 0) {
            nj = -1;
            if (append && m.part == m.nparts - 1 && ctx_s[m.s] > 0) {
                const int pos = ctx_s[m.s] - 1;
                const int rel = pos - m.part * P;
                nj = rel / kStageTokens;
                nrow = rel % kStageTokens;
                npos = pos;
                nid = __ldg(p.block_tables + static_cast<int64_t>(m.s) * p.max_blocks_per_seq + pos / bs);
                const int64_t src = (static_cast<int64_t>(m.s) * Hkv + m.kvh) * D + 4 * lane;
                if constexpr (D == 128) {
                    nk = __ldg(reinterpret_cast<const uint2 *>(static_cast<const uint16_t *>(p.new_k) + src));
                    nv = __ldg(reinterpret_cast<const uint2 *>(static_cast<const uint16_t *>(p.new_v) + src));
                } else if (lane < 16) {
                    nk = __ldg(reinterpret_cast<const uint2 *>(static_cast<const uint16_t *>(p.new_k) + src));
                    nv = __ldg(reinterpret_cast<const uint2 *>(static_cast<const uint16_t *>(p.new_v) + src));
                }
            }
            // New item: the query's B fragments straight from the slot (16-bit).
            const uint32_t *qw = reinterpret_cast<const uint32_t *>(sp + L::kQOffset);
            if constexpr (!kFp8) {
#pragma unroll
                for (int ks = 0; ks < KS; ++ks) {
                    qf[ks][0] = g < G ? qw[(g * D + ks * 16 + 2 * t) >> 1] : 0u;
                    qf[ks][1] = g < G ? qw[(g * D + ks * 16 + 2 * t + 8) >> 1] : 0u;
                }
            } else {
                // Dims in the order the e4m3 K fragments arrive (see QK):
                // step 2kc+hl takes dims 32kc + 4t + 2hl (+1) and the same + 16.
#pragma unroll
                for (int ks = 0; ks < KS; ++ks) {
                    const int d = 32 * (ks >> 1) + 4 * t + 2 * (ks & 1);
#pragma unroll
                    for (int k = 0; k < 2; ++k) {
                        uint32_t w = g < G ? qw[(g * D + d + 16 * k) >> 1] : 0u;
                        if constexpr (kQBf16) {
                            const float2 f = Half2x<true>::to_float2(w);
                            w = pack2<false>(f.x, f.y);
                        }
                        qf[ks][k] = w;
                    }
                }
            }
#pragma unroll
            for (int e = 0; e < 2; ++e) {
                m_run[e] = -INFINITY;
                l_run[e] = 0.f;
            }
#pragma unroll
            for (int mt = 0; mt < MT; ++mt) acc[mt][0] = acc[mt][1] = acc[mt][2] = acc[mt][3] = 0.f;
        }

        // The slot's SUB stages (m.j, m.j + 1, ...) are processed jointly: QK of
        // each, one softmax update over all their tokens, PV of each.  A second
        // stage past the item's end (odd stage count) is skipped.
        const bool second = SUB > 1 && m.j + 1 < m.nst;
        int smask[SUB];
#pragma unroll
        for (int hs = 0; hs < SUB; ++hs)
            smask[hs] = static_cast<int>((static_cast<uint32_t>(m.mask) >> (kStageTokens * hs)) & 0xffffu);

#pragma unroll
        for (int hs = 0; hs < SUB; ++hs) {
            uint8_t *sp_h = sp + hs * L::kHalfBytes;   // stage m.j + hs: K rows here, V at + kVOffset
            if (m.j + hs == nj && ((smask[hs] >> nrow) & 1) && nid >= 0 && nid < p.num_blocks) {
                // This stage holds the step's new token: put its K/V row into the
                // tile (in place of whatever the cache slot held) and into the cache.
                const int64_t nslot = static_cast<int64_t>(nid) * bs + npos % bs;
                const int64_t row_off = (nslot * Hkv + m.kvh) * D;
                if constexpr (kFp8) {
                    const float2 a = Half2x<kQBf16>::to_float2(nk.x), b = Half2x<kQBf16>::to_float2(nk.y);
                    const float2 c2 = Half2x<kQBf16>::to_float2(nv.x), d2 = Half2x<kQBf16>::to_float2(nv.y);
                    const uint32_t ck = f32x2_to_e4m3x2(__fdiv_rn(a.x, p.k_scale_w), __fdiv_rn(a.y, p.k_scale_w)) |
                                        (f32x2_to_e4m3x2(__fdiv_rn(b.x, p.k_scale_w), __fdiv_rn(b.y, p.k_scale_w)) << 16);
                    const uint32_t cv = f32x2_to_e4m3x2(__fdiv_rn(c2.x, p.v_scale_w), __fdiv_rn(c2.y, p.v_scale_w)) |
                                        (f32x2_to_e4m3x2(__fdiv_rn(d2.x, p.v_scale_w), __fdiv_rn(d2.y, p.v_scale_w)) << 16);
                    const int off = nrow * kRowBytes + (((lane >> 2) ^ (nrow & 7)) << 4) + (lane & 3) * 4;
                    *reinterpret_cast<uint32_t *>(sp_h + off) = ck;
                    *reinterpret_cast<uint32_t *>(sp_h + L::kVOffset + off) = cv;
                    reinterpret_cast<uint32_t *>(static_cast<uint8_t *>(p.k_cache_w) + row_off)[lane] = ck;
                    reinterpret_cast<uint32_t *>(static_cast<uint8_t *>(p.v_cache_w) + row_off)[lane] = cv;
                } else {
                    if (D == 128 || lane < 16) {
                        const int hr = D == 128 ? (lane >> 4) : 0, cc = (lane & 15) >> 1, sub = (lane & 1) * 8;
                        const int off = hr * kRegionBytes + nrow * kRowBytes + ((cc ^ (nrow & 7)) << 4) + sub;
                        *reinterpret_cast<uint2 *>(sp_h + off) = nk;
                        *reinterpret_cast<uint2 *>(sp_h + L::kVOffset + off) = nv;
                        uint2 *kd = reinterpret_cast<uint2 *>(static_cast<uint16_t *>(p.k_cache_w) + row_off);
                        uint2 *vd = reinterpret_cast<uint2 *>(static_cast<uint16_t *>(p.v_cache_w) + row_off);
                        kd[lane] = nk;
                        vd[lane] = nv;
                    }
                }
                __syncwarp();
            }
        }

        // ---- QK^T per stage: 16 tokens x 8 heads, two accumulators over the dim steps ----
        // x[hs][i]: i = 0 (token g, head 2t), 1 (g, 2t+1), 2 (g+8, 2t), 3 (g+8, 2t+1)
        float x[SUB][4];
#pragma unroll
        for (int hs = 0; hs < SUB; ++hs) {
            if (hs > 0 && !second) {
                x[hs][0] = x[hs][1] = x[hs][2] = x[hs][3] = -INFINITY;
                continue;
            }
            const uint32_t sa_h = sa + hs * L::kHalfBytes;
            float c[2][4] = {{0.f, 0.f, 0.f, 0.f}, {0.f, 0.f, 0.f, 0.f}};
            {
                const int j = lane >> 3, r = lane & 7;
                const int tok = r + 8 * (j & 1);
                if constexpr (!kFp8) {
#pragma unroll
                    for (int ks = 0; ks < KS; ++ks) {
                        const int ch = 2 * ks + (j >> 1);
                        uint32_t a[4];
                        ldsm_x4(a, sa_h + (ch >> 3) * kRegionBytes + tok * kRowBytes + (((ch & 7) ^ r) << 4));
                        mma_16816<BF16>(c[ks & 1], a, qf[ks][0], qf[ks][1]);
                    }
                } else {
                    // ldmatrix on the byte tile viewed as 16-bit: each register holds
                    // four consecutive dims of one token; split into two f16 pairs,
                    // each 32-dim chunk feeds two MMAs (dims permuted alike in q).
#pragma unroll
                    for (int kc = 0; kc < D / 32; ++kc) {
                        const int ch = 2 * kc + (j >> 1);
                        uint32_t a[4], lo[4], hi[4];
                        ldsm_x4(a, sa_h + tok * kRowBytes + ((ch ^ r) << 4));
#pragma unroll
                        for (int i = 0; i < 4; ++i) e4m3x4_to_f16x2x2(a[i], lo[i], hi[i]);
                        mma_16816<false>(c[0], lo, qf[2 * kc][0], qf[2 * kc][1]);
                        mma_16816<false>(c[1], hi, qf[2 * kc + 1][0], qf[2 * kc + 1][1]);
                    }
                }
            }
            const bool v_lo = (smask[hs] >> g) & 1, v_hi = (smask[hs] >> (g + 8)) & 1;
            const bool h0 = 2 * t < G, h1 = 2 * t + 1 < G;
            const float sc = p.scale_log2;
            x[hs][0] = (v_lo && h0) ? (c[0][0] + c[1][0]) * sc : -INFINITY;
            x[hs][1] = (v_lo && h1) ? (c[0][1] + c[1][1]) * sc : -INFINITY;
            x[hs][2] = (v_hi && h0) ? (c[0][2] + c[1][2]) * sc : -INFINITY;
            x[hs][3] = (v_hi && h1) ? (c[0][3] + c[1][3]) * sc : -INFINITY;
        }

        // ---- one online-softmax update over the slot's tokens ----
        float mx[2] = {fmaxf(x[0][0], x[0][2]), fmaxf(x[0][1], x[0][3])};
#pragma unroll
        for (int hs = 1; hs < SUB; ++hs) {
            mx[0] = fmaxf(mx[0], fmaxf(x[hs][0], x[hs][2]));
            mx[1] = fmaxf(mx[1], fmaxf(x[hs][1], x[hs][3]));
        }
#pragma unroll
        for (int o = 4; o < 32; o <<= 1) {
            mx[0] = fmaxf(mx[0], __shfl_xor_sync(kFull, mx[0], o));
            mx[1] = fmaxf(mx[1], __shfl_xor_sync(kFull, mx[1], o));
        }
        // Lazy rescaling: keep the running reference max unless a new logit
        // exceeds it by more than 2^8 (weights stay <= 256, exact in fp32).
        const bool need = mx[0] > m_run[0] + 8.f || mx[1] > m_run[1] + 8.f;
        if (__any_sync(kFull, need)) {
            float alpha[2];
#pragma unroll
            for (int e = 0; e < 2; ++e) {
                const float m_new = fmaxf(m_run[e], mx[e]);
                alpha[e] = (m_new == -INFINITY) ? 1.f : fast_exp2(m_run[e] - m_new);
                m_run[e] = m_new;
                l_run[e] *= alpha[e];
            }
#pragma unroll
            for (int mt = 0; mt < MT; ++mt) {
                acc[mt][0] *= alpha[0];
                acc[mt][1] *= alpha[1];
                acc[mt][2] *= alpha[0];
                acc[mt][3] *= alpha[1];
            }
        }
        const float mu0 = m_run[0] == -INFINITY ? 0.f : m_run[0];
        const float mu1 = m_run[1] == -INFINITY ? 0.f : m_run[1];

        // ---- per stage: weights, P as the PV B fragment, PV ----
#pragma unroll
        for (int hs = 0; hs < SUB; ++hs) {
            if (hs > 0 && !second) continue;
            const float p0 = fast_exp2(x[hs][0] - mu0), p1 = fast_exp2(x[hs][1] - mu1);
            const float p2 = fast_exp2(x[hs][2] - mu0), p3 = fast_exp2(x[hs][3] - mu1);
            l_run[0] += p0 + p2;
            l_run[1] += p1 + p3;

            // lane needs p(token 2t|2t+1|2t+8|2t+9, head g)
            uint32_t bhi[2], blo[2];
            {
                const int srcA = 8 * t + (g >> 1), srcB = srcA + 4;
                const bool odd = g & 1;
                const float a0 = __shfl_sync(kFull, p0, srcA), a1 = __shfl_sync(kFull, p1, srcA);
                const float a2 = __shfl_sync(kFull, p2, srcA), a3 = __shfl_sync(kFull, p3, srcA);
                const float b0 = __shfl_sync(kFull, p0, srcB), b1 = __shfl_sync(kFull, p1, srcB);
                const float b2 = __shfl_sync(kFull, p2, srcB), b3 = __shfl_sync(kFull, p3, srcB);
                const float w[4] = {odd ? a1 : a0, odd ? b1 : b0, odd ? a3 : a2, odd ? b3 : b2};
                // Split each weight into a 16-bit high part and a 16-bit residual,
                // so the tensor-core product keeps ~16 significant bits of p.
#pragma unroll
                for (int k = 0; k < 2; ++k) {
                    bhi[k] = pack2<BF16>(w[2 * k], w[2 * k + 1]);
                    const float2 h = Cvt::to_float2(bhi[k]);
                    blo[k] = pack2<BF16>(w[2 * k] - h.x, w[2 * k + 1] - h.y);
                }
            }

            // rows past the context are zeroed first
            uint8_t *sp_h = sp + hs * L::kHalfBytes;
            const uint32_t va = sa + hs * L::kHalfBytes + L::kVOffset;
            if (smask[hs] != 0xffff) {
                // Stale rows (past the context, or of a skipped block) may hold
                // NaN; 0 * NaN would poison the tensor-core sums, so clear them.
                uint8_t *vt = sp_h + L::kVOffset;
#pragma unroll
                for (int k = 0; k < kStageTokens * L::kBoxes * 8 / 32; ++k) {
                    const int q16 = lane + 32 * k;                // 16-byte chunk index
                    const int row = (q16 >> 3) % kStageTokens;    // 8 chunks per 128-byte row
                    if (!((smask[hs] >> row) & 1))
                        *reinterpret_cast<uint4 *>(vt + q16 * 16) = make_uint4(0u, 0u, 0u, 0u);
                }
                __syncwarp();
            }
            {
                const int j = lane >> 3, r = lane & 7;
                const int tok = r + 8 * (j >> 1);
                if constexpr (!kFp8) {
#pragma unroll
                    for (int mt = 0; mt < MT; ++mt) {
                        const int ch = 2 * mt + (j & 1);
                        uint32_t a[4];
                        ldsm_x4_trans(a, va + (ch >> 3) * kRegionBytes + tok * kRowBytes + (((ch & 7) ^ r) << 4));
                        mma_16816<BF16>(acc[mt], a, bhi[0], bhi[1]);
                        mma_16816<BF16>(acc[mt], a, blo[0], blo[1]);
                    }
                } else {
                    // Transposed ldmatrix of the byte tile viewed as 16-bit gives
                    // (tokens 2t, 2t+1) x (dims 2g, 2g+1); regroup the bytes so
                    // each f16 pair is one dim over two tokens: even dims feed
                    // acc[2vc], odd dims acc[2vc+1].
#pragma unroll
                    for (int vc = 0; vc < D / 32; ++vc) {
                        const int ch = 2 * vc + (j & 1);
                        uint32_t a[4], ev[4], od[4];
                        ldsm_x4_trans(a, va + tok * kRowBytes + ((ch ^ r) << 4));
#pragma unroll
                        for (int i = 0; i < 4; ++i) e4m3x4_to_f16x2x2(prmt(a[i], 0x3120u), ev[i], od[i]);
                        mma_16816<false>(acc[2 * vc], ev, bhi[0], bhi[1]);
                        mma_16816<false>(acc[2 * vc], ev, blo[0], blo[1]);
                        mma_16816<false>(acc[2 * vc + 1], od, bhi[0], bhi[1]);
                        mma_16816<false>(acc[2 * vc + 1], od, blo[0], blo[1]);
                    }
                }
            }
        }

        // ---- item end: output (or partial state) staged through shared memory ----
        if (m.j + SUB >= m.nst) {
            float lt[2] = {l_run[0], l_run[1]};
#pragma unroll
            for (int o = 4; o < 32; o <<= 1) {
                lt[0] += __shfl_xor_sync(kFull, lt[0], o);
                lt[1] += __shfl_xor_sync(kFull, lt[1], o);
            }
            const bool final_out = m.nparts == 1;
#pragma unroll
            for (int e = 0; e < 2; ++e) {
                const int h = 2 * t + e;
                if (h < G) {
                    const float s = (final_out ? (lt[e] > 0.f ? 1.f / lt[e] : 0.f) : 1.f) * p.v_scale;
                    float *orow = obuf + h * L::kOStride;
                    if constexpr (!kFp8) {
#pragma unroll
                        for (int mt = 0; mt < MT; ++mt) {
                            orow[mt * 16 + g] = acc[mt][e] * s;
                            orow[mt * 16 + g + 8] = acc[mt][2 + e] * s;
                        }
                    } else {
#pragma unroll
                        for (int vc = 0; vc < D / 32; ++vc) {
                            orow[32 * vc + 2 * g] = acc[2 * vc][e] * s;
                            orow[32 * vc + 16 + 2 * g] = acc[2 * vc][2 + e] * s;
                            orow[32 * vc + 2 * g + 1] = acc[2 * vc + 1][e] * s;
                            orow[32 * vc + 16 + 2 * g + 1] = acc[2 * vc + 1][2 + e] * s;
                        }
                    }
                }
            }
            __syncwarp();
            const int d0 = lane * DPL;
            if (final_out) {
                const int64_t orow0 = static_cast<int64_t>(m.s) * Hq + m.kvh * G;
#pragma unroll
                for (int h = 0; h < G; ++h) store_row<D>(p.out, p.out_dtype, (orow0 + h) * D + d0, obuf + h * L::kOStride + d0);
            } else {
                const int64_t slot_id = (static_cast<int64_t>(m.s) * Hkv + m.kvh) * p.max_partitions + m.part;
                // Partials stay in L2 (evict-last) for the merge kernel.
#pragma unroll
                for (int h = 0; h < G; ++h) {
                    float *dst = p.ws_acc + (slot_id * G + h) * D + d0;
                    const float *src = obuf + h * L::kOStride + d0;
                    if constexpr (DPL == 4)
                        st_global_hint(dst, make_float4(src[0], src[1], src[2], src[3]), keep);
                    else
                        st_global_hint(dst, make_float2(src[0], src[1]), keep);
                }
#pragma unroll
                for (int e = 0; e < 2; ++e) {
                    const int h = 2 * t + e;
                    if (g == 0 && h < G)
                        st_global_hint(p.ws_ml + (slot_id * G + h) * 2, make_float2(m_run[e], lt[e]), keep);
                }
            }
            __syncwarp();
        }

        --inflight;
        if (more) {
            fence_proxy_async_smem();
            __syncwarp();
            issue();
            ++inflight;
        } else {
            __syncwarp();
        }
    }
}

// Merge of split sequences: for each (sequence, KV head, query head) with more
// than one partition, combine the partial states (m_j, l_j, acc_j) in
// partition order:  M = max_j m_j,
//   out = sum_j acc_j 2^(m_j - M) / sum_j l_j 2^(m_j - M).
// `wt` warps share one task (1, 2, 4 or 8; more for long partition lists):
// each takes a contiguous run of partitions with eight acc loads in flight,
// and the first folds the runs together in shared memory in run order.
// Launched after the decode kernel with programmatic dependent launch.
template <int D, int G>
__global__ void __launch_bounds__(256)
    paged_decode_merge_kernel(const __grid_constant__ DecodeParams p, int wt) {
    pdl_wait();
    constexpr int DPL = D / 32;
    __shared__ float red_o[8][D];
    __shared__ float red_l[8];
    const int lane = threadIdx.x & 31, warp = threadIdx.x >> 5;
    const int64_t task = static_cast<int64_t>(blockIdx.x) * (8 / wt) + warp / wt;
    const int sub = warp % wt;
    const int Hkv = p.num_kv_heads;
    bool active = task < static_cast<int64_t>(p.num_seqs) * Hkv * G;
    int np = 1, s = 0, kvh = 0, h = 0;
    int64_t pair = 0;
    if (active) {
        h = static_cast<int>(task % G);
        pair = task / G;
        s = static_cast<int>(pair / Hkv);
        kvh = static_cast<int>(pair % Hkv);
        int ctx = p.context_lens[s];
        if (ctx < 0 || ctx > p.max_context_len) ctx = 0;
        np = ctx > 0 ? (ctx + p.partition_size - 1) / p.partition_size : 1;
        active = np > 1;
    }
    const int d0 = lane * DPL;
    float Lp = 0.f, o[DPL];
#pragma unroll
    for (int i = 0; i < DPL; ++i) o[i] = 0.f;
    if (active) {
        const int64_t base = pair * p.max_partitions;
        const float *mlh = p.ws_ml + (base * G + h) * 2;
        float mx = -INFINITY;
        for (int j = lane; j < np; j += 32) mx = fmaxf(mx, __ldcg(mlh + static_cast<int64_t>(j) * G * 2));
        const float M = warp_max(mx);
        const int per = (np + wt - 1) / wt;
        const int jb = min(np, sub * per), je = min(np, jb + per);
        for (int j0 = jb; j0 < je; j0 += 32) {
            const int j = j0 + lane;
            float w = 0.f;
            if (j < je) {
                const float2 ml = __ldcg(reinterpret_cast<const float2 *>(mlh + static_cast<int64_t>(j) * G * 2));
                w = (ml.x == -INFINITY) ? 0.f : fast_exp2(ml.x - M);
                Lp = fmaf(ml.y, w, Lp);
            }
            const int cnt = min(32, je - j0);
            const float *ap0 = p.ws_acc + ((base + j0) * G + h) * D + d0;
            for (int u0 = 0; u0 < cnt; u0 += 8) {
                float v[8][DPL];
#pragma unroll
                for (int u = 0; u < 8; ++u) {
                    if (u0 + u < cnt) {
                        const float *ap = ap0 + static_cast<int64_t>(u0 + u) * G * D;
                        if constexpr (DPL == 4) {
                            const float4 x = __ldcg(reinterpret_cast<const float4 *>(ap));
                            v[u][0] = x.x; v[u][1] = x.y; v[u][2] = x.z; v[u][3] = x.w;
                        } else {
                            const float2 x = __ldcg(reinterpret_cast<const float2 *>(ap));
                            v[u][0] = x.x; v[u][1] = x.y;
                        }
                    } else {
#pragma unroll
                        for (int i = 0; i < DPL; ++i) v[u][i] = 0.f;
                    }
                }
#pragma unroll
                for (int u = 0; u < 8; ++u) {
                    const float wj = __shfl_sync(kFull, w, (u0 + u) & 31);
#pragma unroll
                    for (int i = 0; i < DPL; ++i) o[i] = fmaf(v[u][i], wj, o[i]);
                }
            }
        }
        Lp = warp_sum(Lp);
    }
    if (wt > 1) {
#pragma unroll
        for (int i = 0; i < DPL; ++i) red_o[warp][d0 + i] = o[i];
        if (lane == 0) red_l[warp] = Lp;
        __syncthreads();
        if (!active || sub != 0) return;
        for (int k = 1; k < wt; ++k) {
#pragma unroll
            for (int i = 0; i < DPL; ++i) o[i] += red_o[warp + k][d0 + i];
            Lp += red_l[warp + k];
        }
    } else if (!active) {
        return;
    }
    const float inv = Lp > 0.f ? 1.f / Lp : 0.f;
#pragma unroll
    for (int i = 0; i < DPL; ++i) o[i] *= inv;
    store_row<D>(p.out, p.out_dtype, (static_cast<int64_t>(s) * p.num_heads + kvh * G + h) * D + d0, o);
}

template <int D, int G, int ES>
size_t smem_for(int warps, int stages, int num_seqs) {
    using L = Layout<D, G, ES>;
    size_t per_warp = static_cast<size_t>(stages) * (L::kSlotBytes + kMetaBytes + 8) + L::kOBytes;
    return 1024 + per_warp * warps + 32 * 4 + 4 * static_cast<size_t>(num_seqs) +
           4 * (static_cast<size_t>(num_seqs) + 1);
}

template <int D, int G, int KV>
cudaError_t launch_t(const DecodeParams &p, const CUtensorMap &tk, const CUtensorMap &tv,
                     int grid, int warps, size_t smem, cudaStream_t stream) {
    auto kern = paged_decode_kernel<D, G, KV>;
    cudaError_t e = cudaFuncSetAttribute(kern, cudaFuncAttributeMaxDynamicSharedMemorySize,
                                         static_cast<int>(smem));
    if (e != cudaSuccess) return e;
    e = launch_pdl(kern, dim3(grid), dim3(warps * 32), smem, stream, p, tk, tv);
    if (e != cudaSuccess) return e;
    return launch_decode_merge(p, D, G, stream);
}

// Merge of split sequences: 1-8 warps per (sequence, KV head, query head),
// about 16 partitions per warp.
template <int D, int G>
cudaError_t launch_merge_t(const DecodeParams &p, cudaStream_t stream) {
    int wt = 1;
    while (wt < 8 && wt * 16 < p.max_partitions) wt *= 2;
    const int64_t tasks = static_cast<int64_t>(p.num_seqs) * p.num_kv_heads * G;
    const int64_t per_cta = 8 / wt;
    return launch_pdl(paged_decode_merge_kernel<D, G>,
                      dim3(static_cast<unsigned>((tasks + per_cta - 1) / per_cta)), dim3(256), 0,
                      stream, p, wt);
}

template <int D>
cudaError_t launch_merge_g(const DecodeParams &p, int group, cudaStream_t stream) {
    switch (group) {
        case 1: return launch_merge_t<D, 1>(p, stream);
        case 2: return launch_merge_t<D, 2>(p, stream);
        case 4: return launch_merge_t<D, 4>(p, stream);
        case 8: return launch_merge_t<D, 8>(p, stream);
        default: return cudaErrorInvalidValue;
    }
}

template <int D, int G>
cudaError_t launch_kv(const DecodeParams &p, int kv, const CUtensorMap &tk, const CUtensorMap &tv,
                      int grid, int warps, size_t smem, cudaStream_t stream) {
    switch (kv) {
        case 0: return launch_t<D, G, 0>(p, tk, tv, grid, warps, smem, stream);
        case 1: return launch_t<D, G, 1>(p, tk, tv, grid, warps, smem, stream);
        case 2:
            if constexpr (D == 128) return launch_t<D, G, 2>(p, tk, tv, grid, warps, smem, stream);
            return cudaErrorInvalidValue;
        case 3:
            if constexpr (D == 128) return launch_t<D, G, 3>(p, tk, tv, grid, warps, smem, stream);
            return cudaErrorInvalidValue;
        default: return cudaErrorInvalidValue;
    }
}

template <int D>
cudaError_t launch_g(const DecodeParams &p, int group, int kv, const CUtensorMap &tk,
                     const CUtensorMap &tv, int grid, int warps, size_t smem,
                     cudaStream_t stream) {
    switch (group) {
        case 1: return launch_kv<D, 1>(p, kv, tk, tv, grid, warps, smem, stream);
        case 2: return launch_kv<D, 2>(p, kv, tk, tv, grid, warps, smem, stream);
        case 4: return launch_kv<D, 4>(p, kv, tk, tv, grid, warps, smem, stream);
        case 8: return launch_kv<D, 8>(p, kv, tk, tv, grid, warps, smem, stream);
        default: return cudaErrorInvalidValue;
    }
}

template <int D, int ES>
size_t smem_g(int group, int warps, int stages, int num_seqs) {
    switch (group) {
        case 1: return smem_for<D, 1, ES>(warps, stages, num_seqs);
        case 2: return smem_for<D, 2, ES>(warps, stages, num_seqs);
        case 4: return smem_for<D, 4, ES>(warps, stages, num_seqs);
        case 8: return smem_for<D, 8, ES>(warps, stages, num_seqs);
        default: return 0;
    }
}

}  // namespace

size_t decode_smem_bytes(int head_dim, int group, int elem_bytes, int warps, int stages, int num_seqs) {
    if (head_dim == 64) return smem_g<64, 2>(group, warps, stages, num_seqs);
    return elem_bytes == 1 ? smem_g<128, 1>(group, warps, stages, num_seqs)
                           : smem_g<128, 2>(group, warps, stages, num_seqs);
}

cudaError_t launch_decode_merge(const DecodeParams &p, int head_dim, int group, cudaStream_t stream) {
    if (p.max_partitions <= 1) return cudaSuccess;
    if (head_dim == 64) return launch_merge_g<64>(p, group, stream);
    if (head_dim == 128) return launch_merge_g<128>(p, group, stream);
    return cudaErrorInvalidValue;
}

cudaError_t launch_decode(const DecodeParams &p, int head_dim, int group, int kv,
                          const CUtensorMap &tk, const CUtensorMap &tv, int grid, int warps,
                          size_t smem, cudaStream_t stream) {
    if (head_dim == 64) return launch_g<64>(p, group, kv, tk, tv, grid, warps, smem, stream);
    if (head_dim == 128) return launch_g<128>(p, group, kv, tk, tv, grid, warps, smem, stream);
    return cudaErrorInvalidValue;
}

}  // namespace pa
