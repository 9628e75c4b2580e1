// Paged decode attention, CTA-cooperative variant (16-bit or e4m3 caches,
// KV-head count a multiple of 8, head_dim 128, block_size a multiple of 16).
//
// Computes what the per-warp kernel in pa_decode.cu computes - softmax(q K^T *
// scale) V over each sequence's context_lens[s] cached tokens, reached through
// its block table ("LLM推理优化：vLLM PagedAttention深度解析与工程实践", §二,
// §3.1, §4.1; nano-vllm walkthrough lqnn.cn/news/170268, §2.3), partitions
// merged in order by the same merge kernel - with a different way of moving
// the cache:
//  * A CTA works on items (sequence, partition, group of 8 KV heads).  One
//    producer warp brings each 16-token stage in with one TMA box per 128-byte
//    column block of K and of V covering all 8 heads ({64, 16 rows, 8 heads}
//    for 16-bit caches, two per row; {128, 16, 8} for e4m3, one per row: 16 KB,
//    the heads' 16 rows of one physical block), instead of one 2 KB box per
//    head and column block.  The tensor map orders its dimensions (dim, token,
//    head) so that each head's 16 rows land contiguously with the 128-byte
//    swizzle, as the per-warp kernel's do.
//  * Eight consumer warps each take one head of the group and run the same
//    warp-level MMA math on their slice of the shared stage: QK with the 16
//    tokens as M and the G query heads as N (padded to 8), online softmax in
//    base 2 with lazy rescaling, PV with the weights as a 16-bit high part
//    plus residual.  e4m3 codes are widened to f16 pairs in registers (every
//    e4m3 value is exact in f16) and multiplied as f16, the query rounded to
//    f16; the per-tensor scales are folded into the logit scale and the output.
//  * Slots are CTA-wide: `full` completes when a stage's copies land, `empty`
//    when all eight consumers are done with it; every wait is bounded and a
//    timeout sets PA_FLAG_TIMEOUT.  An item's query rows go to a 2-entry ring
//    of their own (read once, at the item's first stage), so slots hold only
//    K and V and a 3-deep ring fits for groups of up to 4 query heads per KV
//    head.  An e4m3 slot holds two consecutive stages of one item (64 KB, as
//    a 16-bit slot), consumed under one softmax update, so that each consumer's
//    chain of dependent steps covers 32 tokens of 1-byte codes.  The producer also owns the work cursor and the block-table reads,
//    so the consumers' loop holds only the math.
#include "pa_decode_common.cuh"
#include "pa_device.cuh"
#include "pa_internal.h"

namespace pa {

namespace {

using namespace decode_common;

constexpr int kGroupHeads = 8;                    // KV heads per box and consumer warps
constexpr int kCoopThreads = (kGroupHeads + 1) * 32;
constexpr int kRow = 128;                         // bytes of one swizzled 64-element row half
constexpr int kHeadTile = kStageTokens * kRow;    // one head's 16 rows of one half: 2 KB

// ES = bytes per cache element (2: f16/bf16, 1: e4m3).
template <int D, int G, int ES, int SUB = (ES == 1 ? 2 : 1)>
struct CoopLayout {
    static constexpr int kSub = SUB;                                // stages per slot
    static constexpr int kHalves = D * ES / kRow;                   // 128-byte column blocks per row
    static constexpr int kBoxElems = kRow / ES;                     // elements per box row
    static constexpr int kBoxBytes = kGroupHeads * kHeadTile;      // 16 KB
    static constexpr int kKBytes = kHalves * kBoxBytes;
    static constexpr int kVOffset = kKBytes;
    static constexpr int kQBytes = kGroupHeads * G * D * 2;         // the group's query rows
    static constexpr int kStageBytes = 2 * kKBytes;                 // K and V of one stage
    static constexpr int kSlotBytes = SUB * kStageBytes;
    static constexpr int kOStride = D + 4;
    static constexpr int kOBytes = G * kOStride * 4;                // per consumer warp
    static constexpr int kSteps = D / 16;
    static constexpr int kDimsPerLane = D / 32;
};

struct CoopMeta {
    int s, kvh0, part, j;        // s < 0: no more work; j = the slot's first stage
    int nst, nparts, mask, pad;  // mask bit 16 * hs + r: row r of the slot's stage hs is valid
};

// The items' query rows sit in a ring of their own (kQRing entries, one per
// item), so that stage slots hold only K and V.
constexpr int kQRing = 2;

__device__ __forceinline__ void mbar_arrive1(uint64_t *bar) {
    asm volatile("mbarrier.arrive.shared::cta.b64 _, [%0];" ::"r"(smem_addr(bar)) : "memory");
}

// Items (s, part, group) in that order; an item weighs 8 x its stages.
struct CoopCursor {
    int s, part, grp;
    int ctx, nparts, ntok, nst;
    uint32_t start;

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
    __device__ __forceinline__ void advance(const int *ctx_s, int ngroups, int P, int B) {
        start += static_cast<uint32_t>(kGroupHeads * nst);
        if (++grp < ngroups) return;
        grp = 0;
        if (part + 1 < nparts) {
            set_part(part + 1, P);
            return;
        }
        if (s + 1 < B) {
            set_seq(s + 1, ctx_s, P);
            set_part(0, P);
        }
    }
};

// KV: 0 = f16 cache and query, 1 = bf16 cache and query, 2 / 3 = e4m3 cache
// with an f16 / bf16 query (f16 MMAs).
template <int D, int G, int KV>
__global__ void __launch_bounds__(kCoopThreads, 1)
    paged_decode_coop_kernel(const __grid_constant__ DecodeParams p,
                             const __grid_constant__ CUtensorMap tmap_k,
                             const __grid_constant__ CUtensorMap tmap_v) {
    static_assert(D == 128, "the cooperative kernel is built for head_dim 128");
    constexpr bool kFp8 = KV >= 2;
    constexpr bool BF16 = KV == 1;                 // MMA operand type
    constexpr bool kQBf16 = KV == 1 || KV == 3;    // query type
    using L = CoopLayout<D, G, kFp8 ? 1 : 2>;
    constexpr int SUB = L::kSub;
    using Cvt = Half2x<BF16>;
    constexpr int KS = L::kSteps;
    constexpr int MT = L::kSteps;
    constexpr int DPL = L::kDimsPerLane;
    extern __shared__ uint8_t smem_raw[];
    uint8_t *smem = reinterpret_cast<uint8_t *>(
        (reinterpret_cast<uintptr_t>(smem_raw) + 1023) & ~static_cast<uintptr_t>(1023));

    const int lane = threadIdx.x & 31;
    const int warp = threadIdx.x >> 5;
    const int S = p.stages;
    const int B = p.num_seqs;
    const int Hkv = p.num_kv_heads;
    const int Hq = p.num_heads;
    const int P = p.partition_size;
    const int bs = p.block_size;
    const int ngroups = Hkv / kGroupHeads;

    uint8_t *slots = smem;
    uint8_t *qbuf = smem + static_cast<size_t>(S) * L::kSlotBytes;   // kQRing x kQBytes
    uint8_t *misc = qbuf + kQRing * L::kQBytes;
    CoopMeta *meta = reinterpret_cast<CoopMeta *>(misc);
    misc += S * sizeof(CoopMeta);
    uint64_t *full = reinterpret_cast<uint64_t *>(misc);
    uint64_t *empty = full + S;
    uint64_t *qfull = empty + S;
    uint64_t *qempty = qfull + kQRing;
    misc += (2 * S + 2 * kQRing) * 8;
    float *obuf_all = reinterpret_cast<float *>(misc);
    misc += kGroupHeads * L::kOBytes;
    uint32_t *warp_tot = reinterpret_cast<uint32_t *>(misc);
    misc += 32 * 4;
    int *ctx_s = reinterpret_cast<int *>(misc);
    uint32_t *prefix = reinterpret_cast<uint32_t *>(misc + 4 * B);

    if (threadIdx.x == 0) {
        for (int i = 0; i < S; ++i) {
            mbar_init(&full[i], 1);
            mbar_init(&empty[i], kGroupHeads);
        }
        for (int i = 0; i < kQRing; ++i) {
            mbar_init(&qfull[i], 1);
            mbar_init(&qempty[i], kGroupHeads);
        }
        fence_barrier_init();
        prefetch_tensormap(&tmap_k);
        prefetch_tensormap(&tmap_v);
    }
    // Launched with programmatic dependent launch: wait for the previous kernel
    // before reading anything it may have written - at once, or (defer_wait)
    // only before the stages holding a sequence's last position, the one row
    // per sequence that kernel writes.
    const bool defer = p.defer_wait != 0;
    if (!defer) pdl_wait();
    for (int i = threadIdx.x; i < B; i += blockDim.x) {
        int c = p.context_lens[i];
        if (c < 0 || c > p.max_context_len) {
            if (blockIdx.x == 0) report(p.err_flag, 0x4 /* PA_FLAG_BAD_CONTEXT_LEN */);
            c = 0;
        }
        ctx_s[i] = c;
    }
    pdl_launch_dependents();
    __syncthreads();
    {
        // prefix[s] = work (stages x KV heads) of the sequences before s
        const int nthr = blockDim.x;
        const int nw = nthr >> 5;
        const int per = (B + nthr - 1) / nthr;
        const int beg = min(B, threadIdx.x * per);
        const int end = min(B, beg + per);
        uint32_t local = 0;
        for (int i = beg; i < end; ++i) local += seq_weight(ctx_s[i], Hkv);
        uint32_t incl = local;
#pragma unroll
        for (int o = 1; o < 32; o <<= 1) {
            const uint32_t v = __shfl_up_sync(kFull, incl, o);
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
    const uint32_t total = prefix[B];
    const uint32_t lo = static_cast<uint32_t>(static_cast<uint64_t>(total) * blockIdx.x / gridDim.x);
    const uint32_t hi = static_cast<uint32_t>(static_cast<uint64_t>(total) * (blockIdx.x + 1) / gridDim.x);

    if (warp == kGroupHeads) {
        // ------------------------------------------------------------ producer
        const uint64_t policy = l2_policy_evict_first();
        CoopCursor ic;
        {
            // first item whose first stage is >= lo
            int a = 0, b = B;
            while (b - a > 1) {
                const int m = (a + b) >> 1;
                if (prefix[m] <= lo) a = m; else b = m;
            }
            ic.set_seq(a, ctx_s, P);
            const uint32_t off = lo - prefix[a];
            const uint32_t P16 = static_cast<uint32_t>(P / kStageTokens);
            int part = static_cast<int>(off / (static_cast<uint32_t>(Hkv) * P16));
            if (part > ic.nparts - 1) part = ic.nparts - 1;
            ic.set_part(part, P);
            const uint32_t pstart = prefix[a] + static_cast<uint32_t>(part) * Hkv * P16;
            const uint32_t w8 = static_cast<uint32_t>(kGroupHeads * ic.nst);
            int grp = static_cast<int>((off - (pstart - prefix[a]) + w8 - 1) / w8);
            if (grp >= ngroups) {   // step to the next partition or sequence
                ic.grp = ngroups - 1;
                ic.start = pstart + static_cast<uint32_t>(ngroups - 1) * w8;
                ic.advance(ctx_s, ngroups, P, B);
            } else {
                ic.grp = grp;
                ic.start = pstart + static_cast<uint32_t>(grp) * w8;
            }
        }
        int islot = 0;
        uint32_t uses = 0;   // slots filled so far (the empty barrier's phase follows it)
        uint32_t items = 0;  // items started (the query ring's position and phase)
        bool ok = true;
        bool waited = !defer;
        auto take_slot = [&]() -> int {
            const int slot = islot;
            if (uses >= static_cast<uint32_t>(S)) {
                const uint32_t par = ((uses / S) - 1) & 1u;
                if (!mbar_try_wait(&empty[slot], par) && !mbar_wait_bounded(&empty[slot], par)) {
                    if (lane == 0) report(p.err_flag, 0x10 /* PA_FLAG_TIMEOUT */);
                    ok = false;
                }
            }
            islot = (islot + 1 == S) ? 0 : islot + 1;
            ++uses;
            return slot;
        };
        while (ok && ic.start < hi) {
            // this item's block ids, one per lane (an item spans at most 32 blocks)
            const int fb = (ic.part * P) / bs;
            int32_t bid = -1;
            if (ic.ntok > 0) {
                const int lb = (ic.part * P + ic.ntok - 1) / bs;
                if (lane <= lb - fb)
                    bid = __ldg(p.block_tables + static_cast<int64_t>(ic.s) * p.max_blocks_per_seq + fb + lane);
            }
            const int kvh0 = ic.grp * kGroupHeads;
            {
                // the item's query rows into the next entry of the query ring
                const int qi = static_cast<int>(items % kQRing);
                if (items >= static_cast<uint32_t>(kQRing)) {
                    const uint32_t par = ((items / kQRing) - 1) & 1u;
                    if (!mbar_try_wait(&qempty[qi], par) && !mbar_wait_bounded(&qempty[qi], par)) {
                        if (lane == 0) report(p.err_flag, 0x10 /* PA_FLAG_TIMEOUT */);
                        ok = false;
                        break;
                    }
                }
                if (lane == 0) {
                    const bool with_q = ic.ntok > 0;
                    mbar_arrive_expect_tx(&qfull[qi], with_q ? static_cast<uint32_t>(L::kQBytes) : 0u);
                    if (with_q) {
                        const uint16_t *qsrc = static_cast<const uint16_t *>(p.q) +
                                               (static_cast<int64_t>(ic.s) * Hq + kvh0 * G) * D;
                        bulk_load(qbuf + qi * L::kQBytes, qsrc, L::kQBytes, &qfull[qi]);
                    }
                }
                ++items;
                __syncwarp();
            }
            for (int j = 0; ok && j < ic.nst; j += SUB) {
                if (!waited && ic.ntok > 0 && ic.part == ic.nparts - 1 && j + SUB >= ic.nst) {
                    pdl_wait();   // this slot holds the sequence's appended row
                    waited = true;
                }
                const int slot = take_slot();
                if (!ok) break;
                uint8_t *sp = slots + static_cast<size_t>(slot) * L::kSlotBytes;
                uint32_t mask_all = 0, bytes = 0;
                int zs[SUB];
                bool loads[SUB];
#pragma unroll
                for (int hs = 0; hs < SUB; ++hs) {
                    const int jj = j + hs;
                    const int tok0 = ic.part * P + jj * kStageTokens;
                    const int n = (ic.ntok > 0 && jj < ic.nst) ? min(kStageTokens, ic.ntok - jj * kStageTokens) : 0;
                    uint32_t mask = n > 0 ? ((1u << n) - 1u) : 0u;
                    const int id = __shfl_sync(kFull, bid, (tok0 / bs - fb) & 31);
                    const bool load = n > 0 && id >= 0 && static_cast<int64_t>(id) < p.num_blocks;
                    if (n > 0 && !load) {
                        mask = 0;
                        if (lane == 0) report(p.err_flag, 0x2 /* PA_FLAG_BAD_BLOCK_ID */);
                    }
                    mask_all |= mask << (16 * hs);
                    loads[hs] = load;
                    zs[hs] = load ? id * bs + (tok0 % bs) : 0;
                    bytes += load ? 2u * L::kKBytes : 0u;
                }
                if (lane == 0) {
                    CoopMeta m;
                    m.s = ic.s; m.kvh0 = kvh0; m.part = ic.part; m.j = j;
                    m.nst = ic.nst; m.nparts = ic.nparts; m.mask = static_cast<int>(mask_all); m.pad = 0;
                    meta[slot] = m;
                    mbar_arrive_expect_tx(&full[slot], bytes);
#pragma unroll
                    for (int hs = 0; hs < SUB; ++hs) {
                        if (!loads[hs]) continue;
                        uint8_t *st = sp + hs * L::kStageBytes;
#pragma unroll
                        for (int h = 0; h < L::kHalves; ++h) {
                            tma_load_3d(st + h * L::kBoxBytes, &tmap_k, &full[slot], h * L::kBoxElems, zs[hs], kvh0,
                                        policy);
                            tma_load_3d(st + L::kVOffset + h * L::kBoxBytes, &tmap_v, &full[slot],
                                        h * L::kBoxElems, zs[hs], kvh0, policy);
                        }
                    }
                }
                __syncwarp();
            }
            ic.advance(ctx_s, ngroups, P, B);
        }
        // end of work: one more slot tells the consumers to stop
        if (ok) {
            const int slot = take_slot();
            if (ok && lane == 0) {
                CoopMeta m;
                m.s = -1; m.kvh0 = 0; m.part = 0; m.j = 0; m.nst = 0; m.nparts = 0; m.mask = 0; m.pad = 0;
                meta[slot] = m;
                mbar_arrive1(&full[slot]);
            }
        }
        if (!waited) pdl_wait();   // the CTA does not finish before the previous kernel
        __syncwarp();
        return;
    }

    // ---------------------------------------------------------------- consumers
    // Consumer warp w owns KV head kvh0 + w of every item.
    const uint64_t keep = l2_policy_evict_last();
    float *obuf = obuf_all + warp * (L::kOBytes / 4);
    const int g = lane >> 2, t = lane & 3;
    const uint32_t slots_sa = smem_addr(slots);
    uint32_t qf[KS][2];
    float acc[MT][4];
    float m_run[2], l_run[2];
    int cslot = 0;
    uint32_t cphase = 0;
    uint32_t citems = 0;   // items started (the query ring's position and phase)
    for (;;) {
        const int slot = cslot;
        uint8_t *sp = slots + static_cast<size_t>(slot) * L::kSlotBytes;
        const uint32_t sa = slots_sa + slot * L::kSlotBytes;
        if (!mbar_try_wait(&full[slot], cphase) && !mbar_wait_bounded(&full[slot], cphase)) {
            if (lane == 0) report(p.err_flag, 0x10 /* PA_FLAG_TIMEOUT */);
            return;
        }
        if (++cslot == S) {
            cslot = 0;
            cphase ^= 1u;
        }
        const CoopMeta m = meta[slot];
        if (m.s < 0) {
            if (defer) pdl_wait();   // the CTA does not finish before the previous kernel
            break;
        }
        const int kvh = m.kvh0 + warp;

        if (m.j == 0) {
            // new item: my query heads' B fragments from the query ring
            const int qi = static_cast<int>(citems % kQRing);
            const uint32_t qpar = (citems / kQRing) & 1u;
            ++citems;
            if (!mbar_try_wait(&qfull[qi], qpar) && !mbar_wait_bounded(&qfull[qi], qpar)) {
                if (lane == 0) report(p.err_flag, 0x10 /* PA_FLAG_TIMEOUT */);
                return;
            }
            const uint32_t *qw =
                reinterpret_cast<const uint32_t *>(qbuf + qi * L::kQBytes) + warp * (G * D / 2);
            if constexpr (!kFp8) {
#pragma unroll
                for (int ks = 0; ks < KS; ++ks) {
                    qf[ks][0] = g < G ? qw[(g * D + ks * 16 + 2 * t) >> 1] : 0u;
                    qf[ks][1] = g < G ? qw[(g * D + ks * 16 + 2 * t + 8) >> 1] : 0u;
                }
            } else {
                // Dims in the order the widened K fragments arrive (see QK):
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
            fence_proxy_async_smem();
            __syncwarp();
            if (lane == 0) mbar_arrive1(&qempty[qi]);
#pragma unroll
            for (int e = 0; e < 2; ++e) {
                m_run[e] = -INFINITY;
                l_run[e] = 0.f;
            }
#pragma unroll
            for (int mt = 0; mt < MT; ++mt) acc[mt][0] = acc[mt][1] = acc[mt][2] = acc[mt][3] = 0.f;
        }

        // A slot carries SUB stages (two for e4m3 caches, whose 16-token stage is
        // half the bytes of a 16-bit one): QK of each, one softmax update over
        // all of them, then PV of each.  The second stage of an item's last slot
        // may be absent.
        const uint32_t msk = static_cast<uint32_t>(m.mask);
        const bool second = SUB > 1 && m.j + 1 < m.nst;
        float x[SUB][4];
#pragma unroll
        for (int hs = 0; hs < SUB; ++hs) {
            if (hs > 0 && !second) {
                x[hs][0] = x[hs][1] = x[hs][2] = x[hs][3] = -INFINITY;
                continue;
            }
            const uint32_t ka = sa + hs * L::kStageBytes + warp * kHeadTile;
            const uint32_t smask = (msk >> (16 * hs)) & 0xffffu;
            // ---- QK^T: 16 tokens x 8 heads ----
            float c[2][4] = {{0.f, 0.f, 0.f, 0.f}, {0.f, 0.f, 0.f, 0.f}};
            {
                const int j = lane >> 3, r = lane & 7;
                const int tok = r + 8 * (j & 1);
                if constexpr (!kFp8) {
#pragma unroll
                    for (int ks = 0; ks < KS; ++ks) {
                        const int ch = 2 * ks + (j >> 1);
                        uint32_t a[4];
                        ldsm_x4(a, ka + (ch >> 3) * L::kBoxBytes + tok * kRow + (((ch & 7) ^ r) << 4));
                        mma_16816<BF16>(c[ks & 1], a, qf[ks][0], qf[ks][1]);
                    }
                } else {
                    // ldmatrix on the byte rows viewed as 16-bit: each register holds
                    // four consecutive dims of one token, widened to two f16 pairs;
                    // each 32-dim chunk feeds two MMAs (dims permuted alike in q).
#pragma unroll
                    for (int kc = 0; kc < D / 32; ++kc) {
                        const int ch = 2 * kc + (j >> 1);
                        uint32_t a[4], lo[4], hi[4];
                        ldsm_x4(a, ka + tok * kRow + ((ch ^ r) << 4));
#pragma unroll
                        for (int i = 0; i < 4; ++i) e4m3x4_to_f16x2x2(a[i], lo[i], hi[i]);
                        mma_16816<false>(c[0], lo, qf[2 * kc][0], qf[2 * kc][1]);
                        mma_16816<false>(c[1], hi, qf[2 * kc + 1][0], qf[2 * kc + 1][1]);
                    }
                }
            }
            {
                const bool v_lo = (smask >> g) & 1, v_hi = (smask >> (g + 8)) & 1;
                const bool h0 = 2 * t < G, h1 = 2 * t + 1 < G;
                const float sc = p.scale_log2;
                x[hs][0] = (v_lo && h0) ? (c[0][0] + c[1][0]) * sc : -INFINITY;
                x[hs][1] = (v_lo && h1) ? (c[0][1] + c[1][1]) * sc : -INFINITY;
                x[hs][2] = (v_hi && h0) ? (c[0][2] + c[1][2]) * sc : -INFINITY;
                x[hs][3] = (v_hi && h1) ? (c[0][3] + c[1][3]) * sc : -INFINITY;
            }
        }
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
        // lazy rescaling: the reference max moves only when a logit exceeds it by > 2^8
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
#pragma unroll
        for (int hs = 0; hs < SUB; ++hs) {
            if (hs > 0 && !second) continue;
            const uint32_t smask = (msk >> (16 * hs)) & 0xffffu;
            const uint32_t va = sa + hs * L::kStageBytes + L::kVOffset + warp * kHeadTile;
            const float p0 = fast_exp2(x[hs][0] - mu0), p1 = fast_exp2(x[hs][1] - mu1);
            const float p2 = fast_exp2(x[hs][2] - mu0), p3 = fast_exp2(x[hs][3] - mu1);
            l_run[0] += p0 + p2;
            l_run[1] += p1 + p3;

            // ---- P as the PV B fragment: lane needs p(token 2t|2t+1|2t+8|2t+9, head g) ----
            uint32_t bhi[2], blo[2];
            {
                const int srcA = 8 * t + (g >> 1), srcB = srcA + 4;
                const bool odd = g & 1;
                const float a0 = __shfl_sync(kFull, p0, srcA), a1 = __shfl_sync(kFull, p1, srcA);
                const float a2 = __shfl_sync(kFull, p2, srcA), a3 = __shfl_sync(kFull, p3, srcA);
                const float b0 = __shfl_sync(kFull, p0, srcB), b1 = __shfl_sync(kFull, p1, srcB);
                const float b2 = __shfl_sync(kFull, p2, srcB), b3 = __shfl_sync(kFull, p3, srcB);
                const float w[4] = {odd ? a1 : a0, odd ? b1 : b0, odd ? a3 : a2, odd ? b3 : b2};
#pragma unroll
                for (int k = 0; k < 2; ++k) {
                    bhi[k] = pack2<BF16>(w[2 * k], w[2 * k + 1]);
                    const float2 h = Cvt::to_float2(bhi[k]);
                    blo[k] = pack2<BF16>(w[2 * k] - h.x, w[2 * k + 1] - h.y);
                }
            }

            // ---- PV; my V rows past the context are zeroed first (stale slots may hold NaN) ----
            if (smask != 0xffffu) {
                uint8_t *vt = sp + hs * L::kStageBytes + L::kVOffset + warp * kHeadTile;
#pragma unroll
                for (int k = 0; k < kStageTokens * L::kHalves * 8 / 32; ++k) {
                    const int q16 = lane + 32 * k;             // 16-byte chunk of my head's V rows
                    const int half = q16 >> 7;                 // 128 chunks per half
                    const int within = q16 & 127;
                    const int row = within >> 3;
                    if (!((smask >> row) & 1))
                        *reinterpret_cast<uint4 *>(vt + half * L::kBoxBytes + within * 16) = make_uint4(0u, 0u, 0u, 0u);
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
                        ldsm_x4_trans(a, va + (ch >> 3) * L::kBoxBytes + tok * kRow + (((ch & 7) ^ r) << 4));
                        mma_16816<BF16>(acc[mt], a, bhi[0], bhi[1]);
                        mma_16816<BF16>(acc[mt], a, blo[0], blo[1]);
                    }
                } else {
                    // Transposed ldmatrix of the byte rows viewed as 16-bit gives
                    // (tokens 2t, 2t+1) x (dims 2g, 2g+1); regroup the bytes so each
                    // f16 pair is one dim over two tokens: even dims feed acc[2vc],
                    // odd dims acc[2vc+1].
#pragma unroll
                    for (int vc = 0; vc < D / 32; ++vc) {
                        const int ch = 2 * vc + (j & 1);
                        uint32_t a[4], ev[4], od[4];
                        ldsm_x4_trans(a, va + tok * kRow + ((ch ^ r) << 4));
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
        // my reads (and zeroing) of the slot are done: it may be refilled once all
        // eight consumers say so
        fence_proxy_async_smem();
        __syncwarp();
        if (lane == 0) mbar_arrive1(&empty[slot]);

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
                const int64_t orow0 = static_cast<int64_t>(m.s) * Hq + kvh * G;
#pragma unroll
                for (int h = 0; h < G; ++h)
                    store_row<D>(p.out, p.out_dtype, (orow0 + h) * D + d0, obuf + h * L::kOStride + d0);
            } else {
                const int64_t slot_id = (static_cast<int64_t>(m.s) * Hkv + kvh) * p.max_partitions + m.part;
#pragma unroll
                for (int h = 0; h < G; ++h) {
                    float *dst = p.ws_acc + (slot_id * G + h) * D + d0;
                    const float *src = obuf + h * L::kOStride + d0;
                    st_global_hint(dst, make_float4(src[0], src[1], src[2], src[3]), keep);
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
    }
}

template <int G, int KV>
cudaError_t launch_coop_t(const DecodeParams &p, const CUtensorMap &tk, const CUtensorMap &tv, int grid,
                          size_t smem, cudaStream_t stream) {
    auto kern = paged_decode_coop_kernel<128, G, KV>;
    cudaError_t e = cudaFuncSetAttribute(kern, cudaFuncAttributeMaxDynamicSharedMemorySize, static_cast<int>(smem));
    if (e != cudaSuccess) return e;
    e = launch_pdl(kern, dim3(grid), dim3(kCoopThreads), smem, stream, p, tk, tv);
    if (e != cudaSuccess) return e;
    return launch_decode_merge(p, 128, G, stream);
}

template <int G, int ES>
size_t coop_smem_for(int stages, int num_seqs) {
    using L = CoopLayout<128, G, ES>;
    return 1024 + static_cast<size_t>(stages) * (L::kSlotBytes + sizeof(CoopMeta) + 16) +
           static_cast<size_t>(kQRing) * (L::kQBytes + 16) +
           kGroupHeads * L::kOBytes + 32 * 4 + 4 * static_cast<size_t>(num_seqs) +
           4 * (static_cast<size_t>(num_seqs) + 1);
}

}  // namespace

size_t decode_coop_smem_bytes(int group, int es, int stages, int num_seqs) {
    if (es != 1 && es != 2) return 0;
    switch (group) {
        case 1: return es == 1 ? coop_smem_for<1, 1>(stages, num_seqs) : coop_smem_for<1, 2>(stages, num_seqs);
        case 2: return es == 1 ? coop_smem_for<2, 1>(stages, num_seqs) : coop_smem_for<2, 2>(stages, num_seqs);
        case 4: return es == 1 ? coop_smem_for<4, 1>(stages, num_seqs) : coop_smem_for<4, 2>(stages, num_seqs);
        case 8: return es == 1 ? coop_smem_for<8, 1>(stages, num_seqs) : coop_smem_for<8, 2>(stages, num_seqs);
        default: return 0;
    }
}

template <int G>
cudaError_t launch_coop_g(const DecodeParams &p, int kv, const CUtensorMap &tk, const CUtensorMap &tv, int grid,
                          size_t smem, cudaStream_t stream) {
    switch (kv) {
        case 0: return launch_coop_t<G, 0>(p, tk, tv, grid, smem, stream);
        case 1: return launch_coop_t<G, 1>(p, tk, tv, grid, smem, stream);
        case 2: return launch_coop_t<G, 2>(p, tk, tv, grid, smem, stream);
        case 3: return launch_coop_t<G, 3>(p, tk, tv, grid, smem, stream);
        default: return cudaErrorInvalidValue;
    }
}

cudaError_t launch_decode_coop(const DecodeParams &p, int group, int kv, const CUtensorMap &tk,
                               const CUtensorMap &tv, int grid, size_t smem, cudaStream_t stream) {
    switch (group) {
        case 1: return launch_coop_g<1>(p, kv, tk, tv, grid, smem, stream);
        case 2: return launch_coop_g<2>(p, kv, tk, tv, grid, smem, stream);
        case 4: return launch_coop_g<4>(p, kv, tk, tv, grid, smem, stream);
        case 8: return launch_coop_g<8>(p, kv, tk, tv, grid, smem, stream);
        default: return cudaErrorInvalidValue;
    }
}

}  // namespace pa
