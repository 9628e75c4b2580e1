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

#include <type_traits>

namespace pa {

namespace {

using namespace decode_common;

constexpr int kGroupHeads = 8;                    // KV heads per box and consumer warps
constexpr int kCoopThreads = (kGroupHeads + 1) * 32;
constexpr int kRow = 128;                         // bytes of one swizzled 64-element row half
constexpr int kHeadTile = kStageTokens * kRow;    // one head's 16 rows of one half: 2 KB
constexpr int kORow = 128 + 4;                    // floats per staged output row (head_dim 128, padded)

// ES = bytes per cache element (2: f16/bf16, 1: e4m3).
template <int D, int G, int ES>
struct CoopLayout {
    static constexpr bool kFp8 = ES == 1;
    // Stages per slot: two for e4m3 caches, whose 16-token stage is half the
    // bytes of a 16-bit one, so that a slot is 64 KB either way.
    static constexpr int kSub = kFp8 ? 2 : 1;
    // Query columns per consumer warp.  The MMAs' N dimension is 8 and a KV
    // head has G query heads; for 16-bit caches with G <= 2, up to 4 / G
    // sequences whose stage lies in the same physical block are served from
    // one copy of it, their query heads side by side in the columns.
    static constexpr int kCols = (!kFp8 && G <= 2) ? 4 : G;
    static constexpr int kMaxMembers = kCols / G;
    static constexpr int kHalves = D * ES / kRow;                   // 128-byte column blocks per row
    static constexpr int kBoxElems = kRow / ES;                     // elements per box row
    static constexpr int kBoxBytes = kGroupHeads * kHeadTile;      // 16 KB
    static constexpr int kKBytes = kHalves * kBoxBytes;
    static constexpr int kVOffset = kKBytes;
    static constexpr int kStageBytes = 2 * kKBytes;                 // K and V of one stage
    static constexpr int kSlotBytes = kSub * kStageBytes;
    static constexpr int kQMember = kGroupHeads * G * D * 2;        // one sequence's query rows of the group
    static constexpr int kQBytes = kMaxMembers * kQMember;          // one query-ring entry
    static constexpr int kOBytes = G * kORow * 4;                   // output staging per consumer warp
    static constexpr int kSteps = D / 16;
};

// One ring slot: one stage (two for e4m3 caches) of one tile of an item.
struct CoopMeta {
    int s;         // the item's first sequence; < 0: no more work
    int kvh0;      // first KV head of the item's group
    int part;      // partition
    int flags;     // kFirstSlot | kLastSlot | kSecondStage
    int members;   // bit m: member m's query columns read this slot's rows
    int rows;      // bit 16 * hs + r: row r of the slot's stage hs is valid
    int run;       // members | (members writing a result) << 8 | (members whose result is final) << 16
    int pad;
};
constexpr int kFirstSlot = 1;     // the item's first slot: load the queries, reset the softmax state
constexpr int kLastSlot = 2;      // the item's last slot: write the results
constexpr int kSecondStage = 4;   // e4m3: the slot's second stage belongs to the item

// The items' query rows sit in a ring of their own (kQRing entries, one per
// item), so that stage slots hold only K and V.
constexpr int kQRing = 2;

__device__ __forceinline__ void mbar_arrive1(uint64_t *bar) {
    asm volatile("mbarrier.arrive.shared::cta.b64 _, [%0];" ::"r"(smem_addr(bar)) : "memory");
}

// 16-token stages of a context (a context of 0 tokens still costs one: it
// writes a zero row).
__device__ __forceinline__ int stages_of(int ctx) {
    return ctx > 0 ? (ctx + kStageTokens - 1) / kStageTokens : 1;
}

__device__ __forceinline__ int overlap(int a0, int a1, int b0, int b1) {
    return max(0, min(a1, b1) - max(a0, b0));
}

// Runs.  Consecutive sequences whose first physical block is the same (the
// samples of one prompt sharing its blocks, "优化大模型推理：PagedAttention 如何实现
// GPU 显存高效管理", copy-on-write section) are taken together, at most
// kMaxMembers at a time.  rinfo[s] holds, for sequence s:
//   bits 0-3   its index in its run (0: the run's first sequence),
//   bits 4-7   the member count (first sequences only),
//   bits 8-31  (other members) how many 16-token stages at the start of its
//              context lie in blocks it shares with the first sequence; this
//              estimate only balances the work between CTAs, the stages a run
//              actually shares are found block by block as they are loaded.
//
// Estimated slots of item (run s, partition part), in stages: every stage of
// the longest member once, plus each other member's stages past the blocks it
// shares with the first.
__device__ __forceinline__ int item_tiles(const int *ctx_s, const int *rinfo, int s, int M, int mx, int part,
                                          int P16) {
    const int lo = part * P16, hi = lo + P16;
    int n = overlap(0, mx, lo, hi);
    for (int m = 1; m < M; ++m) {
        const int nst = stages_of(ctx_s[s + m]);
        n += overlap(min(nst, rinfo[s + m] >> 8), nst, lo, hi);
    }
    return n;
}

// Work of the run starting at s (its items summed over the KV heads), 0 for
// the other members of a run.
__device__ __forceinline__ uint32_t run_weight(const int *ctx_s, const int *rinfo, int s, int hkv) {
    const int info = rinfo[s];
    if (info & 15) return 0;
    const int M = max(1, (info >> 4) & 15);
    int mx = 0, extra = 0;
    for (int m = 0; m < M; ++m) {
        const int nst = stages_of(ctx_s[s + m]);
        mx = max(mx, nst);
        if (m > 0) extra += nst - min(nst, rinfo[s + m] >> 8);
    }
    return static_cast<uint32_t>(mx + extra) * static_cast<uint32_t>(hkv);
}

// Items (run, partition, group) in that order; an item weighs 8 x its
// estimated slots.
struct RunCursor {
    int s, M, mx, nparts, part, grp;
    uint32_t start, w;

    __device__ __forceinline__ void set_run(int s_, const int *ctx_s, const int *rinfo, int P) {
        s = s_;
        M = max(1, (rinfo[s_] >> 4) & 15);
        int cmax = 0;
        for (int m = 0; m < M; ++m) cmax = max(cmax, ctx_s[s_ + m]);
        mx = stages_of(cmax);
        nparts = cmax > 0 ? (cmax + P - 1) / P : 1;
    }
    __device__ __forceinline__ void set_part(int part_, const int *ctx_s, const int *rinfo, int P16) {
        part = part_;
        w = static_cast<uint32_t>(kGroupHeads * item_tiles(ctx_s, rinfo, s, M, mx, part_, P16));
    }
    __device__ __forceinline__ void advance(const int *ctx_s, const int *rinfo, int ngroups, int P, int B) {
        start += w;
        if (++grp < ngroups) return;
        grp = 0;
        if (part + 1 < nparts) {
            set_part(part + 1, ctx_s, rinfo, P / kStageTokens);
            return;
        }
        if (s + M < B) {
            set_run(s + M, ctx_s, rinfo, P);
            set_part(0, ctx_s, rinfo, P / kStageTokens);
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
    constexpr int KM = L::kMaxMembers;
    static_assert(SUB == 1 || KM == 1, "runs of several sequences take one stage per slot");
    using Cvt = Half2x<BF16>;
    constexpr int KS = L::kSteps;
    constexpr int MT = L::kSteps;
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
    float *obuf_all = reinterpret_cast<float *>(qbuf + kQRing * L::kQBytes);   // G rows per consumer warp
    uint8_t *misc = qbuf + kQRing * L::kQBytes + kGroupHeads * L::kOBytes;
    CoopMeta *meta = reinterpret_cast<CoopMeta *>(misc);
    misc += S * sizeof(CoopMeta);
    uint64_t *full = reinterpret_cast<uint64_t *>(misc);
    uint64_t *empty = full + S;
    uint64_t *qfull = empty + S;
    uint64_t *qempty = qfull + kQRing;
    misc += (2 * S + 2 * kQRing) * 8;
    uint32_t *warp_tot = reinterpret_cast<uint32_t *>(misc);
    misc += 32 * 4;
    int *ctx_s = reinterpret_cast<int *>(misc);
    uint32_t *prefix = reinterpret_cast<uint32_t *>(misc + 4 * B);
    int *rinfo = reinterpret_cast<int *>(misc + 4 * B + 4 * (B + 1));
    int *scratch = reinterpret_cast<int *>(prefix);   // before the prefix sum is taken

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
        int first = 0;
        if constexpr (KM > 1) first = __ldg(p.block_tables + static_cast<int64_t>(i) * p.max_blocks_per_seq);
        if (c < 0 || c > p.max_context_len) {
            if (blockIdx.x == 0) report(p.err_flag, 0x4 /* PA_FLAG_BAD_CONTEXT_LEN */);
            c = 0;
        }
        ctx_s[i] = c;
        if constexpr (KM > 1)   // the first block id, or a value no other sequence has
            scratch[i] = (c > 0 && first >= 0 && static_cast<int64_t>(first) < p.num_blocks) ? first : -1 - i;
        else
            rinfo[i] = 1 << 4;
    }
    pdl_launch_dependents();
    __syncthreads();
    // Runs of several sequences exist only if some sequence starts in the
    // block its predecessor starts in; without any, the CTA takes the plain
    // paths (one sequence per item, G query columns per consumer warp).
    bool packed = false;
    if constexpr (KM > 1) {
        bool chained = false;
        for (int i = threadIdx.x + 1; i < B; i += blockDim.x) chained = chained || scratch[i] == scratch[i - 1];
        packed = __syncthreads_or(chained) != 0;
        if (!packed) {
            for (int i = threadIdx.x; i < B; i += blockDim.x) rinfo[i] = 1 << 4;
            __syncthreads();
        } else {
            // runs: chains of equal first blocks, cut into pieces of at most KM
            if (warp == 0) {
                int carry = 0;   // the last chain start before this chunk
                for (int base = 0; base < B; base += 32) {
                    const int i = base + lane;
                    const bool head = i < B && (i == 0 || scratch[i] != scratch[i - 1]);
                    const uint32_t le = __ballot_sync(kFull, head) & (kFull >> (31 - lane));
                    const int h = le ? base + 31 - __clz(le) : carry;
                    if (i < B) rinfo[i] = (i - h) % KM;
                    carry = __shfl_sync(kFull, h, 31);
                }
            }
            __syncthreads();
            for (int i = threadIdx.x; i < B; i += blockDim.x) {
                const int mi = rinfo[i];
                int v;
                if (mi == 0) {
                    int M = 1;
                    while (M < KM && i + M < B && rinfo[i + M] == M) ++M;
                    v = M << 4;
                } else {
                    // blocks shared with the run's first sequence, by bisection
                    // (shared blocks form a prefix of the table; the first is shared)
                    const int h = i - mi;
                    const int cmin = min(ctx_s[i], ctx_s[h]);
                    const int32_t *ti = p.block_tables + static_cast<int64_t>(i) * p.max_blocks_per_seq;
                    const int32_t *th = p.block_tables + static_cast<int64_t>(h) * p.max_blocks_per_seq;
                    int lo = 1, hi = (cmin + bs - 1) / bs;
                    while (lo < hi) {
                        const int mid = (lo + hi + 1) >> 1;
                        if (__ldg(ti + mid - 1) == __ldg(th + mid - 1))
                            lo = mid;
                        else
                            hi = mid - 1;
                    }
                    v = (min(lo * bs, cmin) / kStageTokens) << 8;
                }
                scratch[i] = v;
            }
            __syncthreads();
            for (int i = threadIdx.x; i < B; i += blockDim.x) rinfo[i] |= scratch[i];
            __syncthreads();
        }
    }
    {
        // prefix[s] = work (stages x KV heads) of the runs before s
        const int nthr = blockDim.x;
        const int nw = nthr >> 5;
        const int per = (B + nthr - 1) / nthr;
        const int beg = min(B, threadIdx.x * per);
        const int end = min(B, beg + per);
        uint32_t local = 0;
        for (int i = beg; i < end; ++i) local += run_weight(ctx_s, rinfo, i, Hkv);
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
            run += run_weight(ctx_s, rinfo, i, Hkv);
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
        const int P16 = P / kStageTokens;
        RunCursor ic;
        const bool work = lo < hi;
        if (work) {
            // the run holding work unit lo (the last entry of prefix <= lo has
            // a non-zero weight, so it starts a run), then its first item
            // whose first unit is >= lo
            int a = 0, b = B;
            while (b - a > 1) {
                const int m = (a + b) >> 1;
                if (prefix[m] <= lo) a = m; else b = m;
            }
            ic.set_run(a, ctx_s, rinfo, P);
            uint32_t pstart = prefix[a];
            int part = 0;
            if (ic.M == 1) {
                // a single sequence: every partition but its last weighs Hkv x P16
                const uint32_t pw = static_cast<uint32_t>(Hkv) * static_cast<uint32_t>(P16);
                part = min(ic.nparts - 1, static_cast<int>((lo - pstart) / pw));
                pstart += static_cast<uint32_t>(part) * pw;
            } else {
                for (; part + 1 < ic.nparts; ++part) {
                    ic.set_part(part, ctx_s, rinfo, P16);
                    const uint32_t pw = ic.w * static_cast<uint32_t>(ngroups);
                    if (lo < pstart + pw) break;
                    pstart += pw;
                }
            }
            ic.set_part(part, ctx_s, rinfo, P16);
            const uint32_t grp = lo > pstart ? (lo - pstart + ic.w - 1) / ic.w : 0u;
            if (grp >= static_cast<uint32_t>(ngroups)) {   // step to the next partition or run
                ic.grp = ngroups - 1;
                ic.start = pstart + static_cast<uint32_t>(ngroups - 1) * ic.w;
                ic.advance(ctx_s, rinfo, ngroups, P, B);
            } else {
                ic.grp = static_cast<int>(grp);
                ic.start = pstart + grp * ic.w;
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
        while (ok && work && ic.start < hi) {
            const int s0 = ic.s, M = ic.M, part = ic.part;
            const int kvh0 = ic.grp * kGroupHeads;
            // per member: tokens and stages in this partition; who writes a
            // result (the partition exists for it), whose result is final (its
            // only partition), who holds its last position here
            int ntok[KM], nst[KM];
            uint32_t wmask = 0, fmask = 0, amask = 0, lmask = 0;
            int nst_item = 1;
#pragma unroll
            for (int m = 0; m < KM; ++m) {
                ntok[m] = 0;
                nst[m] = 0;
                if (m < M) {
                    const int c = ctx_s[s0 + m];
                    const int np = c > 0 ? (c + P - 1) / P : 1;
                    if (part < np) wmask |= 1u << m;
                    if (np == 1) fmask |= 1u << m;
                    if (part == np - 1) lmask |= 1u << m;
                    ntok[m] = c > part * P ? min(P, c - part * P) : 0;
                    nst[m] = (ntok[m] + kStageTokens - 1) / kStageTokens;
                    if (ntok[m] > 0) amask |= 1u << m;
                    nst_item = max(nst_item, nst[m]);
                }
            }
            // the members' block ids of this partition, one per lane (a
            // partition spans at most 32 blocks)
            const int fb = (part * P) / bs;
            int32_t bid[KM];
#pragma unroll
            for (int m = 0; m < KM; ++m) {
                bid[m] = -1;
                if (ntok[m] > 0) {
                    const int lb = (part * P + ntok[m] - 1) / bs;
                    if (lane <= lb - fb)
                        bid[m] = __ldg(p.block_tables + static_cast<int64_t>(s0 + m) * p.max_blocks_per_seq + fb +
                                       lane);
                }
            }
            {
                // the members' query rows into the next entry of the query ring
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
                    mbar_arrive_expect_tx(&qfull[qi], static_cast<uint32_t>(__popc(amask) * L::kQMember));
#pragma unroll
                    for (int m = 0; m < KM; ++m) {
                        if ((amask >> m) & 1u) {
                            const uint16_t *qsrc = static_cast<const uint16_t *>(p.q) +
                                                   (static_cast<int64_t>(s0 + m) * Hq + kvh0 * G) * D;
                            bulk_load(qbuf + qi * L::kQBytes + m * L::kQMember, qsrc, L::kQMember, &qfull[qi]);
                        }
                    }
                }
                ++items;
                __syncwarp();
            }
            const int run = M | static_cast<int>(wmask << 8) | static_cast<int>(fmask << 16);
            bool first = true;
            for (int j = 0; ok && j < nst_item; j += SUB) {
                if (!waited) {
                    bool hold = false;   // this slot holds some member's appended row
#pragma unroll
                    for (int m = 0; m < KM; ++m)
                        hold = hold || (((lmask >> m) & 1u) && nst[m] > 0 && j <= nst[m] - 1 && nst[m] - 1 < j + SUB);
                    if (hold) {
                        pdl_wait();
                        waited = true;
                    }
                }
                const int tok0 = part * P + j * kStageTokens;
                if (SUB == 1 && M == 1) {
                    // one sequence: one slot per stage
                    const int slot = take_slot();
                    if (!ok) break;
                    const int n = j < nst[0] ? min(kStageTokens, ntok[0] - j * kStageTokens) : 0;
                    const int id = __shfl_sync(kFull, bid[0], (tok0 / bs - fb) & 31);
                    const bool load = n > 0 && id >= 0 && static_cast<int64_t>(id) < p.num_blocks;
                    if (n > 0 && !load && lane == 0) report(p.err_flag, 0x2 /* PA_FLAG_BAD_BLOCK_ID */);
                    const int flags = (first ? kFirstSlot : 0) | (j + 1 >= nst_item ? kLastSlot : 0);
                    first = false;
                    uint8_t *sp = slots + static_cast<size_t>(slot) * L::kSlotBytes;
                    if (lane == 0) {
                        CoopMeta mt;
                        mt.s = s0; mt.kvh0 = kvh0; mt.part = part; mt.flags = flags;
                        mt.members = static_cast<int>(amask);
                        mt.rows = load ? static_cast<int>((1u << n) - 1u) : 0;
                        mt.run = run; mt.pad = 0;
                        meta[slot] = mt;
                        mbar_arrive_expect_tx(&full[slot], load ? 2u * L::kKBytes : 0u);
                        if (load) {
                            const int z = id * bs + (tok0 % bs);
#pragma unroll
                            for (int h = 0; h < L::kHalves; ++h) {
                                tma_load_3d(sp + h * L::kBoxBytes, &tmap_k, &full[slot], h * L::kBoxElems, z, kvh0,
                                            policy);
                                tma_load_3d(sp + L::kVOffset + h * L::kBoxBytes, &tmap_v, &full[slot],
                                            h * L::kBoxElems, z, kvh0, policy);
                            }
                        }
                    }
                    __syncwarp();
                } else if constexpr (SUB == 1 && KM > 1) {
                    // The members' rows of this stage; those in the same block
                    // (with the same row count) as the first present member
                    // share one tile, every other member gets one of its own.
                    const int col = (tok0 / bs - fb) & 31;
                    int n[KM], id[KM];
                    uint32_t pend = 0, good = 0;
#pragma unroll
                    for (int m = 0; m < KM; ++m) {
                        n[m] = j < nst[m] ? min(kStageTokens, ntok[m] - j * kStageTokens) : 0;
                        id[m] = __shfl_sync(kFull, bid[m], col);
                        if (n[m] > 0) {
                            pend |= 1u << m;
                            if (id[m] >= 0 && static_cast<int64_t>(id[m]) < p.num_blocks)
                                good |= 1u << m;
                            else if (lane == 0)
                                report(p.err_flag, 0x2 /* PA_FLAG_BAD_BLOCK_ID */);
                        }
                    }
                    do {
                        const int lead = pend ? __ffs(pend) - 1 : 0;
                        int idL = 0, nL = 0;
#pragma unroll
                        for (int m = 0; m < KM; ++m)
                            if (m == lead) {
                                idL = id[m];
                                nL = n[m];
                            }
                        uint32_t tm = 0;
#pragma unroll
                        for (int m = 0; m < KM; ++m)
                            if (((pend >> m) & 1u) && id[m] == idL && n[m] == nL) tm |= 1u << m;
                        pend &= ~tm;
                        const bool load = tm != 0 && ((good >> lead) & 1u);
                        const int flags = (first ? kFirstSlot : 0) | ((j + 1 >= nst_item && pend == 0) ? kLastSlot : 0);
                        first = false;
                        const int slot = take_slot();
                        if (!ok) break;
                        uint8_t *sp = slots + static_cast<size_t>(slot) * L::kSlotBytes;
                        if (lane == 0) {
                            CoopMeta mt;
                            mt.s = s0; mt.kvh0 = kvh0; mt.part = part; mt.flags = flags;
                            mt.members = static_cast<int>(tm);
                            mt.rows = load ? static_cast<int>((1u << nL) - 1u) : 0;
                            mt.run = run; mt.pad = 0;
                            meta[slot] = mt;
                            mbar_arrive_expect_tx(&full[slot], load ? 2u * L::kKBytes : 0u);
                            if (load) {
                                const int z = idL * bs + (tok0 % bs);
#pragma unroll
                                for (int h = 0; h < L::kHalves; ++h) {
                                    tma_load_3d(sp + h * L::kBoxBytes, &tmap_k, &full[slot], h * L::kBoxElems, z,
                                                kvh0, policy);
                                    tma_load_3d(sp + L::kVOffset + h * L::kBoxBytes, &tmap_v, &full[slot],
                                                h * L::kBoxElems, z, kvh0, policy);
                                }
                            }
                        }
                        __syncwarp();
                    } while (pend != 0);
                } else if constexpr (SUB == 2) {
                    // e4m3: SUB consecutive stages of the one member per slot
                    uint32_t rows = 0, bytes = 0;
                    int zs[SUB];
                    bool lds[SUB];
#pragma unroll
                    for (int hs = 0; hs < SUB; ++hs) {
                        const int jj = j + hs;
                        const int tk = tok0 + hs * kStageTokens;
                        const int nn = jj < nst[0] ? min(kStageTokens, ntok[0] - jj * kStageTokens) : 0;
                        const int id = __shfl_sync(kFull, bid[0], (tk / bs - fb) & 31);
                        const bool ld = nn > 0 && id >= 0 && static_cast<int64_t>(id) < p.num_blocks;
                        if (nn > 0 && !ld && lane == 0) report(p.err_flag, 0x2 /* PA_FLAG_BAD_BLOCK_ID */);
                        rows |= (ld ? ((1u << nn) - 1u) : 0u) << (16 * hs);
                        lds[hs] = ld;
                        zs[hs] = ld ? id * bs + (tk % bs) : 0;
                        bytes += ld ? 2u * L::kKBytes : 0u;
                    }
                    const int flags = (first ? kFirstSlot : 0) | (j + SUB >= nst_item ? kLastSlot : 0) |
                                      (j + 1 < nst_item ? kSecondStage : 0);
                    first = false;
                    const int slot = take_slot();
                    if (!ok) break;
                    uint8_t *sp = slots + static_cast<size_t>(slot) * L::kSlotBytes;
                    if (lane == 0) {
                        CoopMeta mt;
                        mt.s = s0; mt.kvh0 = kvh0; mt.part = part; mt.flags = flags;
                        mt.members = static_cast<int>(amask);
                        mt.rows = static_cast<int>(rows);
                        mt.run = run; mt.pad = 0;
                        meta[slot] = mt;
                        mbar_arrive_expect_tx(&full[slot], bytes);
#pragma unroll
                        for (int hs = 0; hs < SUB; ++hs) {
                            if (!lds[hs]) continue;
                            uint8_t *st = sp + hs * L::kStageBytes;
#pragma unroll
                            for (int h = 0; h < L::kHalves; ++h) {
                                tma_load_3d(st + h * L::kBoxBytes, &tmap_k, &full[slot], h * L::kBoxElems, zs[hs],
                                            kvh0, policy);
                                tma_load_3d(st + L::kVOffset + h * L::kBoxBytes, &tmap_v, &full[slot],
                                            h * L::kBoxElems, zs[hs], kvh0, policy);
                            }
                        }
                    }
                    __syncwarp();
                }
            }
            ic.advance(ctx_s, rinfo, ngroups, P, B);
        }
        // end of work: one more slot tells the consumers to stop
        if (ok) {
            const int slot = take_slot();
            if (ok && lane == 0) {
                CoopMeta mt;
                mt.s = -1; mt.kvh0 = 0; mt.part = 0; mt.flags = 0; mt.members = 0; mt.rows = 0; mt.run = 0;
                mt.pad = 0;
                meta[slot] = mt;
                mbar_arrive1(&full[slot]);
            }
        }
        if (!waited) pdl_wait();   // the CTA does not finish before the previous kernel
        __syncwarp();
        return;
    }

    // ---------------------------------------------------------------- consumers
    // Consumer warp w owns KV head kvh0 + w of every item.  Column c of its
    // MMAs' N dimension (c < 8) is query head c % G of KV head kvh0 + w in
    // member c / G of the item's run.
    const uint64_t keep = l2_policy_evict_last();
    const int g = lane >> 2, t = lane & 3;
    const uint32_t slots_sa = smem_addr(slots);
    // The loop is compiled twice: packed (columns of several sequences, G <= 2
    // with 16-bit caches) and plain (G columns of one sequence, the unused
    // columns known at compile time).
    auto consume = [&](auto packed_tag) {
        constexpr bool kPacked = decltype(packed_tag)::value;
        constexpr int NC = kPacked ? L::kCols : G;   // columns that may be in use
        uint32_t qf[KS][2];
        float acc[MT][4];
        float m_run[2], l_run[2];   // columns 2t and 2t + 1
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
            const int ncol = kPacked ? (m.run & 15) * G : G;   // columns in use: the run's members x G

            if (m.flags & kFirstSlot) {
                // new item: my query columns' B fragments from the query ring
                const int qi = static_cast<int>(citems % kQRing);
                const uint32_t qpar = (citems / kQRing) & 1u;
                ++citems;
                if (!mbar_try_wait(&qfull[qi], qpar) && !mbar_wait_bounded(&qfull[qi], qpar)) {
                    if (lane == 0) report(p.err_flag, 0x10 /* PA_FLAG_TIMEOUT */);
                    return;
                }
                const bool cv = g < ncol;
                const uint32_t *qw = reinterpret_cast<const uint32_t *>(qbuf + qi * L::kQBytes +
                                                                         min(g / G, KM - 1) * L::kQMember) +
                                     (warp * G + g % G) * (D / 2);
                if constexpr (!kFp8) {
#pragma unroll
                    for (int ks = 0; ks < KS; ++ks) {
                        qf[ks][0] = cv ? qw[(ks * 16 + 2 * t) >> 1] : 0u;
                        qf[ks][1] = cv ? qw[(ks * 16 + 2 * t + 8) >> 1] : 0u;
                    }
                } else {
                    // Dims in the order the widened K fragments arrive (see QK):
                    // step 2kc+hl takes dims 32kc + 4t + 2hl (+1) and the same + 16.
#pragma unroll
                    for (int ks = 0; ks < KS; ++ks) {
                        const int d = 32 * (ks >> 1) + 4 * t + 2 * (ks & 1);
#pragma unroll
                        for (int k = 0; k < 2; ++k) {
                            uint32_t w = cv ? qw[(d + 16 * k) >> 1] : 0u;
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

            // My columns that read this slot's rows.
            const uint32_t tm = static_cast<uint32_t>(m.members);
            const bool h0 = kPacked ? (2 * t < ncol && ((tm >> ((2 * t) / G)) & 1u)) : 2 * t < G;
            const bool h1 = kPacked ? (2 * t + 1 < ncol && ((tm >> ((2 * t + 1) / G)) & 1u)) : 2 * t + 1 < G;
            // A slot carries SUB stages (two for e4m3 caches): QK of each, one
            // softmax update over all of them, then PV of each.  The second stage
            // of an item's last slot may be absent.
            const uint32_t msk = static_cast<uint32_t>(m.rows);
            const bool second = SUB > 1 && (m.flags & kSecondStage) != 0;
            float x[SUB][4];
#pragma unroll
            for (int hs = 0; hs < SUB; ++hs) {
                if (hs > 0 && !second) {
                    x[hs][0] = x[hs][1] = x[hs][2] = x[hs][3] = -INFINITY;
                    continue;
                }
                const uint32_t ka = sa + hs * L::kStageBytes + warp * kHeadTile;
                const uint32_t smask = (msk >> (16 * hs)) & 0xffffu;
                // ---- QK^T: 16 tokens x 8 columns ----
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
            // Lazy rescaling: a sequence's reference max moves only when one of its
            // logits exceeds it by > 2^8, decided for the G columns of each member
            // together (lane t holds columns 2t and 2t + 1): with one member per
            // item, over the whole warp; with several (G <= 2), per column (G = 1)
            // or per lane (G = 2).
            bool nd0 = mx[0] > m_run[0] + 8.f, nd1 = mx[1] > m_run[1] + 8.f;
            if constexpr (!kPacked) {
                if (__any_sync(kFull, nd0 || nd1)) {
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
            } else {
                if constexpr (G == 2) nd0 = nd1 = nd0 || nd1;
                if (__any_sync(kFull, nd0 || nd1)) {
                    const bool nd[2] = {nd0, nd1};
                    float alpha[2];
#pragma unroll
                    for (int e = 0; e < 2; ++e) {
                        alpha[e] = 1.f;
                        if (nd[e]) {
                            const float m_new = fmaxf(m_run[e], mx[e]);
                            alpha[e] = (m_new == -INFINITY) ? 1.f : fast_exp2(m_run[e] - m_new);
                            m_run[e] = m_new;
                            l_run[e] *= alpha[e];
                        }
                    }
#pragma unroll
                    for (int mt = 0; mt < MT; ++mt) {
                        acc[mt][0] *= alpha[0];
                        acc[mt][1] *= alpha[1];
                        acc[mt][2] *= alpha[0];
                        acc[mt][3] *= alpha[1];
                    }
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

                // ---- P as the PV B fragment: lane needs p(token 2t|2t+1|2t+8|2t+9, column g) ----
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
            // Plain path: my reads (and zeroing) of the slot are done, it may be
            // refilled once all eight consumers say so; the results are staged
            // in my own rows of obuf.
            if constexpr (!kPacked) {
                fence_proxy_async_smem();
                __syncwarp();
                if (lane == 0) mbar_arrive1(&empty[slot]);
            }
            // ---- item end: each member's output row (or partial state), staged
            // through shared memory: obuf (plain path), or my head's tiles of
            // this slot (packed path, up to 4 rows; the slot is released after) ----
            if (m.flags & kLastSlot) {
                float lt[2] = {l_run[0], l_run[1]};
#pragma unroll
                for (int o = 4; o < 32; o <<= 1) {
                    lt[0] += __shfl_xor_sync(kFull, lt[0], o);
                    lt[1] += __shfl_xor_sync(kFull, lt[1], o);
                }
                const uint32_t wmask = (static_cast<uint32_t>(m.run) >> 8) & 0xffu;
                const uint32_t fmask = (static_cast<uint32_t>(m.run) >> 16) & 0xffu;
                // column c's row: kORow floats, in obuf or three to each of my head's 2 KB tiles
                auto orow = [&](int c) -> float * {
                    if constexpr (!kPacked) return obuf_all + (warp * G + c) * kORow;
                    const int i = c / 3;
                    return reinterpret_cast<float *>(sp + (i / (2 * L::kHalves)) * L::kStageBytes +
                                                     ((i / L::kHalves) & 1) * L::kVOffset +
                                                     (i % L::kHalves) * L::kBoxBytes + warp * kHeadTile) +
                           (c % 3) * kORow;
                };
#pragma unroll
                for (int e = 0; e < 2; ++e) {
                    const int c = 2 * t + e;
                    if (c < ncol) {
                        const bool fin = ((fmask >> min(c / G, KM - 1)) & 1u) != 0;
                        const float sc = (fin ? (lt[e] > 0.f ? 1.f / lt[e] : 0.f) : 1.f) * p.v_scale;
                        float *o = orow(c);
                        if constexpr (!kFp8) {
#pragma unroll
                            for (int mt = 0; mt < MT; ++mt) {
                                o[mt * 16 + g] = acc[mt][e] * sc;
                                o[mt * 16 + g + 8] = acc[mt][2 + e] * sc;
                            }
                        } else {
#pragma unroll
                            for (int vc = 0; vc < D / 32; ++vc) {
                                o[32 * vc + 2 * g] = acc[2 * vc][e] * sc;
                                o[32 * vc + 16 + 2 * g] = acc[2 * vc][2 + e] * sc;
                                o[32 * vc + 2 * g + 1] = acc[2 * vc + 1][e] * sc;
                                o[32 * vc + 16 + 2 * g + 1] = acc[2 * vc + 1][2 + e] * sc;
                            }
                        }
                    }
                }
                __syncwarp();
                const int d0 = lane * (D / 32);
#pragma unroll
                for (int c = 0; c < NC; ++c) {
                    const int mem = min(c / G, KM - 1), hq = c % G;
                    if (c >= ncol || !((wmask >> mem) & 1u)) continue;
                    const int64_t sm = static_cast<int64_t>(m.s) + mem;
                    const float *src = orow(c) + d0;
                    if ((fmask >> mem) & 1u) {
                        store_row<D>(p.out, p.out_dtype, (sm * Hq + kvh * G + hq) * D + d0, src);
                    } else {
                        const int64_t r = ((sm * Hkv + kvh) * p.max_partitions + m.part) * G + hq;
                        st_global_hint(p.ws_acc + r * D + d0, make_float4(src[0], src[1], src[2], src[3]), keep);
                    }
                }
                if (g == 0) {
#pragma unroll
                    for (int e = 0; e < 2; ++e) {
                        const int c = 2 * t + e;
                        const int mem = min(c / G, KM - 1), hq = c % G;
                        if (c < ncol && ((wmask >> mem) & 1u) && !((fmask >> mem) & 1u)) {
                            const int64_t sm = static_cast<int64_t>(m.s) + mem;
                            const int64_t r = ((sm * Hkv + kvh) * p.max_partitions + m.part) * G + hq;
                            st_global_hint(p.ws_ml + r * 2, make_float2(m_run[e], lt[e]), keep);
                        }
                    }
                }
                __syncwarp();   // the staged rows are read before the next item end writes them
            }
            // Packed path: my reads (and zeroing, and staging) of the slot are
            // done, it may be refilled once all eight consumers say so.
            if constexpr (kPacked) {
                fence_proxy_async_smem();
                __syncwarp();
                if (lane == 0) mbar_arrive1(&empty[slot]);
            }
        }
    };
    if constexpr (KM > 1) {
        if (packed) {
            consume(std::true_type{});
            return;
        }
    }
    consume(std::false_type{});
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
           static_cast<size_t>(kQRing) * (L::kQBytes + 16) + kGroupHeads * L::kOBytes + 32 * 4 +
           4 * static_cast<size_t>(num_seqs) * 2 + 4 * (static_cast<size_t>(num_seqs) + 1);
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
