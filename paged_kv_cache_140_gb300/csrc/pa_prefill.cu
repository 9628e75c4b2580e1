// Prefill over a paged KV cache on the fifth-generation tensor cores.
//
// After a prefix-cache hit only a sequence's tail is computed: its new query
// tokens attend, causally, to the cached prefix blocks and to themselves
// (nano-vllm walkthrough, lqnn.cn/news/170268, §3.4; the block table and
// [block, offset] cache layout of §2.2).  Query token i of a sequence with
// q_len new tokens and ctx total tokens sits at position ctx - q_len + i and
// attends positions 0 .. that position.
//
// A query tile is 128 rows of one (sequence, KV head): 128/G tokens times the
// G query heads that share the KV head.  One CTA runs two consecutive query
// tiles, X = A and B, against every 128-token K/V tile it loads, so each K/V
// byte brought into shared memory feeds 256 query rows and the two tiles'
// MMAs interleave in the tensor pipe.  Per K/V tile j and query tile X:
//   S_X = Q_X K_j^T   tcgen05.mma, Q and K tiles in shared memory (TMA,
//                     128-byte swizzle), S in tensor memory;
//   softmax           four warps per query tile, one thread per row holding
//                     the row's 128 scores in registers (one tensor-memory
//                     read, no exchange between threads); running max and
//                     sum in registers, the output rescaled only when the max
//                     grows by more than 2^8; the weights P written as 16-bit
//                     pairs over the S columns they came from, released to
//                     the MMA in four 32-key chunks so that PV starts while
//                     the later chunks are made;
//   O_X += P_X V_j    tcgen05.mma with P read from tensor memory and V
//                     (MN-major) from shared memory, O in tensor memory.
// The MMA stream runs ... PV_A(j), QK_A(j+1), PV_B(j), QK_B(j+1) ...; tcgen05
// operations of one thread execute in issue order, so QK_X(j+1) overwrites
// S_X only after PV_X(j) has read P_X from it, and when the softmax of tile
// j+1 starts, O_X already holds tile j.  bfloat16 weights carry only 8
// significant bits, so for bf16 inputs P is split into P_hi + P_lo (both
// bf16, P_lo = P - P_hi) and PV runs twice; binary16 weights are used as is.
// Full query tiles leave through shared-memory staging and TMA stores.
//
// A unit with a single query tile (a short tail) leaves the second tile's S
// columns idle; there they serve as a second S buffer, so that QK of the next
// K/V tile runs while the softmax of this one does (S no longer waits for the
// PV that reads P out of the same columns).
//
// Warp roles (11 warps, so that a sub-partition holds at most 3 and every
// thread gets 168 registers): warps 0-7 run the softmax and the epilogue
// (warp w: query tile w / 4, TMEM lanes 32 (w % 4)..); warp 8 loads the query
// tiles and the K tiles, warp 10 the V tiles (both read the block table 32
// entries at a time); warp 9 owns the tensor memory and runs the MMA issue
// loop in uniform control flow, one elected lane issuing (tcgen05 operands
// computed per lane inside a one-lane branch cost ~40 % of the MMA rate).
// Every mbarrier wait is bounded (2 s); a timeout sets PA_FLAG_TIMEOUT and the
// CTA winds down without further MMAs.
#include <math_constants.h>

#include "pa.h"
#include "pa_device.cuh"
#include "pa_prefill.h"
#include "pa_umma.cuh"

namespace pa {
namespace {

constexpr int kTile = kPrefillTile;
constexpr int kRegion = kTile * 128;     // 128 rows x 128 bytes: one swizzled operand region
constexpr uint32_t kTmemCols = 512;
// Tensor memory: S/P of query tile X at columns 128 X, O of X at 256 + 128 X
// (a single-tile unit alternates its S/P between columns 0 and 128).
// P of a 32-key chunk sits in that chunk's own S columns: 16 columns of hi
// pairs, then (bf16) 16 columns of lo pairs.
constexpr uint32_t kColS = 0, kColO = 256;
constexpr int kSoftmaxWarps = 8;        // four per query tile, one thread per row
constexpr int kWarpK = 8, kWarpMma = 9, kWarpV = 10;
constexpr int kChunks = 4;              // 32-key chunks of a row's weights, released one by one
constexpr int kMaxRing = 4;
constexpr uint64_t kWaitLimitNs = 2000000000ull;

// K and V ring depths (tiles of 128 tokens).
template <int D> struct Rings;
template <> struct Rings<128> { static constexpr int K = 2, V = 2; };
template <> struct Rings<64> { static constexpr int K = 4, V = 4; };

struct Shared {
    uint64_t q_full;
    uint64_t k_full[kMaxRing], k_empty[kMaxRing], v_full[kMaxRing], v_empty[kMaxRing];
    uint64_t s_full[2];                  // per S/P buffer (a query tile's own; alternating in a single-tile unit)
    uint64_t p_full[2][kChunks];         // [S/P buffer][32-key chunk of the row]
    uint64_t zeroed;                     // once: stale V rows of the last K/V tile zeroed
    uint64_t done;
    uint64_t pv_done;                    // single-tile unit: each PV has completed
    uint64_t staged[2];                  // per query tile: its output rows staged for the TMA store
    int ctx[kRankSeqs];                  // context lengths, for the longest-first order
    int cu[kRankSeqs + 1];               // their cu_seqlens_q entries
    int seq;                             // this CTA's sequence
    uint32_t tmem_base;
    int abort;
    int bad;
};

// Bounded wait that also gives up once another thread has aborted the CTA.
__device__ __forceinline__ bool wait_bar(uint64_t *bar, uint32_t parity, Shared &sh, int *err_flag) {
    if (mbar_try_wait(bar, parity)) return true;
    const uint64_t t0 = global_timer_ns();
    for (uint32_t i = 0;; ++i) {
        if (mbar_try_wait(bar, parity)) return true;
        if ((i & 63u) == 63u) {
            if (*reinterpret_cast<volatile int *>(&sh.abort)) return false;
            if (global_timer_ns() - t0 > kWaitLimitNs) {
                *reinterpret_cast<volatile int *>(&sh.abort) = 1;
                report(err_flag, PA_FLAG_TIMEOUT);
                return false;
            }
        }
    }
}

// Warp-uniform bounded wait: every lane waits, and the warp goes on only if
// all of them saw the phase complete (so warp-collective tensor-memory
// instructions after it are reached by the whole warp or by none of it).
__device__ __forceinline__ bool warp_wait_bar(uint64_t *bar, uint32_t parity, Shared &sh, int *err_flag) {
    return __all_sync(0xffffffffu, wait_bar(bar, parity, sh, err_flag));
}

// One lane of the (converged) warp, the same one on every call.
__device__ __forceinline__ bool elect_one() {
    uint32_t r;
    asm volatile(
        "{\n\t.reg .pred P;\n\t"
        "elect.sync _|P, 0xffffffff;\n\t"
        "selp.u32 %0, 1, 0, P;\n\t}"
        : "=r"(r));
    return r != 0;
}

__device__ __forceinline__ void mbar_arrive(uint64_t *bar) {
    asm volatile("mbarrier.arrive.shared::cta.b64 _, [%0];" ::"r"(smem_addr(bar)) : "memory");
}

// 3-D tiled TMA load without an L2 hint (K/V tiles are re-read by the other
// query tiles of the same sequence and head, which run next to this one).
__device__ __forceinline__ void tma_load_3d_plain(void *dst, const CUtensorMap *map, uint64_t *bar,
                                                  int x, int y, int z) {
    asm volatile(
        "cp.async.bulk.tensor.3d.shared::cluster.global.tile.mbarrier::complete_tx::bytes"
        " [%0], [%1, {%2, %3, %4}], [%5];" ::"r"(smem_addr(dst)),
        "l"(map), "r"(x), "r"(y), "r"(z), "r"(smem_addr(bar))
        : "memory");
}

// ------------------------------------------------ packed fp32 pair arithmetic

__device__ __forceinline__ uint64_t f2(float a, float b) {
    uint64_t r;
    asm("mov.b64 %0, {%1, %2};" : "=l"(r) : "f"(a), "f"(b));
    return r;
}
__device__ __forceinline__ float2 unf2(uint64_t r) {
    float2 v;
    asm("mov.b64 {%0, %1}, %2;" : "=f"(v.x), "=f"(v.y) : "l"(r));
    return v;
}
__device__ __forceinline__ uint64_t fma2(uint64_t a, uint64_t b, uint64_t c) {
    uint64_t r;
    asm("fma.rn.f32x2 %0, %1, %2, %3;" : "=l"(r) : "l"(a), "l"(b), "l"(c));
    return r;
}
__device__ __forceinline__ uint64_t add2(uint64_t a, uint64_t b) {
    uint64_t r;
    asm("add.rn.f32x2 %0, %1, %2;" : "=l"(r) : "l"(a), "l"(b));
    return r;
}
__device__ __forceinline__ uint64_t sub2(uint64_t a, uint64_t b) {
    uint64_t r;
    asm("sub.rn.f32x2 %0, %1, %2;" : "=l"(r) : "l"(a), "l"(b));
    return r;
}
__device__ __forceinline__ uint64_t mul2(uint64_t a, uint64_t b) {
    uint64_t r;
    asm("mul.rn.f32x2 %0, %1, %2;" : "=l"(r) : "l"(a), "l"(b));
    return r;
}
__device__ __forceinline__ float max3(float a, float b, float c) {
    float r;
    asm("max.f32 %0, %1, %2, %3;" : "=f"(r) : "f"(a), "f"(b), "f"(c));
    return r;
}

// 3-D tiled TMA store of one box from shared memory; completion is tracked
// with the bulk-group of the issuing thread.
__device__ __forceinline__ void tma_store_3d(const CUtensorMap *map, const void *src, int x, int y, int z) {
    asm volatile("cp.async.bulk.tensor.3d.global.shared::cta.bulk_group [%0, {%1, %2, %3}], [%4];" ::"l"(map),
                 "r"(x), "r"(y), "r"(z), "r"(smem_addr(src))
                 : "memory");
}
__device__ __forceinline__ void tma_store_commit_and_wait_read() {
    asm volatile("cp.async.bulk.commit_group;" ::: "memory");
    asm volatile("cp.async.bulk.wait_group.read 0;" ::: "memory");
}

// One 32-column chunk (columns col0 .. col0 + 31) of output row `row` into a
// staging tile laid out as the output tensor map's boxes: 128-byte-wide
// regions of 128 rows, 128-byte swizzle.
__device__ __forceinline__ void stage_chunk(uint8_t *stage, int out_dtype, int row, int col0, const float (&v)[32]) {
    if (out_dtype == PA_F32) {
        uint8_t *rowp = stage + (col0 / 32) * kRegion + row * 128;
#pragma unroll
        for (int u = 0; u < 8; ++u)
            *reinterpret_cast<float4 *>(rowp + ((u ^ (row & 7)) << 4)) =
                make_float4(v[4 * u], v[4 * u + 1], v[4 * u + 2], v[4 * u + 3]);
    } else {
        uint8_t *rowp = stage + (col0 / 64) * kRegion + row * 128;
        const int k0 = (col0 % 64) / 8;
#pragma unroll
        for (int u = 0; u < 4; ++u) {
            uint32_t w[4];
#pragma unroll
            for (int k = 0; k < 4; ++k)
                w[k] = out_dtype == PA_BF16 ? pack2<true>(v[8 * u + 2 * k], v[8 * u + 2 * k + 1])
                                            : pack2<false>(v[8 * u + 2 * k], v[8 * u + 2 * k + 1]);
            *reinterpret_cast<uint4 *>(rowp + (((k0 + u) ^ (row & 7)) << 4)) = make_uint4(w[0], w[1], w[2], w[3]);
        }
    }
}

// One 32-column chunk of an output row -> global memory (out_dtype).
__device__ __forceinline__ void store_chunk(void *out, int out_dtype, int64_t elem_off,
                                            const float (&v)[32]) {
    if (out_dtype == PA_F32) {
        float4 *d = reinterpret_cast<float4 *>(static_cast<float *>(out) + elem_off);
#pragma unroll
        for (int i = 0; i < 8; ++i) d[i] = make_float4(v[4 * i], v[4 * i + 1], v[4 * i + 2], v[4 * i + 3]);
    } else {
        uint4 *d = reinterpret_cast<uint4 *>(static_cast<uint16_t *>(out) + elem_off);
#pragma unroll
        for (int i = 0; i < 4; ++i) {
            uint32_t w[4];
#pragma unroll
            for (int k = 0; k < 4; ++k)
                w[k] = out_dtype == PA_BF16 ? pack2<true>(v[8 * i + 2 * k], v[8 * i + 2 * k + 1])
                                            : pack2<false>(v[8 * i + 2 * k], v[8 * i + 2 * k + 1]);
            d[i] = make_uint4(w[0], w[1], w[2], w[3]);
        }
    }
}

// A loader warp's view of the block table: 32 consecutive entries, one per
// lane, with the next 32 already requested (tiles never straddle two groups:
// 128 / bs divides 32).
struct TableWindow {
    const int32_t *table;
    int needed;          // entries that may be read: blocks holding positions <= qpos_max
    int base = -64;
    int32_t cur = -1, nxt = -1;
    __device__ int32_t fetch(int b, int lane) const {
        return (b + lane < needed) ? __ldg(table + b + lane) : -1;
    }
    // Block id of entry `entry + i` (entry = the tile's first entry, i < 32 - entry % 32).
    __device__ int32_t id_for(int entry, int i, int lane) {
        const int b = entry & ~31;
        if (b != base) {
            if (b == base + 32) {
                cur = nxt;
            } else {
                cur = fetch(b, lane);
            }
            nxt = fetch(b + 32, lane);
            base = b;
        }
        return __shfl_sync(0xffffffffu, cur, (entry & 31) + i);
    }
};

// Issue one 128-token K or V tile (8 blocks of 16 tokens for bs = 16, two
// 64-column boxes each); returns false on an abort.
template <int R>
__device__ __forceinline__ void load_tile(TableWindow &win, int t, int bs, int qpos_max, int kvh, int64_t num_blocks,
                                          uint8_t *dst, const CUtensorMap *map, uint64_t *full, int lane,
                                          Shared &sh, int *err_flag) {
    const int bpt = kTile / bs;
    const int last = min(qpos_max, t * kTile + kTile - 1);
    const int nb = (last - t * kTile) / bs + 1;
    const int32_t bid = win.id_for(t * bpt, lane < nb ? lane : 0, lane);
    const bool ok = lane < nb && bid >= 0 && static_cast<int64_t>(bid) < num_blocks;
    const unsigned okmask = __ballot_sync(0xffffffffu, ok);
    const unsigned want = (nb >= 32) ? 0xffffffffu : ((1u << nb) - 1u);
    if (lane == 0) {
        if (okmask != want) {
            report(err_flag, PA_FLAG_BAD_BLOCK_ID);
            sh.bad = 1;
        }
        mbar_arrive_expect_tx(full, static_cast<uint32_t>(__popc(okmask)) * bs * 128u * R);
    }
    __syncwarp();
    if (ok) {
#pragma unroll
        for (int r = 0; r < R; ++r)
            tma_load_3d_plain(dst + r * kRegion + lane * bs * 128, map, full, r * 64, kvh, bid * bs);
    }
}

template <int D, bool BF16>
__global__ void __launch_bounds__(kPrefillThreads, 1)
    paged_prefill_kernel(const __grid_constant__ PrefillParams p,
                         const __grid_constant__ CUtensorMap tq,
                         const __grid_constant__ CUtensorMap tk,
                         const __grid_constant__ CUtensorMap tv,
                         const __grid_constant__ CUtensorMap to) {
    constexpr int R = D / 64;               // 128-byte regions per row
    constexpr int kOp = R * kRegion;        // one 128-row operand tile
    constexpr int NK = Rings<D>::K, NV = Rings<D>::V;
    constexpr int kKSteps = D / 16;         // QK MMAs per tile (K = 16 each)
    constexpr int kPVSteps = kTile / 16;    // PV MMAs per tile and weight part
    constexpr uint32_t kIdescQK = umma::idesc_f16(BF16, kTile, kTile, false);
    constexpr uint32_t kIdescPV = umma::idesc_f16(BF16, kTile, D, true);

    __shared__ Shared sh;
    extern __shared__ uint8_t smem_raw[];
    uint8_t *base = reinterpret_cast<uint8_t *>((reinterpret_cast<uintptr_t>(smem_raw) + 1023) &
                                                ~static_cast<uintptr_t>(1023));
    uint8_t *sQ = base;                     // query tiles A, B
    uint8_t *sK = sQ + 2 * kOp;             // K ring: NK tiles
    uint8_t *sV = sK + NK * kOp;            // V ring: NV tiles

    const int warp = threadIdx.x >> 5, lane = threadIdx.x & 31;

    // ---- work unit: (sequence, pair of query tiles, KV head).  CTAs start
    // roughly in index order.  For up to kRankSeqs sequences the index runs
    // over sequences by falling context length (ties by index), then pairs
    // heaviest first, then KV heads: the longest CTAs start first and the
    // last wave holds short ones (longest-processing-time-first list
    // scheduling).  Larger batches run in sequence order, then KV head, then
    // pair, heaviest first.
    const int pairs = p.pairs_per_seq;
    const bool ranked = p.num_seqs <= kRankSeqs;
    const int per_seq = pairs * p.num_kv_heads;
    const int rank = static_cast<int>(blockIdx.x) / per_seq;
    const int rem = static_cast<int>(blockIdx.x) % per_seq;
    const int pi = pairs - 1 - (ranked ? rem / p.num_kv_heads : rem % pairs);
    const int kvh = ranked ? rem % p.num_kv_heads : rem / pairs;
    const int lg = p.log2_group;
    const int G = 1 << lg;
    const int TT = kTile >> lg;             // query tokens per tile

    int s = rank, q0, q1, ctx;
    if (ranked) {
        for (int j = threadIdx.x; j <= p.num_seqs; j += blockDim.x) {
            sh.cu[j] = __ldg(p.cu_seqlens_q + j);
            if (j < p.num_seqs) sh.ctx[j] = __ldg(p.context_lens + j);
        }
        __syncthreads();
        if (static_cast<int>(threadIdx.x) < p.num_seqs) {
            const int j = threadIdx.x, cj = sh.ctx[j];
            int above = 0;
#pragma unroll 8
            for (int i = 0; i < p.num_seqs; ++i) {
                const int ci = sh.ctx[i];
                above += (ci > cj) | ((ci == cj) & (i < j));
            }
            if (above == rank) sh.seq = j;
        }
        __syncthreads();
        s = sh.seq;
        q0 = sh.cu[s];
        q1 = sh.cu[s + 1];
        ctx = sh.ctx[s];
    } else {
        q0 = __ldg(p.cu_seqlens_q + s);
        q1 = __ldg(p.cu_seqlens_q + s + 1);
        ctx = __ldg(p.context_lens + s);
    }
    if (q0 < 0 || q1 < q0 || static_cast<int64_t>(q1) > p.num_tokens) {
        if (threadIdx.x == 0 && pi == 0 && kvh == 0) report(p.err_flag, PA_FLAG_BAD_CONTEXT_LEN);
        return;
    }
    const int ql = q1 - q0;
    if (ql > p.max_q_len && pi == 0 && kvh == 0 && threadIdx.x == 0) report(p.err_flag, PA_FLAG_BAD_CONTEXT_LEN);
    const int t0A = 2 * pi * TT;            // first token of query tile A (B follows)
    if (t0A >= ql) return;
    const bool hasB = t0A + TT < ql;

    // Softmax threads: query tile x, row `row` (token rtok, head kvh * G + row % G),
    // all 128 columns of S and all D columns of O.
    const int x = (warp >> 2) & 1, q4 = warp & 3;
    const int row = 32 * q4 + lane;
    const int rtok = row >> lg;
    const int t0x = t0A + x * TT;
    const int ntokx = max(0, min(TT, ql - t0x));
    const int64_t out_row = (static_cast<int64_t>(q0) + t0x + rtok) * p.num_heads +
                            static_cast<int64_t>(kvh) * G + (row & (G - 1));

    if (ctx < ql || static_cast<int64_t>(ctx) > static_cast<int64_t>(p.max_blocks_per_seq) * p.block_size) {
        if (threadIdx.x == 0 && pi == 0 && kvh == 0) report(p.err_flag, PA_FLAG_BAD_CONTEXT_LEN);
        if (warp < kSoftmaxWarps && rtok < ntokx) {
            float z[32];
#pragma unroll
            for (int i = 0; i < 32; ++i) z[i] = 0.f;
#pragma unroll
            for (int c = 0; c < D / 32; ++c) store_chunk(p.out, p.out_dtype, out_row * D + c * 32, z);
        }
        return;
    }
    const int qstartA = ctx - ql + t0A;     // position of tile A's first query token
    const int nA = (qstartA + min(TT, ql - t0A) - 1) / kTile + 1;
    const int qpos_max = qstartA + (hasB ? TT + min(TT, ql - t0A - TT) : min(TT, ql - t0A)) - 1;
    const int nB = hasB ? qpos_max / kTile + 1 : 0;
    const int n_tiles = hasB ? nB : nA;     // K/V tiles loaded (nB >= nA)
    // The last K/V tile reaches past the last attended position: its stale or
    // unloaded V rows are zeroed (by the query tile that reaches furthest)
    // before any PV reads it, so that 0-weights cannot meet NaNs.
    const bool zero_tail = n_tiles * kTile - 1 > qpos_max;
    // A unit with a single query tile over two or more K/V tiles uses the
    // second tile's S columns as a second S buffer: QK of K/V tile j + 1 runs
    // while the softmax of tile j does, instead of after PV(j) (which reads P(j)
    // from the columns S(j) came in).  The output is then rescaled only after
    // the previous PV has completed.
    const bool solo = !hasB && nA >= 2;

    if (threadIdx.x == 0) {
        mbar_init(&sh.q_full, 1);
        for (int i = 0; i < kMaxRing; ++i) {
            mbar_init(&sh.k_full[i], 1);
            mbar_init(&sh.k_empty[i], 1);
            mbar_init(&sh.v_full[i], 1);
            mbar_init(&sh.v_empty[i], 1);
        }
        for (int i = 0; i < 2; ++i) {
            mbar_init(&sh.s_full[i], 1);
            for (int c = 0; c < kChunks; ++c) mbar_init(&sh.p_full[i][c], 128);
        }
        mbar_init(&sh.done, 1);
        mbar_init(&sh.pv_done, 1);
        mbar_init(&sh.zeroed, 128);
        mbar_init(&sh.staged[0], 128);
        mbar_init(&sh.staged[1], 128);
        sh.abort = 0;
        sh.bad = 0;
        fence_barrier_init();
    }
    if (warp == kWarpMma) {
        umma::tmem_alloc(smem_addr(&sh.tmem_base), kTmemCols);
        umma::tmem_relinquish();
    }
    umma::fence_before_sync();
    __syncthreads();
    umma::fence_after_sync();
    const uint32_t tmem = sh.tmem_base;

    if (warp == kWarpK || warp == kWarpV) {
        // ---------------------------------------------------- TMA loaders
        const bool is_k = warp == kWarpK;
        const CUtensorMap *map = is_k ? &tk : &tv;
        const int NR = is_k ? NK : NV;
        uint64_t *full = is_k ? sh.k_full : sh.v_full;
        uint64_t *empty = is_k ? sh.k_empty : sh.v_empty;
        uint8_t *ring = is_k ? sK : sV;
        if (lane == 0) {
            prefetch_tensormap(map);
            if (is_k) {
                prefetch_tensormap(&tq);
                mbar_arrive_expect_tx(&sh.q_full, kOp * (hasB ? 2 : 1));
#pragma unroll
                for (int r = 0; r < R; ++r) {
                    tma_load_3d_plain(sQ + r * kRegion, &tq, &sh.q_full, r * 64, kvh * G, q0 + t0A);
                    if (hasB)
                        tma_load_3d_plain(sQ + kOp + r * kRegion, &tq, &sh.q_full, r * 64, kvh * G, q0 + t0A + TT);
                }
            }
        }
        TableWindow win{p.block_tables + static_cast<int64_t>(s) * p.max_blocks_per_seq,
                        qpos_max / p.block_size + 1};
        int issued = 0;
        for (int t = 0; t < n_tiles; ++t) {
            const int st = t % NR;
            if (t >= NR && !warp_wait_bar(&empty[st], ((t / NR) - 1) & 1, sh, p.err_flag)) break;
            load_tile<R>(win, t, p.block_size, qpos_max, kvh, p.num_blocks, ring + st * kOp, map, &full[st], lane,
                         sh, p.err_flag);
            ++issued;
        }
        // On an abort, let the copies still in flight land before the CTA exits.
        if (lane == 0 && sh.abort) {
            for (int t = max(0, issued - NR); t < issued; ++t)
                mbar_wait_bounded(&full[t % NR], (t / NR) & 1, kWaitLimitNs);
            if (is_k) mbar_wait_bounded(&sh.q_full, 0, kWaitLimitNs);
        }
    } else if (warp == kWarpMma) {
        // ------------------------------------------------------- MMA issuer
        // The whole warp runs this loop in uniform control flow, so the
        // descriptors (ring bases built once, k-step offsets as immediates)
        // stay warp-uniform; one elected lane issues each MMA and commit.
        const bool leader = elect_one();
        const uint64_t qd0 = umma::desc_sw128(smem_addr(sQ), 16, 1024);
        const uint64_t kd0 = umma::desc_sw128(smem_addr(sK), 16, 1024);
        const uint64_t vd0 = umma::desc_sw128(smem_addr(sV), kRegion, 1024);
        constexpr uint32_t kOpDesc = kOp >> 4;
        bool ok = warp_wait_bar(&sh.q_full, 0, sh, p.err_flag);
        if (!solo) {
            const int nx[2] = {nA, nB};
            int k_ready = -1;                      // last K tile known to have landed
            auto qk = [&](int xx, int t) -> bool {      // S_xx = Q_xx K_t^T
                const int kst = t % NK;
                if (k_ready < t) {
                    if (!warp_wait_bar(&sh.k_full[kst], (t / NK) & 1, sh, p.err_flag)) return false;
                    k_ready = t;
                }
                umma::fence_after_sync();
                const uint64_t qd = qd0 + static_cast<uint32_t>(xx) * kOpDesc;
                const uint64_t kd = kd0 + static_cast<uint32_t>(kst) * kOpDesc;
                const uint32_t ts = tmem + kColS + 128u * xx;
                if (leader) {
    #pragma unroll
                    for (int k = 0; k < kKSteps; ++k) {
                        constexpr uint32_t kRegDesc = kRegion >> 4;
                        const uint32_t off = (k >> 2) * kRegDesc + (k & 3) * 2;
                        umma::mma_ss(ts, qd + off, kd + off, kIdescQK, k > 0 ? 1u : 0u);
                    }
                    umma::commit(smem_addr(&sh.s_full[xx]));
                }
                __syncwarp();
                return true;
            };
            if (ok) ok = qk(0, 0);
            if (ok && hasB) ok = qk(1, 0);
            if (ok && leader) umma::commit(smem_addr(&sh.k_empty[0]));
            __syncwarp();
            for (int j = 0; ok && j < n_tiles; ++j) {
                const int vst = j % NV;
                if (zero_tail && j == n_tiles - 1 && !warp_wait_bar(&sh.zeroed, 0, sh, p.err_flag)) {
                    ok = false;
                    break;
                }
                if (!warp_wait_bar(&sh.v_full[vst], (j / NV) & 1, sh, p.err_flag)) { ok = false; break; }
                const uint64_t vd = vd0 + static_cast<uint32_t>(vst) * kOpDesc;
                for (int xx = 0; ok && xx < 2; ++xx) {
                    if (j >= nx[xx]) continue;
                    const uint32_t tP = tmem + kColS + 128u * xx;
                    const uint32_t tO = tmem + kColO + 128u * xx;
                    const uint32_t acc0 = j > 0 ? 1u : 0u;
                    // Each softmax thread writes its row's weights in four 32-key
                    // chunks; chunk c feeds k-steps 2c and 2c + 1, so PV starts
                    // while the later chunks are still being made.
    #pragma unroll
                    for (int c = 0; c < kChunks; ++c) {
                        if (!warp_wait_bar(&sh.p_full[xx][c], j & 1, sh, p.err_flag)) { ok = false; break; }
                        umma::fence_after_sync();
                        if (leader) {
    #pragma unroll
                            for (int kk = 0; kk < kPVSteps / kChunks; ++kk) {
                                const int k = (kPVSteps / kChunks) * c + kk;
                                umma::mma_ts(tO, tP + 32u * (k >> 1) + 8u * (k & 1),
                                             vd + static_cast<uint32_t>(k * (2048 >> 4)), kIdescPV,
                                             (c > 0 || kk > 0) ? 1u : acc0);
                                if constexpr (BF16)
                                    umma::mma_ts(tO, tP + 32u * (k >> 1) + 8u * (k & 1) + 16u,
                                                 vd + static_cast<uint32_t>(k * (2048 >> 4)), kIdescPV, 1u);
                            }
                        }
                        __syncwarp();
                    }
                    if (!ok) break;
                    if (j + 1 < nx[xx]) ok = qk(xx, j + 1);
                }
                if (!ok) break;
                if (leader) {
                    umma::commit(smem_addr(&sh.v_empty[vst]));
                    if (j + 1 < n_tiles) umma::commit(smem_addr(&sh.k_empty[(j + 1) % NK]));
                }
                __syncwarp();
            }
        } else {
            // S(t) goes to buffer t & 1; QK(t + 2) follows PV(t), which has read
            // P(t) from the same columns (tcgen05 operations of one thread run in
            // issue order).
            auto qk_solo = [&](int t) -> bool {
                const int kst = t % NK, b = t & 1;
                if (!warp_wait_bar(&sh.k_full[kst], (t / NK) & 1, sh, p.err_flag)) return false;
                umma::fence_after_sync();
                const uint64_t kd = kd0 + static_cast<uint32_t>(kst) * kOpDesc;
                const uint32_t ts = tmem + kColS + 128u * b;
                if (leader) {
#pragma unroll
                    for (int k = 0; k < kKSteps; ++k) {
                        constexpr uint32_t kRegDesc = kRegion >> 4;
                        const uint32_t off = (k >> 2) * kRegDesc + (k & 3) * 2;
                        umma::mma_ss(ts, qd0 + off, kd + off, kIdescQK, k > 0 ? 1u : 0u);
                    }
                    umma::commit(smem_addr(&sh.s_full[b]));
                    umma::commit(smem_addr(&sh.k_empty[kst]));
                }
                __syncwarp();
                return true;
            };
            if (ok) ok = qk_solo(0);
            if (ok) ok = qk_solo(1);
            const uint32_t tO = tmem + kColO;
            for (int j = 0; ok && j < nA; ++j) {
                const int vst = j % NV, b = j & 1;
                if (zero_tail && j == nA - 1 && !warp_wait_bar(&sh.zeroed, 0, sh, p.err_flag)) {
                    ok = false;
                    break;
                }
                if (!warp_wait_bar(&sh.v_full[vst], (j / NV) & 1, sh, p.err_flag)) { ok = false; break; }
                const uint64_t vd = vd0 + static_cast<uint32_t>(vst) * kOpDesc;
                const uint32_t tP = tmem + kColS + 128u * b;
                const uint32_t acc0 = j > 0 ? 1u : 0u;
#pragma unroll
                for (int c = 0; c < kChunks; ++c) {
                    if (!warp_wait_bar(&sh.p_full[b][c], (j >> 1) & 1, sh, p.err_flag)) { ok = false; break; }
                    umma::fence_after_sync();
                    if (leader) {
#pragma unroll
                        for (int kk = 0; kk < kPVSteps / kChunks; ++kk) {
                            const int k = (kPVSteps / kChunks) * c + kk;
                            umma::mma_ts(tO, tP + 32u * (k >> 1) + 8u * (k & 1),
                                         vd + static_cast<uint32_t>(k * (2048 >> 4)), kIdescPV,
                                         (c > 0 || kk > 0) ? 1u : acc0);
                            if constexpr (BF16)
                                umma::mma_ts(tO, tP + 32u * (k >> 1) + 8u * (k & 1) + 16u,
                                             vd + static_cast<uint32_t>(k * (2048 >> 4)), kIdescPV, 1u);
                        }
                    }
                    __syncwarp();
                }
                if (!ok) break;
                if (leader) {
                    umma::commit(smem_addr(&sh.pv_done));
                    umma::commit(smem_addr(&sh.v_empty[vst]));
                }
                __syncwarp();
                if (j + 2 < nA) ok = qk_solo(j + 2);
            }
        }
        if (leader) {
            umma::commit(smem_addr(&sh.done));
            mbar_wait_bounded(&sh.done, 0, kWaitLimitNs);
        }
        __syncwarp();
    } else if (warp < kSoftmaxWarps && (x == 0 || hasB)) {
        // ------------------------------------------- softmax and epilogue
        const int nx = x == 0 ? nA : nB;
        const int qpos = rtok < ntokx ? qstartA + x * TT + rtok : -1;
        const uint32_t lane_off = static_cast<uint32_t>(32 * q4) << 16;
        const uint32_t tS0 = tmem + kColS + lane_off;
        const uint32_t tO = tmem + kColO + 128u * x + lane_off;
        // The tile that reaches furthest zeroes the stale V rows of the last K/V tile.
        const bool zeroer = zero_tail && x == (hasB ? 1 : 0);
        const float sl = p.scale_log2;
        const uint64_t sl2 = f2(sl, sl);
        float m_run = -CUDART_INF_F;
        float l_run = 0.f;
        bool ok = true;
        for (int j = 0; j < nx; ++j) {
            // S buffer: the tile's own, or (single-tile unit) alternating
            const int b = solo ? (j & 1) : x;
            if (!warp_wait_bar(&sh.s_full[b], solo ? (j >> 1) & 1 : j & 1, sh, p.err_flag)) { ok = false; break; }
            umma::fence_after_sync();
            const uint32_t tS = tS0 + 128u * b;
            const int lim = qpos - j * kTile;   // columns c <= lim are attended
            const bool masked = !__all_sync(0xffffffffu, lim >= kTile - 1);
            // the whole S row in registers: four loads in flight, one wait
            uint32_t v[kTile];
#pragma unroll
            for (int c = 0; c < kChunks; ++c)
                umma::ld_32x32b_x32(tS + 32 * c, *reinterpret_cast<uint32_t(*)[32]>(v + 32 * c));
            umma::wait_ld();
            if (masked) {
#pragma unroll
                for (int i = 0; i < kTile; ++i)
                    if (i > lim) v[i] = 0xff800000u;     // -inf
            }
            float a[8];
#pragma unroll
            for (int k = 0; k < 8; ++k) a[k] = fmaxf(__uint_as_float(v[k]), __uint_as_float(v[k + 8]));
#pragma unroll
            for (int i = 1; i < kTile / 16; ++i)
#pragma unroll
                for (int k = 0; k < 8; ++k)
                    a[k] = max3(a[k], __uint_as_float(v[16 * i + k]), __uint_as_float(v[16 * i + 8 + k]));
            const float mx = max3(max3(a[0], a[1], a[2]), max3(a[3], a[4], a[5]), fmaxf(a[6], a[7]));
            const float x_tile = mx * sl;
            const bool need = x_tile > m_run + 8.f;
            if (__any_sync(0xffffffffu, need)) {
                // O_x already holds tile j-1: PV(j-1) preceded QK(j) in the MMA stream.
                const float f = need ? fast_exp2(m_run - x_tile) : 1.f;
                if (j > 0) {
                    // single-tile unit: PV(j-1) may still be running
                    if (solo && !warp_wait_bar(&sh.pv_done, (j - 1) & 1, sh, p.err_flag)) { ok = false; break; }
                    umma::fence_after_sync();
                    const uint64_t f2x = f2(f, f);
                    // 16 columns at a time: the S row stays live in registers meanwhile
#pragma unroll
                    for (int c = 0; c < D / 16; ++c) {
                        uint32_t o[16];
                        umma::ld_32x32b_x16(tO + 16 * c, o);
                        umma::wait_ld();
#pragma unroll
                        for (int i = 0; i < 8; ++i) {
                            const float2 w = unf2(mul2(f2(__uint_as_float(o[2 * i]), __uint_as_float(o[2 * i + 1])), f2x));
                            o[2 * i] = __float_as_uint(w.x);
                            o[2 * i + 1] = __float_as_uint(w.y);
                        }
                        umma::st_32x32b_x16(tO + 16 * c, o);
                    }
                }
                if (need) {
                    l_run *= f;
                    m_run = x_tile;
                }
            }
            if (zeroer && j == nx - 1) {
                const int vst = j % NV;
                if (!warp_wait_bar(&sh.v_full[vst], (j / NV) & 1, sh, p.err_flag)) { ok = false; break; }
                if (j * kTile + row > qpos_max) {
#pragma unroll
                    for (int r = 0; r < R; ++r) {
                        uint4 *d = reinterpret_cast<uint4 *>(sV + vst * kOp + r * kRegion + row * 128);
#pragma unroll
                        for (int i = 0; i < 8; ++i) d[i] = make_uint4(0u, 0u, 0u, 0u);
                    }
                }
                fence_proxy_async_smem();
                mbar_arrive(&sh.zeroed);
            }
            // weights p = 2^(s * scale_log2 - m) as 16-bit pairs, each 32-key
            // chunk written over its own S columns and released on its own
            const float mref = m_run == -CUDART_INF_F ? 0.f : m_run;
            const uint64_t nm2 = f2(-mref, -mref);
            uint64_t acc0 = f2(0.f, 0.f), acc1 = f2(0.f, 0.f);
#pragma unroll
            for (int c = 0; c < kChunks; ++c) {
                uint32_t hi[16];
                [[maybe_unused]] uint32_t lo[16];
#pragma unroll
                for (int i = 0; i < 16; ++i) {
                    const float2 xv = unf2(fma2(f2(__uint_as_float(v[32 * c + 2 * i]), __uint_as_float(v[32 * c + 2 * i + 1])),
                                                sl2, nm2));
                    const float p0 = fast_exp2(xv.x), p1 = fast_exp2(xv.y);
                    hi[i] = pack2<BF16>(p0, p1);
                    const float2 hv = Half2x<BF16>::to_float2(hi[i]);
                    if constexpr (BF16) {
                        const float2 lv = unf2(sub2(f2(p0, p1), f2(hv.x, hv.y)));
                        lo[i] = pack2<true>(lv.x, lv.y);
                        if (i & 1) acc1 = add2(acc1, f2(p0, p1)); else acc0 = add2(acc0, f2(p0, p1));
                    } else {
                        if (i & 1) acc1 = add2(acc1, f2(hv.x, hv.y)); else acc0 = add2(acc0, f2(hv.x, hv.y));
                    }
                }
                umma::st_32x32b_x16(tS + 32 * c, hi);
                if constexpr (BF16) umma::st_32x32b_x16(tS + 32 * c + 16, lo);
                umma::wait_st();
                umma::fence_before_sync();
                mbar_arrive(&sh.p_full[b][c]);
            }
            const float2 acc = unf2(add2(acc0, acc1));
            l_run += acc.x + acc.y;
        }
        // `done` completes once every MMA of the CTA (the last PV included) has.
        if (ok && warp_wait_bar(&sh.done, 0, sh, p.err_flag)) {
            umma::fence_after_sync();
            const bool zero = *reinterpret_cast<volatile int *>(&sh.bad) != 0;
            const float inv = (l_run > 0.f && !zero) ? 1.f / l_run : 0.f;
            // A full query tile (all its rows belong to this sequence) is staged in
            // shared memory, idle now that every MMA is done (K ring for tile A,
            // V ring for tile B), and written by TMA stores; a partial tile is
            // written row by row so that no other sequence's rows are touched.
            const bool full_tile = ntokx == TT;
            uint8_t *stage = x == 0 ? sK : sV;
#pragma unroll
            for (int c = 0; c < D / 32; ++c) {
                uint32_t o[32];
                umma::ld_32x32b_x32(tO + 32 * c, o);
                umma::wait_ld();
                float ov[32];
#pragma unroll
                for (int i = 0; i < 32; ++i) ov[i] = zero ? 0.f : __uint_as_float(o[i]) * inv;
                if (full_tile)
                    stage_chunk(stage, p.out_dtype, row, 32 * c, ov);
                else if (qpos >= 0)
                    store_chunk(p.out, p.out_dtype, out_row * D + c * 32, ov);
            }
            if (full_tile) {
                fence_proxy_async_smem();
                mbar_arrive(&sh.staged[x]);
                if (warp == 4 * x && lane == 0 && mbar_wait_bounded(&sh.staged[x], 0, kWaitLimitNs)) {
                    const int es = p.out_dtype == PA_F32 ? 4 : 2;
                    const int regions = D * es / 128;
                    for (int r = 0; r < regions; ++r)
                        tma_store_3d(&to, stage + r * kRegion, r * (128 / es), kvh * G, q0 + t0x);
                    tma_store_commit_and_wait_read();
                }
            }
        }
    }

    umma::fence_before_sync();
    __syncthreads();
    if (warp == kWarpMma) {
        umma::fence_after_sync();
        umma::tmem_dealloc(tmem, kTmemCols);
    }
}

template <int D, bool BF16>
cudaError_t launch_t(const PrefillParams &p, const CUtensorMap &tq, const CUtensorMap &tk, const CUtensorMap &tv,
                     const CUtensorMap &to, size_t smem, cudaStream_t stream) {
    auto kern = paged_prefill_kernel<D, BF16>;
    cudaError_t e = cudaFuncSetAttribute(kern, cudaFuncAttributeMaxDynamicSharedMemorySize,
                                         static_cast<int>(smem));
    if (e != cudaSuccess) return e;
    const int64_t grid = static_cast<int64_t>(p.num_seqs) * p.num_kv_heads * p.pairs_per_seq;
    kern<<<static_cast<unsigned>(grid), kPrefillThreads, smem, stream>>>(p, tq, tk, tv, to);
    return cudaGetLastError();
}

}  // namespace

size_t prefill_smem_bytes(int head_dim) {
    const size_t op = static_cast<size_t>(head_dim / 64) * kRegion;
    const int rings = head_dim == 128 ? Rings<128>::K + Rings<128>::V : Rings<64>::K + Rings<64>::V;
    return 1024 + op * (2 + rings);
}

cudaError_t launch_prefill(const PrefillParams &p, int head_dim, bool bf16, const CUtensorMap &tq,
                           const CUtensorMap &tk, const CUtensorMap &tv, const CUtensorMap &to, size_t smem,
                           cudaStream_t stream) {
    if (head_dim == 128)
        return bf16 ? launch_t<128, true>(p, tq, tk, tv, to, smem, stream)
                    : launch_t<128, false>(p, tq, tk, tv, to, smem, stream);
    if (head_dim == 64)
        return bf16 ? launch_t<64, true>(p, tq, tk, tv, to, smem, stream)
                    : launch_t<64, false>(p, tq, tk, tv, to, smem, stream);
    return cudaErrorInvalidValue;
}

}  // namespace pa
