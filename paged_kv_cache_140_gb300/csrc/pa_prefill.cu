// Prefill over a paged KV cache on the fifth-generation tensor cores.
//
// After a prefix-cache hit only a sequence's tail is computed: its new query
// tokens attend, causally, to the cached prefix blocks and to themselves
// ("SGLang / nano-vllm ... PagedAttention" walkthrough, §3.4; the block table
// and [block, offset] cache layout of §2.2).  Query token i of a sequence
// with q_len new tokens and ctx total tokens sits at position
// ctx - q_len + i and attends positions 0 .. that position.
//
// One CTA computes 128 query rows of one (sequence, KV head): 128/G tokens
// times the G query heads that share the KV head, so every K/V tile read is
// used by all of them.  Per 128-token KV tile:
//   S = Q K^T   tcgen05.mma, Q and K tiles in shared memory (TMA, 128-byte
//               swizzle), S in tensor memory (double-buffered);
//   softmax     four warps, one query row per thread, read S from tensor
//               memory, keep the running max / sum in registers (rescaling
//               the output only when the max grows by more than 2^8) and
//               write the weights P back over S as 16-bit pairs;
//   O += P V    tcgen05.mma with P read from tensor memory and V (MN-major)
//               from shared memory, O accumulated in tensor memory.
// bfloat16 weights carry only 8 significant bits, so for bf16 inputs P is
// split into P_hi + P_lo (both bf16, P_lo = P - P_hi) and PV runs twice;
// binary16 weights (11 bits) are used directly.
//
// Warp roles: warps 0-3 softmax + epilogue (warp w owns TMEM lanes 32w..),
// warp 4 issues the TMA loads (block ids read through the block table), warp
// 5 owns the tensor memory and one of its lanes issues every MMA.  Every
// mbarrier wait is bounded (2 s); a timeout sets PA_FLAG_TIMEOUT and the CTA
// winds down without further MMAs.
#include <math_constants.h>

#include "pa.h"
#include "pa_device.cuh"
#include "pa_prefill.h"
#include "pa_umma.cuh"

namespace pa {
namespace {

constexpr int kTile = kPrefillTile;
constexpr int kRegion = kTile * 128;     // 128 rows x 128 bytes: one swizzled operand region
constexpr uint32_t kTmemCols = 512;      // S0 [0,128), S1 [128,256), O [256, 256 + D)
constexpr int kMaxStages = 4;
constexpr uint64_t kWaitLimitNs = 2000000000ull;

struct Shared {
    uint64_t q_full;
    uint64_t k_full[kMaxStages], v_full[kMaxStages], kv_empty[kMaxStages];
    uint64_t s_full[2], p_full[2], pv_done[2];
    uint64_t done;
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

__device__ __forceinline__ void mbar_arrive(uint64_t *bar) {
    asm volatile("mbarrier.arrive.shared::cta.b64 _, [%0];" ::"r"(smem_addr(bar)) : "memory");
}

// Warp-uniform bounded wait: every lane waits, and the warp goes on only if
// all of them saw the phase complete (so warp-collective tensor-memory
// instructions after it are reached by the whole warp or by none of it).
__device__ __forceinline__ bool warp_wait_bar(uint64_t *bar, uint32_t parity, Shared &sh, int *err_flag) {
    return __all_sync(0xffffffffu, wait_bar(bar, parity, sh, err_flag));
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

__device__ __forceinline__ void st_32x32b_x32(uint32_t taddr, const uint32_t (&r)[32]) {
    umma::st_32x32b_x16(taddr, r);
    umma::st_32x32b_x16(taddr + 16, r + 16);
}

template <bool BF16>
__device__ __forceinline__ uint32_t pack_pair(float lo, float hi) {
    return pack2<BF16>(lo, hi);
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

template <int D, bool BF16>
__global__ void __launch_bounds__(kPrefillThreads, 1)
    paged_prefill_kernel(const __grid_constant__ PrefillParams p,
                         const __grid_constant__ CUtensorMap tq,
                         const __grid_constant__ CUtensorMap tk,
                         const __grid_constant__ CUtensorMap tv) {
    constexpr int R = D / 64;               // 128-byte regions per row
    constexpr int kOp = R * kRegion;        // one 128-row operand tile
    constexpr int kKSteps = D / 16;         // QK MMAs per tile (K = 16 each)
    constexpr int kPVSteps = kTile / 16;    // PV MMAs per tile and weight part
    constexpr uint32_t kIdescQK = umma::idesc_f16(BF16, kTile, kTile, false);
    constexpr uint32_t kIdescPV = umma::idesc_f16(BF16, kTile, D, true);

    __shared__ Shared sh;
    extern __shared__ uint8_t smem_raw[];
    uint8_t *base = reinterpret_cast<uint8_t *>((reinterpret_cast<uintptr_t>(smem_raw) + 1023) &
                                                ~static_cast<uintptr_t>(1023));
    uint8_t *sQ = base;
    uint8_t *sKV = base + kOp;              // stage st: K at sKV + 2 st kOp, V right after

    const int warp = threadIdx.x >> 5, lane = threadIdx.x & 31;
    const int NS = p.stages;

    // ---- work unit: (sequence, KV head, query tile), heaviest tiles first
    const int tiles = p.tiles_per_seq;
    const int qt = tiles - 1 - static_cast<int>(blockIdx.x % tiles);
    const int sk = static_cast<int>(blockIdx.x / tiles);
    const int kvh = sk % p.num_kv_heads;
    const int s = sk / p.num_kv_heads;
    const int lg = p.log2_group;
    const int G = 1 << lg;
    const int TT = kTile >> lg;             // query tokens per tile

    const int q0 = __ldg(p.cu_seqlens_q + s), q1 = __ldg(p.cu_seqlens_q + s + 1);
    if (q0 < 0 || q1 < q0 || static_cast<int64_t>(q1) > p.num_tokens) {
        if (threadIdx.x == 0 && qt == 0 && kvh == 0) report(p.err_flag, PA_FLAG_BAD_CONTEXT_LEN);
        return;
    }
    const int ql = q1 - q0;
    if (ql > tiles * TT && qt == 0 && kvh == 0 && threadIdx.x == 0) report(p.err_flag, PA_FLAG_BAD_CONTEXT_LEN);
    const int t0 = qt * TT;
    if (t0 >= ql) return;                   // no query tokens in this tile
    const int ntok = min(TT, ql - t0);
    const int ctx = __ldg(p.context_lens + s);
    const int row = threadIdx.x;            // softmax threads: query row
    const int rtok = row >> lg;
    // Output row of softmax thread `row` (token rtok, head kvh * G + row % G).
    const int64_t out_row = (static_cast<int64_t>(q0) + t0 + rtok) * p.num_heads +
                            static_cast<int64_t>(kvh) * G + (row & (G - 1));

    if (ctx < ql || static_cast<int64_t>(ctx) > static_cast<int64_t>(p.max_blocks_per_seq) * p.block_size) {
        if (threadIdx.x == 0 && qt == 0 && kvh == 0) report(p.err_flag, PA_FLAG_BAD_CONTEXT_LEN);
        if (row < kTile && rtok < ntok) {
            float z[32];
#pragma unroll
            for (int i = 0; i < 32; ++i) z[i] = 0.f;
#pragma unroll
            for (int c = 0; c < D / 32; ++c)
                store_chunk(p.out, p.out_dtype, out_row * D + c * 32, z);
        }
        return;
    }
    const int qstart = ctx - ql + t0;       // position of the tile's first query token
    const int qpos_max = qstart + ntok - 1;
    const int n_tiles = qpos_max / kTile + 1;

    if (threadIdx.x == 0) {
        mbar_init(&sh.q_full, 1);
        for (int i = 0; i < kMaxStages; ++i) {
            mbar_init(&sh.k_full[i], 1);
            mbar_init(&sh.v_full[i], 1);
            mbar_init(&sh.kv_empty[i], 1);
        }
        for (int i = 0; i < 2; ++i) {
            mbar_init(&sh.s_full[i], 1);
            mbar_init(&sh.p_full[i], kTile);
            mbar_init(&sh.pv_done[i], 1);
        }
        mbar_init(&sh.done, 1);
        sh.abort = 0;
        sh.bad = 0;
        fence_barrier_init();
    }
    if (warp == 5) {
        umma::tmem_alloc(smem_addr(&sh.tmem_base), kTmemCols);
        umma::tmem_relinquish();
    }
    umma::fence_before_sync();
    __syncthreads();
    umma::fence_after_sync();
    const uint32_t tmem = sh.tmem_base;
    const uint32_t tO = tmem + 256;

    if (warp == 4) {
        // ------------------------------------------------------ TMA producer
        const int bs = p.block_size;
        const int bpt = kTile / bs;
        const int32_t *table = p.block_tables + static_cast<int64_t>(s) * p.max_blocks_per_seq;
        if (lane == 0) {
            prefetch_tensormap(&tq);
            prefetch_tensormap(&tk);
            prefetch_tensormap(&tv);
            mbar_arrive_expect_tx(&sh.q_full, kOp);
#pragma unroll
            for (int r = 0; r < R; ++r)
                tma_load_3d_plain(sQ + r * kRegion, &tq, &sh.q_full, r * 64, kvh * G, q0 + t0);
        }
        int st = 0, round = 0;
        int issued = 0;
        for (int j = 0; j < n_tiles; ++j) {
            if (j >= NS && !warp_wait_bar(&sh.kv_empty[st], (round - 1) & 1, sh, p.err_flag)) break;
            const int last = min(qpos_max, j * kTile + kTile - 1);
            const int nb = (last - j * kTile) / bs + 1;
            int bid = -1;
            bool ok = false;
            if (lane < nb) {
                bid = __ldg(table + j * bpt + lane);
                ok = bid >= 0 && static_cast<int64_t>(bid) < p.num_blocks;
            }
            const unsigned okmask = __ballot_sync(0xffffffffu, ok);
            const unsigned want = (nb >= 32) ? 0xffffffffu : ((1u << nb) - 1u);
            if (lane == 0) {
                if (okmask != want) {
                    report(p.err_flag, PA_FLAG_BAD_BLOCK_ID);
                    sh.bad = 1;
                }
                const uint32_t bytes = static_cast<uint32_t>(__popc(okmask)) * bs * 128u * R;
                mbar_arrive_expect_tx(&sh.k_full[st], bytes);
                mbar_arrive_expect_tx(&sh.v_full[st], bytes);
            }
            __syncwarp();
            if (ok) {
                uint8_t *sK = sKV + static_cast<size_t>(st) * 2 * kOp;
                uint8_t *sV = sK + kOp;
#pragma unroll
                for (int r = 0; r < R; ++r)
                    tma_load_3d_plain(sK + r * kRegion + lane * bs * 128, &tk, &sh.k_full[st], r * 64,
                                      kvh, bid * bs);
#pragma unroll
                for (int r = 0; r < R; ++r)
                    tma_load_3d_plain(sV + r * kRegion + lane * bs * 128, &tv, &sh.v_full[st], r * 64,
                                      kvh, bid * bs);
            }
            ++issued;
            if (++st == NS) {
                st = 0;
                ++round;
            }
        }
        // On an abort, let the copies still in flight land before the CTA exits.
        if (lane == 0 && sh.abort) {
            for (int j = max(0, issued - NS); j < issued; ++j) {
                const int s2 = j % NS;
                mbar_wait_bounded(&sh.k_full[s2], (j / NS) & 1, kWaitLimitNs);
                mbar_wait_bounded(&sh.v_full[s2], (j / NS) & 1, kWaitLimitNs);
            }
        }
    } else if (warp == 5) {
        // ------------------------------------------------------- MMA issuer
        if (lane == 0) {
            const uint32_t q_addr = smem_addr(sQ);
            const uint32_t kv_addr = smem_addr(sKV);
            bool ok = wait_bar(&sh.q_full, 0, sh, p.err_flag);
            auto issue_pv = [&](int i) -> bool {
                const int b = i & 1;
                const int st = i % NS;
                if (!wait_bar(&sh.v_full[st], (i / NS) & 1, sh, p.err_flag)) return false;
                if (!wait_bar(&sh.p_full[b], (i >> 1) & 1, sh, p.err_flag)) return false;
                umma::fence_after_sync();
                const uint32_t v_addr = kv_addr + static_cast<uint32_t>((2 * st + 1) * kOp);
                const uint32_t tP = tmem + 128u * b;
#pragma unroll
                for (int k = 0; k < kPVSteps; ++k)
                    umma::mma_ts(tO, tP + 8u * k, umma::desc_sw128(v_addr + k * 2048, kRegion, 1024),
                                 kIdescPV, (i > 0 || k > 0) ? 1u : 0u);
                if constexpr (BF16) {
#pragma unroll
                    for (int k = 0; k < kPVSteps; ++k)
                        umma::mma_ts(tO, tP + 64u + 8u * k,
                                     umma::desc_sw128(v_addr + k * 2048, kRegion, 1024), kIdescPV, 1u);
                }
                umma::commit(smem_addr(&sh.pv_done[b]));
                umma::commit(smem_addr(&sh.kv_empty[st]));
                return true;
            };
            for (int j = 0; ok && j < n_tiles; ++j) {
                const int b = j & 1;
                const int st = j % NS;
                if (!wait_bar(&sh.k_full[st], (j / NS) & 1, sh, p.err_flag)) { ok = false; break; }
                if (j >= 2 && !wait_bar(&sh.pv_done[b], ((j - 2) >> 1) & 1, sh, p.err_flag)) {
                    ok = false;
                    break;
                }
                umma::fence_after_sync();
                const uint32_t k_addr = kv_addr + static_cast<uint32_t>(2 * st * kOp);
#pragma unroll
                for (int k = 0; k < kKSteps; ++k) {
                    const uint32_t off = (k >> 2) * kRegion + (k & 3) * 32;
                    umma::mma_ss(tmem + 128u * b, umma::desc_sw128(q_addr + off, 16, 1024),
                                 umma::desc_sw128(k_addr + off, 16, 1024), kIdescQK, k > 0 ? 1u : 0u);
                }
                umma::commit(smem_addr(&sh.s_full[b]));
                if (j >= 1 && !issue_pv(j - 1)) { ok = false; break; }
            }
            if (ok) issue_pv(n_tiles - 1);
            umma::commit(smem_addr(&sh.done));
            mbar_wait_bounded(&sh.done, 0, kWaitLimitNs);
        }
        __syncwarp();
    } else {
        // ------------------------------------------- softmax and epilogue
        const bool row_valid = rtok < ntok;
        const int qpos = row_valid ? qstart + rtok : -1;
        const uint32_t lane_off = static_cast<uint32_t>(warp * 32) << 16;
        const float sl = p.scale_log2;
        float m_run = -CUDART_INF_F;
        float l_run = 0.f;
        bool ok = true;
        for (int j = 0; j < n_tiles; ++j) {
            const int b = j & 1;
            if (!warp_wait_bar(&sh.s_full[b], (j >> 1) & 1, sh, p.err_flag)) { ok = false; break; }
            umma::fence_after_sync();
            const uint32_t tS = tmem + 128u * b + lane_off;
            uint32_t sv[kTile];
#pragma unroll
            for (int c = 0; c < kTile / 32; ++c)
                umma::ld_32x32b_x32(tS + 32 * c, *reinterpret_cast<uint32_t(*)[32]>(sv + 32 * c));
            umma::wait_ld();
            const int lim = qpos - j * kTile;        // columns c <= lim are attended
            float mx = -CUDART_INF_F;
#pragma unroll
            for (int c = 0; c < kTile; ++c)
                if (c <= lim) mx = fmaxf(mx, __uint_as_float(sv[c]));
            const float x_tile = mx * sl;
            const bool need = x_tile > m_run + 8.f;
            if (__any_sync(0xffffffffu, need)) {
                const float f = need ? fast_exp2(m_run - x_tile) : 1.f;
                if (j > 0) {
                    if (!warp_wait_bar(&sh.pv_done[(j - 1) & 1], ((j - 1) >> 1) & 1, sh, p.err_flag)) {
                        ok = false;
                        break;
                    }
                    umma::fence_after_sync();
#pragma unroll
                    for (int c = 0; c < D / 32; ++c) {
                        uint32_t o[32];
                        umma::ld_32x32b_x32(tO + lane_off + 32 * c, o);
                        umma::wait_ld();
#pragma unroll
                        for (int i = 0; i < 32; ++i) o[i] = __float_as_uint(__uint_as_float(o[i]) * f);
                        st_32x32b_x32(tO + lane_off + 32 * c, o);
                    }
                }
                if (need) {
                    l_run *= f;
                    m_run = x_tile;
                }
            }
            // weights, written back over S as 16-bit pairs
            float lsum = 0.f;
#pragma unroll
            for (int c = 0; c < kTile / 32; ++c) {
                uint32_t hi[16], lo[16];
#pragma unroll
                for (int i = 0; i < 16; ++i) {
                    const int k = 32 * c + 2 * i;
                    const float p0 = (k <= lim) ? fast_exp2(fmaf(__uint_as_float(sv[k]), sl, -m_run)) : 0.f;
                    const float p1 =
                        (k + 1 <= lim) ? fast_exp2(fmaf(__uint_as_float(sv[k + 1]), sl, -m_run)) : 0.f;
                    hi[i] = pack_pair<BF16>(p0, p1);
                    const float2 h = Half2x<BF16>::to_float2(hi[i]);
                    if constexpr (BF16) {
                        lo[i] = pack_pair<true>(p0 - h.x, p1 - h.y);
                        lsum += p0 + p1;
                    } else {
                        lsum += h.x + h.y;
                    }
                }
                umma::st_32x32b_x16(tS + 16 * c, hi);
                if constexpr (BF16) umma::st_32x32b_x16(tS + 64 + 16 * c, lo);
            }
            l_run += lsum;
            if (j == n_tiles - 1 && j * kTile + kTile - 1 > qpos_max) {
                // V rows past the last attended position hold stale or unloaded
                // data; zero them so that 0-weights cannot meet NaNs.
                const int st = j % NS;
                if (!warp_wait_bar(&sh.v_full[st], (j / NS) & 1, sh, p.err_flag)) { ok = false; break; }
                if (j * kTile + row > qpos_max) {
                    uint8_t *sV = sKV + static_cast<size_t>(2 * st + 1) * kOp;
#pragma unroll
                    for (int r = 0; r < R; ++r) {
                        uint4 *d = reinterpret_cast<uint4 *>(sV + r * kRegion + row * 128);
#pragma unroll
                        for (int i = 0; i < 8; ++i) d[i] = make_uint4(0u, 0u, 0u, 0u);
                    }
                }
                fence_proxy_async_smem();
            }
            umma::wait_st();
            umma::fence_before_sync();
            mbar_arrive(&sh.p_full[b]);
        }
        if (ok && warp_wait_bar(&sh.pv_done[(n_tiles - 1) & 1], ((n_tiles - 1) >> 1) & 1, sh, p.err_flag)) {
            umma::fence_after_sync();
            const bool zero = *reinterpret_cast<volatile int *>(&sh.bad) != 0;
            const float inv = (l_run > 0.f && !zero) ? 1.f / l_run : 0.f;
#pragma unroll
            for (int c = 0; c < D / 32; ++c) {
                uint32_t o[32];
                umma::ld_32x32b_x32(tO + lane_off + 32 * c, o);
                umma::wait_ld();
                float v[32];
#pragma unroll
                for (int i = 0; i < 32; ++i) v[i] = zero ? 0.f : __uint_as_float(o[i]) * inv;
                if (row_valid) store_chunk(p.out, p.out_dtype, out_row * D + c * 32, v);
            }
        }
    }

    umma::fence_before_sync();
    __syncthreads();
    if (warp == 5) {
        umma::fence_after_sync();
        umma::tmem_dealloc(tmem, kTmemCols);
    }
}

template <int D, bool BF16>
cudaError_t launch_t(const PrefillParams &p, const CUtensorMap &tq, const CUtensorMap &tk,
                     const CUtensorMap &tv, size_t smem, cudaStream_t stream) {
    auto kern = paged_prefill_kernel<D, BF16>;
    cudaError_t e = cudaFuncSetAttribute(kern, cudaFuncAttributeMaxDynamicSharedMemorySize,
                                         static_cast<int>(smem));
    if (e != cudaSuccess) return e;
    const int64_t grid = static_cast<int64_t>(p.num_seqs) * p.num_kv_heads * p.tiles_per_seq;
    kern<<<static_cast<unsigned>(grid), kPrefillThreads, smem, stream>>>(p, tq, tk, tv);
    return cudaGetLastError();
}

}  // namespace

size_t prefill_smem_bytes(int head_dim, int stages) {
    const size_t op = static_cast<size_t>(head_dim / 64) * kRegion;
    return 1024 + op + static_cast<size_t>(stages) * 2 * op;
}

cudaError_t launch_prefill(const PrefillParams &p, int head_dim, bool bf16, const CUtensorMap &tq,
                           const CUtensorMap &tk, const CUtensorMap &tv, size_t smem,
                           cudaStream_t stream) {
    if (p.stages < 1 || p.stages > kMaxStages) return cudaErrorInvalidValue;
    if (head_dim == 128)
        return bf16 ? launch_t<128, true>(p, tq, tk, tv, smem, stream)
                    : launch_t<128, false>(p, tq, tk, tv, smem, stream);
    if (head_dim == 64)
        return bf16 ? launch_t<64, true>(p, tq, tk, tv, smem, stream)
                    : launch_t<64, false>(p, tq, tk, tv, smem, stream);
    return cudaErrorInvalidValue;
}

}  // namespace pa
