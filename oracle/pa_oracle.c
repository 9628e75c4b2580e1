/*
 * CPU oracle for paged decode attention -- TEST INFRASTRUCTURE ONLY.
 *
 * Plain, slow, obviously correct C in double precision.  Only the test suite,
 * the package's smoke check and the benchmark's CPU-baseline leg load it; the
 * product path never does.  It shares no code, header or constant with the
 * CUDA library.
 *
 * What it computes (sources are the pages on vLLM PagedAttention):
 *   - reshape_and_cache: each new token's K/V row is written into the cache
 *     slot  slot = physical_block * block_size + offset  ("nano-vllm"
 *     walkthrough, lqnn.cn/news/170268, §2.2: write into the current block
 *     while it has room; §2.3 step 3: write back and update the count).
 *   - copy_blocks: copy-on-write duplicates a whole shared block before a
 *     write ("优化大模型推理：PagedAttention 如何实现 GPU 显存高效管理",
 *     section on copy-on-write; "LLM推理优化：vLLM PagedAttention深度解析与
 *     工程实践", §3.1).
 *   - paged attention: for every sequence and query head, gather the K/V
 *     rows of positions 0..ctx-1 through the block table and evaluate
 *     softmax(q K^T * scale) V  ("LLM推理优化…", §二 formula; §4.1 layout
 *     [num_blocks, block_size, num_heads, head_dim]; nano-vllm §2.3 steps 1-2).
 *     Paging changes where rows live, not the mathematics ("优化大模型推理…",
 *     section on decoupling logical and physical contiguity).
 *   - partitioned attention: the "partial accumulate, then merge" reading of
 *     paged_attention_v2 ("LLM推理优化…", §4.1): per partition a running max,
 *     a sum of exponentials and an unnormalised weighted V sum, then a merge.
 *
 * Readings where the pages are silent (each listed in the design notes):
 *   - GQA grouping: query head hq reads KV head hq / (Hq / Hkv).
 *   - Positions >= ctx are never read (stale slots must not matter, nano-vllm §6).
 *   - ctx <= 0 gives an all-zero output row.
 *   - Half inputs are decoded exactly from their bits (binary16 / bfloat16).
 */
#include <math.h>
#include <stdint.h>
#include <stdlib.h>
#include <string.h>

#define ORACLE_F16 0
#define ORACLE_BF16 1

/* Exact value of an IEEE binary16 bit pattern. */
static double decode_binary16(uint16_t h) {
    int sign = (h >> 15) & 1;
    int e = (h >> 10) & 0x1f;
    int m = h & 0x3ff;
    double v;
    if (e == 0) {
        v = ldexp((double)m, -24);                 /* zero / subnormal */
    } else if (e == 31) {
        v = (m == 0) ? INFINITY : NAN;
    } else {
        v = ldexp((double)(1024 + m), e - 25);     /* 1.m * 2^(e-15) */
    }
    return sign ? -v : v;
}

/* Exact value of a bfloat16 bit pattern (8 exponent bits, 7 mantissa bits). */
static double decode_bfloat16(uint16_t h) {
    int sign = (h >> 15) & 1;
    int e = (h >> 7) & 0xff;
    int m = h & 0x7f;
    double v;
    if (e == 0) {
        v = ldexp((double)m, -133);                /* zero / subnormal: m * 2^(-126-7) */
    } else if (e == 255) {
        v = (m == 0) ? INFINITY : NAN;
    } else {
        v = ldexp((double)(128 + m), e - 134);     /* 1.m * 2^(e-127) */
    }
    return sign ? -v : v;
}

double oracle_half_to_double(uint16_t bits, int dtype) {
    return dtype == ORACLE_BF16 ? decode_bfloat16(bits) : decode_binary16(bits);
}

/* key/value: [T, Hkv, D]; caches: [NB, bs, Hkv, D] (16-bit elements).
 * A negative slot means "no write".  Slots >= NB*bs are skipped and counted;
 * the return value is the number of skipped out-of-range slots. */
int64_t oracle_reshape_and_cache(const uint16_t *key, const uint16_t *value,
                                 uint16_t *k_cache, uint16_t *v_cache,
                                 const int64_t *slot_mapping, int64_t num_tokens,
                                 int64_t num_blocks, int block_size,
                                 int num_kv_heads, int head_dim) {
    int64_t row = (int64_t)num_kv_heads * head_dim;
    int64_t bad = 0;
    for (int64_t t = 0; t < num_tokens; ++t) {
        int64_t slot = slot_mapping[t];
        if (slot < 0) continue;
        if (slot >= num_blocks * block_size) { ++bad; continue; }
        int64_t block = slot / block_size;
        int64_t offset = slot % block_size;
        int64_t dst = (block * block_size + offset) * row;
        for (int64_t i = 0; i < row; ++i) {
            k_cache[dst + i] = key[t * row + i];
            v_cache[dst + i] = value[t * row + i];
        }
    }
    return bad;
}

/* block_mapping: [P, 2] pairs (src, dst), applied in pair order.  Pairs with
 * an id outside [0, NB) are skipped and counted. */
int64_t oracle_copy_blocks(uint16_t *k_cache, uint16_t *v_cache,
                           const int64_t *block_mapping, int64_t num_pairs,
                           int64_t num_blocks, int block_size,
                           int num_kv_heads, int head_dim) {
    size_t block_bytes = (size_t)block_size * num_kv_heads * head_dim * sizeof(uint16_t);
    size_t block_elems = (size_t)block_size * num_kv_heads * head_dim;
    int64_t bad = 0;
    for (int64_t p = 0; p < num_pairs; ++p) {
        int64_t src = block_mapping[2 * p];
        int64_t dst = block_mapping[2 * p + 1];
        if (src < 0 || src >= num_blocks || dst < 0 || dst >= num_blocks) { ++bad; continue; }
        memcpy(k_cache + dst * block_elems, k_cache + src * block_elems, block_bytes);
        memcpy(v_cache + dst * block_elems, v_cache + src * block_elems, block_bytes);
    }
    return bad;
}

/* Gather the K and V rows of positions [p0, p1) of sequence s, KV head kvh,
 * through the block table, as doubles: Kg/Vg are [(p1-p0), D]. */
static void gather_rows(double *Kg, double *Vg, const uint16_t *k_cache, const uint16_t *v_cache,
                        int dtype, const int32_t *table_row, int p0, int p1,
                        int num_kv_heads, int head_dim, int block_size, int kvh) {
    for (int p = p0; p < p1; ++p) {
        int64_t block = table_row[p / block_size];
        int64_t offset = p % block_size;
        const uint16_t *kr = k_cache + ((block * block_size + offset) * num_kv_heads + kvh) * (int64_t)head_dim;
        const uint16_t *vr = v_cache + ((block * block_size + offset) * num_kv_heads + kvh) * (int64_t)head_dim;
        for (int d = 0; d < head_dim; ++d) {
            Kg[(int64_t)(p - p0) * head_dim + d] = oracle_half_to_double(kr[d], dtype);
            Vg[(int64_t)(p - p0) * head_dim + d] = oracle_half_to_double(vr[d], dtype);
        }
    }
}

/* out: [B, Hq, D] doubles.  q: [B, Hq, D]; caches [NB, bs, Hkv, D];
 * block_tables: [B, max_blocks_per_seq]; context_lens: [B]. */
void oracle_paged_attention(double *out, const uint16_t *q,
                            const uint16_t *k_cache, const uint16_t *v_cache, int dtype,
                            const int32_t *block_tables, int max_blocks_per_seq,
                            const int32_t *context_lens, int num_seqs, int num_heads,
                            int num_kv_heads, int head_dim, int block_size, double scale) {
    int group = num_heads / num_kv_heads;
#pragma omp parallel for collapse(2) schedule(dynamic, 1)
    for (int s = 0; s < num_seqs; ++s) {
        for (int hq = 0; hq < num_heads; ++hq) {
            double *o = out + ((int64_t)s * num_heads + hq) * head_dim;
            int n = context_lens[s];
            for (int d = 0; d < head_dim; ++d) o[d] = 0.0;
            if (n <= 0) continue;
            int kvh = hq / group;
            double *Kg = (double *)malloc(sizeof(double) * (size_t)n * head_dim);
            double *Vg = (double *)malloc(sizeof(double) * (size_t)n * head_dim);
            double *x = (double *)malloc(sizeof(double) * (size_t)n);
            double *qd = (double *)malloc(sizeof(double) * (size_t)head_dim);
            gather_rows(Kg, Vg, k_cache, v_cache, dtype,
                        block_tables + (int64_t)s * max_blocks_per_seq, 0, n,
                        num_kv_heads, head_dim, block_size, kvh);
            for (int d = 0; d < head_dim; ++d)
                qd[d] = oracle_half_to_double(q[((int64_t)s * num_heads + hq) * head_dim + d], dtype);
            /* logits x_p = scale * <q, K_p> */
            double m = -INFINITY;
            for (int p = 0; p < n; ++p) {
                double dot = 0.0;
                for (int d = 0; d < head_dim; ++d) dot += qd[d] * Kg[(int64_t)p * head_dim + d];
                x[p] = scale * dot;
                if (x[p] > m) m = x[p];
            }
            /* softmax weights w_p = exp(x_p - m), then o = sum_p w_p V_p / sum_p w_p */
            double den = 0.0;
            for (int p = 0; p < n; ++p) {
                x[p] = exp(x[p] - m);
                den += x[p];
            }
            for (int d = 0; d < head_dim; ++d) {
                double acc = 0.0;
                for (int p = 0; p < n; ++p) acc += x[p] * Vg[(int64_t)p * head_dim + d];
                o[d] = acc / den;
            }
            free(Kg); free(Vg); free(x); free(qd);
        }
    }
}

/* The partition-then-merge reading of paged_attention_v2.
 * Each sequence's context is cut into partitions of `partition_size` tokens.
 * For partition j of (s, hq):  m_j = max x,  l_j = sum exp(x - m_j),
 * acc_j[d] = sum exp(x - m_j) V[d].  Merge:  M = max_j m_j,
 * L = sum_j l_j exp(m_j - M),  out = sum_j acc_j exp(m_j - M) / L, taking the
 * partitions in order.  part_max/part_sum: [B, Hq, max_partitions];
 * part_acc: [B, Hq, max_partitions, D]; any of the three may be NULL.
 * Partitions past a sequence's end are written as (-inf, 0, 0). */
void oracle_paged_attention_partitioned(double *out, double *part_max, double *part_sum,
                                        double *part_acc, const uint16_t *q,
                                        const uint16_t *k_cache, const uint16_t *v_cache, int dtype,
                                        const int32_t *block_tables, int max_blocks_per_seq,
                                        const int32_t *context_lens, int num_seqs, int num_heads,
                                        int num_kv_heads, int head_dim, int block_size, double scale,
                                        int partition_size, int max_partitions) {
    int group = num_heads / num_kv_heads;
#pragma omp parallel for collapse(2) schedule(dynamic, 1)
    for (int s = 0; s < num_seqs; ++s) {
        for (int hq = 0; hq < num_heads; ++hq) {
            int64_t sh = (int64_t)s * num_heads + hq;
            double *o = out + sh * head_dim;
            int n = context_lens[s];
            int nparts = n > 0 ? (n + partition_size - 1) / partition_size : 0;
            for (int d = 0; d < head_dim; ++d) o[d] = 0.0;
            for (int j = 0; j < max_partitions; ++j) {
                if (part_max) part_max[sh * max_partitions + j] = -INFINITY;
                if (part_sum) part_sum[sh * max_partitions + j] = 0.0;
                if (part_acc)
                    for (int d = 0; d < head_dim; ++d) part_acc[(sh * max_partitions + j) * head_dim + d] = 0.0;
            }
            if (n <= 0) continue;
            int kvh = hq / group;
            double *Kg = (double *)malloc(sizeof(double) * (size_t)partition_size * head_dim);
            double *Vg = (double *)malloc(sizeof(double) * (size_t)partition_size * head_dim);
            double *x = (double *)malloc(sizeof(double) * (size_t)partition_size);
            double *qd = (double *)malloc(sizeof(double) * (size_t)head_dim);
            double *mj = (double *)malloc(sizeof(double) * (size_t)nparts);
            double *lj = (double *)malloc(sizeof(double) * (size_t)nparts);
            double *aj = (double *)malloc(sizeof(double) * (size_t)nparts * head_dim);
            for (int d = 0; d < head_dim; ++d)
                qd[d] = oracle_half_to_double(q[sh * head_dim + d], dtype);
            for (int j = 0; j < nparts; ++j) {
                int p0 = j * partition_size;
                int p1 = p0 + partition_size < n ? p0 + partition_size : n;
                gather_rows(Kg, Vg, k_cache, v_cache, dtype,
                            block_tables + (int64_t)s * max_blocks_per_seq, p0, p1,
                            num_kv_heads, head_dim, block_size, kvh);
                double m = -INFINITY;
                for (int p = 0; p < p1 - p0; ++p) {
                    double dot = 0.0;
                    for (int d = 0; d < head_dim; ++d) dot += qd[d] * Kg[(int64_t)p * head_dim + d];
                    x[p] = scale * dot;
                    if (x[p] > m) m = x[p];
                }
                double l = 0.0;
                for (int p = 0; p < p1 - p0; ++p) {
                    x[p] = exp(x[p] - m);
                    l += x[p];
                }
                for (int d = 0; d < head_dim; ++d) {
                    double acc = 0.0;
                    for (int p = 0; p < p1 - p0; ++p) acc += x[p] * Vg[(int64_t)p * head_dim + d];
                    aj[(int64_t)j * head_dim + d] = acc;
                }
                mj[j] = m;
                lj[j] = l;
                if (j < max_partitions) {
                    if (part_max) part_max[sh * max_partitions + j] = m;
                    if (part_sum) part_sum[sh * max_partitions + j] = l;
                    if (part_acc)
                        for (int d = 0; d < head_dim; ++d)
                            part_acc[(sh * max_partitions + j) * head_dim + d] = aj[(int64_t)j * head_dim + d];
                }
            }
            /* merge, partitions in order */
            double M = -INFINITY;
            for (int j = 0; j < nparts; ++j) if (mj[j] > M) M = mj[j];
            double L = 0.0;
            for (int j = 0; j < nparts; ++j) L += lj[j] * exp(mj[j] - M);
            for (int d = 0; d < head_dim; ++d) {
                double acc = 0.0;
                for (int j = 0; j < nparts; ++j) acc += aj[(int64_t)j * head_dim + d] * exp(mj[j] - M);
                o[d] = acc / L;
            }
            free(Kg); free(Vg); free(x); free(qd); free(mj); free(lj); free(aj);
        }
    }
}

/* ------------------------------------------------------------------------
 * FP8 (e4m3, "fn": no infinities, max 448) KV cache.
 *
 * The pages list FP8 among vLLM's quantisation options ("LLM推理优化：vLLM
 * PagedAttention深度解析与工程实践", §八 comparison table).  Readings used here
 * (the pages give no detail): one scale per tensor for K and one for V; the
 * cache stores code = e4m3(x / scale) with x widened to fp32, the division in
 * fp32, rounding to nearest-even and saturation of finite values to +-448
 * (NaN stays NaN); attention reads K = e4m3_value(code) * k_scale (V alike).
 * ------------------------------------------------------------------------ */

/* Exact value of an e4m3 code: s eeee mmm, bias 7; e=15,m=7 is NaN. */
double oracle_e4m3_decode(uint8_t c) {
    int sign = (c >> 7) & 1;
    int e = (c >> 3) & 0xf;
    int m = c & 7;
    double v;
    if (e == 15 && m == 7) return NAN;
    if (e == 0) v = ldexp((double)m, -9);              /* subnormal: m * 2^-9 */
    else v = ldexp((double)(8 + m), e - 10);           /* 1.m * 2^(e-7) */
    return sign ? -v : v;
}

/* Round a float to the nearest e4m3 code (ties to even), saturating finite
 * values (and infinities) to +-448; NaN -> 0x7f. */
uint8_t oracle_e4m3_encode(float x) {
    if (x != x) return 0x7f;
    uint8_t sign = (x < 0.0f || (x == 0.0f && signbit(x))) ? 0x80 : 0x00;
    double a = fabs((double)x);
    if (a >= 448.0) return (uint8_t)(sign | 0x7e);
    int code;
    if (a < ldexp(1.0, -6)) {
        /* subnormal grid, step 2^-9; a result of 8 is the smallest normal */
        code = (int)rint(a / ldexp(1.0, -9));
    } else {
        int e;
        frexp(a, &e);                    /* a = f * 2^e, f in [0.5, 1) */
        int ue = e - 1;                  /* a in [2^ue, 2^(ue+1)) */
        double q = rint(a / ldexp(1.0, ue - 3));   /* in [8, 16] */
        code = ((ue + 7) << 3) + ((int)q - 8);     /* q = 16 carries into the exponent */
    }
    if (code > 0x7e) code = 0x7e;
    return (uint8_t)(sign | code);
}

static double half_or_bf16(uint16_t bits, int dtype) { return oracle_half_to_double(bits, dtype); }

/* reshape_and_cache into an e4m3 cache: key/value hold 16-bit values of
 * `dtype`; caches hold one byte per element.  Returns the number of skipped
 * out-of-range slots (negative slots are padding and skipped silently). */
int64_t oracle_reshape_and_cache_fp8(const uint16_t *key, const uint16_t *value, int dtype,
                                     uint8_t *k_cache, uint8_t *v_cache,
                                     const int64_t *slot_mapping, int64_t num_tokens,
                                     int64_t num_blocks, int block_size,
                                     int num_kv_heads, int head_dim, float k_scale, float v_scale) {
    int64_t row = (int64_t)num_kv_heads * head_dim;
    int64_t bad = 0;
    for (int64_t t = 0; t < num_tokens; ++t) {
        int64_t slot = slot_mapping[t];
        if (slot < 0) continue;
        if (slot >= num_blocks * block_size) { ++bad; continue; }
        for (int64_t i = 0; i < row; ++i) {
            float kx = (float)half_or_bf16(key[t * row + i], dtype);
            float vx = (float)half_or_bf16(value[t * row + i], dtype);
            volatile float kq = kx / k_scale;    /* fp32 division */
            volatile float vq = vx / v_scale;
            k_cache[slot * row + i] = oracle_e4m3_encode(kq);
            v_cache[slot * row + i] = oracle_e4m3_encode(vq);
        }
    }
    return bad;
}

/* Paged attention over an e4m3 cache: q holds 16-bit values of `q_dtype`;
 * K_p = e4m3(k_cache) * k_scale, V_p = e4m3(v_cache) * v_scale; otherwise as
 * oracle_paged_attention (fp64 throughout). */
void oracle_paged_attention_fp8(double *out, const uint16_t *q, int q_dtype,
                                const uint8_t *k_cache, const uint8_t *v_cache,
                                double k_scale, double v_scale,
                                const int32_t *block_tables, int max_blocks_per_seq,
                                const int32_t *context_lens, int num_seqs, int num_heads,
                                int num_kv_heads, int head_dim, int block_size, double scale) {
    int group = num_heads / num_kv_heads;
#pragma omp parallel for collapse(2) schedule(dynamic, 1)
    for (int s = 0; s < num_seqs; ++s) {
        for (int hq = 0; hq < num_heads; ++hq) {
            double *o = out + ((int64_t)s * num_heads + hq) * head_dim;
            int n = context_lens[s];
            for (int d = 0; d < head_dim; ++d) o[d] = 0.0;
            if (n <= 0) continue;
            int kvh = hq / group;
            const int32_t *table_row = block_tables + (int64_t)s * max_blocks_per_seq;
            double *Kg = (double *)malloc(sizeof(double) * (size_t)n * head_dim);
            double *Vg = (double *)malloc(sizeof(double) * (size_t)n * head_dim);
            double *x = (double *)malloc(sizeof(double) * (size_t)n);
            double *qd = (double *)malloc(sizeof(double) * (size_t)head_dim);
            for (int p = 0; p < n; ++p) {
                int64_t block = table_row[p / block_size];
                int64_t offset = p % block_size;
                int64_t base = ((block * block_size + offset) * num_kv_heads + kvh) * (int64_t)head_dim;
                for (int d = 0; d < head_dim; ++d) {
                    Kg[(int64_t)p * head_dim + d] = oracle_e4m3_decode(k_cache[base + d]) * k_scale;
                    Vg[(int64_t)p * head_dim + d] = oracle_e4m3_decode(v_cache[base + d]) * v_scale;
                }
            }
            for (int d = 0; d < head_dim; ++d)
                qd[d] = oracle_half_to_double(q[((int64_t)s * num_heads + hq) * head_dim + d], q_dtype);
            double m = -INFINITY;
            for (int p = 0; p < n; ++p) {
                double dot = 0.0;
                for (int d = 0; d < head_dim; ++d) dot += qd[d] * Kg[(int64_t)p * head_dim + d];
                x[p] = scale * dot;
                if (x[p] > m) m = x[p];
            }
            double den = 0.0;
            for (int p = 0; p < n; ++p) {
                x[p] = exp(x[p] - m);
                den += x[p];
            }
            for (int d = 0; d < head_dim; ++d) {
                double acc = 0.0;
                for (int p = 0; p < n; ++p) acc += x[p] * Vg[(int64_t)p * head_dim + d];
                o[d] = acc / den;
            }
            free(Kg); free(Vg); free(x); free(qd);
        }
    }
}

/* Elementwise helpers for the Python wrapper. */
void oracle_e4m3_encode_array(const float *x, uint8_t *out, int64_t n) {
    for (int64_t i = 0; i < n; ++i) out[i] = oracle_e4m3_encode(x[i]);
}
void oracle_e4m3_decode_array(const uint8_t *c, double *out, int64_t n) {
    for (int64_t i = 0; i < n; ++i) out[i] = oracle_e4m3_decode(c[i]);
}

/* ------------------------------------------------------------------------
 * swap_blocks: copy whole blocks between two caches (swap-mode preemption:
 * a preempted request's KV blocks go to CPU memory and come back later,
 * "vLLM 核心：PagedAttention 与 Continuous Batching", §5 strategy 1).
 * For each pair (src, dst), in pair order: dst_k[dst] = src_k[src],
 * dst_v[dst] = src_v[src].  `block_bytes` bytes per block and tensor.
 * Pairs with an id outside its cache are skipped and counted.
 * ------------------------------------------------------------------------ */
int64_t oracle_swap_blocks(const uint8_t *src_k, const uint8_t *src_v, uint8_t *dst_k, uint8_t *dst_v,
                           const int64_t *block_mapping, int64_t num_pairs, int64_t src_num_blocks,
                           int64_t dst_num_blocks, int64_t block_bytes) {
    int64_t bad = 0;
    for (int64_t p = 0; p < num_pairs; ++p) {
        int64_t src = block_mapping[2 * p];
        int64_t dst = block_mapping[2 * p + 1];
        if (src < 0 || src >= src_num_blocks || dst < 0 || dst >= dst_num_blocks) { ++bad; continue; }
        memcpy(dst_k + dst * block_bytes, src_k + src * block_bytes, (size_t)block_bytes);
        memcpy(dst_v + dst * block_bytes, src_v + src * block_bytes, (size_t)block_bytes);
    }
    return bad;
}
