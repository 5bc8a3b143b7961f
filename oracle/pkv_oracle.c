/*
 * pkv_oracle.c -- plain float64 CPU oracle for paged decode attention,
 * paged (chunked) prefill attention, the slot-mapped KV append and the
 * copy-on-write block copy.
 *
 * TEST INFRASTRUCTURE ONLY.  Nothing on the product path may link, load or
 * call this file: only tests/, __graft_entry__.smoke() and the cpu_baseline
 * leg of bench.py use it.  It shares no code, header or constant table with
 * the CUDA library; every format below is decoded from its published
 * definition.
 *
 * Sources (web pages on vLLM's PagedAttention):
 *  [P1] "vLLM 高性能大语言模型推理引擎深度技术评估与分布式架构展望",
 *       sections "PagedAttention 内存管理与核心数据结构", "逻辑块到物理块的映射转换",
 *       "束搜索与并行采样的三大调度原语".
 *  [P3] "vLLM：大语言模型推理与服务库", section 4.2 (physical block, block table,
 *       block pool), 4.3 (memory-management flow), 4.4 (PagedAttention CUDA
 *       kernel: inputs q / k_cache / v_cache / block_tables / context_lens;
 *       per query: walk the block table, q.K -> softmax -> weighted V).
 *  [P4] "vLLM 深度解析：从 PagedAttention 到生产部署", sections
 *       "PagedAttention 的解法" and "Prefix Caching 与 Copy-on-Write".
 *
 * Readings where the pages are silent (each is listed with its reason in the
 * design notes of the repository):
 *  - KV pool layout: K and V are separate pools laid out [NB][Hkv][b][D]
 *    (row-major); element (blk, h, off, d) is at ((blk*Hkv + h)*b + off)*D + d.
 *  - seq_lens count the token appended in the same step.
 *  - slot = physical_block * b + offset; a negative slot is padding, skipped.
 *  - GQA: query head i reads KV head i / (Hq / Hkv).
 *  - fp8 is OCP E4M3FN (bias 7, max finite 448, no infinities, S.1111.111 is
 *    NaN) with one per-tensor scale: stored value = code_value * scale.
 *    Encoding divides in IEEE binary32 and rounds to nearest, ties to even,
 *    saturating to +-448.
 *  - seq_len 0 gives an all-zero output row.
 */
#include <math.h>
#include <stdint.h>
#include <stdlib.h>
#include <string.h>
#ifdef _OPENMP
#include <omp.h>
#endif

/* element type codes (same meaning as the library's public enum) */
#define PKVO_F16 0
#define PKVO_BF16 1
#define PKVO_E4M3 2

#define PKVO_OK 0
#define PKVO_EINVAL 1

/* ---------------------------------------------------------------- formats */

/* IEEE 754 binary16: 1 sign bit, 5 exponent bits (bias 15), 10 fraction bits. */
double pkvo_f16_to_double(uint16_t h) {
    int sign = (h >> 15) & 1;
    int e = (h >> 10) & 0x1f;
    int f = h & 0x3ff;
    double v;
    if (e == 0)
        v = ldexp((double)f, -24);                 /* subnormal: f * 2^-14 / 2^10 */
    else if (e == 31)
        v = f ? NAN : INFINITY;
    else
        v = ldexp(1.0 + f / 1024.0, e - 15);
    return sign ? -v : v;
}

/* bfloat16: the upper 16 bits of an IEEE binary32 (8 exponent bits, bias 127,
 * 7 fraction bits). */
double pkvo_bf16_to_double(uint16_t h) {
    int sign = (h >> 15) & 1;
    int e = (h >> 7) & 0xff;
    int f = h & 0x7f;
    double v;
    if (e == 0)
        v = ldexp((double)f, -133);                /* f * 2^-126 / 2^7 */
    else if (e == 255)
        v = f ? NAN : INFINITY;
    else
        v = ldexp(1.0 + f / 128.0, e - 127);
    return sign ? -v : v;
}

/* OCP 8-bit E4M3 ("FN"): 1 sign, 4 exponent bits (bias 7), 3 fraction bits;
 * exponent 0 is subnormal (f * 2^-9); S.1111.111 is NaN; no infinities. */
double pkvo_e4m3_to_double(uint8_t c) {
    int sign = (c >> 7) & 1;
    int e = (c >> 3) & 0xf;
    int f = c & 0x7;
    double v;
    if (e == 15 && f == 7)
        v = NAN;
    else if (e == 0)
        v = ldexp((double)f, -9);
    else
        v = ldexp(1.0 + f / 8.0, e - 7);
    return sign ? -v : v;
}

/* Round a binary32 value to the nearest E4M3 code, ties to the even code,
 * saturating finite overflow to +-448.  Written as a search over the 127
 * non-negative finite codes so that it follows the definition directly. */
uint8_t pkvo_e4m3_encode(float x) {
    uint8_t sign = signbit(x) ? 0x80 : 0x00;
    if (isnan(x)) return (uint8_t)(sign | 0x7f);
    double a = fabs((double)x);
    if (a >= 448.0) return (uint8_t)(sign | 0x7e);
    int best = 0;
    double best_err = INFINITY;
    for (int c = 0; c <= 0x7e; ++c) {
        double err = fabs(pkvo_e4m3_to_double((uint8_t)c) - a);
        if (err < best_err || (err == best_err && (c & 1) == 0 && (best & 1) == 1)) {
            best = c;
            best_err = err;
        }
    }
    return (uint8_t)(sign | best);
}

static double elem_to_double(const void* base, int dtype, int64_t idx) {
    switch (dtype) {
    case PKVO_F16: return pkvo_f16_to_double(((const uint16_t*)base)[idx]);
    case PKVO_BF16: return pkvo_bf16_to_double(((const uint16_t*)base)[idx]);
    default: return pkvo_e4m3_to_double(((const uint8_t*)base)[idx]);
    }
}

static int elem_bytes(int dtype) { return dtype == PKVO_E4M3 ? 1 : 2; }

/* Pool accessor for the [NB][Hkv][b][D] layout. */
static int64_t pool_index(int64_t blk, int h, int off, int d, int Hkv, int b, int D) {
    return ((blk * Hkv + h) * (int64_t)b + off) * D + d;
}

/* -------------------------------------------------------------- attention */

typedef struct {
    const void* q; int q_dtype; int S; int Hq;
    const void* k_pool; const void* v_pool; int kv_dtype;
    int NB; int b; int Hkv; int D; double k_scale; double v_scale;
    const int32_t* block_tables; int MB; const int32_t* seq_lens; double scale;
} pkvo_args;

/* Scores of one (sequence, query head) over tokens [t0, t1) into sc[].
 * Returns PKVO_EINVAL on a block id outside the pool. */
static int scores_range(const pkvo_args* a, int s, int i, int t0, int t1, double* sc) {
    int G = a->Hq / a->Hkv;
    int h = i / G;
    double* qrow = (double*)malloc(sizeof(double) * (size_t)a->D);
    for (int d = 0; d < a->D; ++d)
        qrow[d] = elem_to_double(a->q, a->q_dtype, ((int64_t)s * a->Hq + i) * a->D + d);
    for (int t = t0; t < t1; ++t) {
        int32_t blk = a->block_tables[(int64_t)s * a->MB + t / a->b];
        if (blk < 0 || blk >= a->NB) { free(qrow); return PKVO_EINVAL; }
        int off = t % a->b;
        double dot = 0.0;
        for (int d = 0; d < a->D; ++d) {
            double kv = elem_to_double(a->k_pool, a->kv_dtype,
                                       pool_index(blk, h, off, d, a->Hkv, a->b, a->D)) * a->k_scale;
            dot += qrow[d] * kv;
        }
        sc[t - t0] = a->scale * dot;
    }
    free(qrow);
    return PKVO_OK;
}

/* Adds sum_t w[t] * v_t into acc[D] for tokens [t0, t1). */
static void weighted_v(const pkvo_args* a, int s, int i, int t0, int t1, const double* w, double* acc) {
    int G = a->Hq / a->Hkv;
    int h = i / G;
    for (int t = t0; t < t1; ++t) {
        int32_t blk = a->block_tables[(int64_t)s * a->MB + t / a->b];
        int off = t % a->b;
        for (int d = 0; d < a->D; ++d)
            acc[d] += w[t - t0] * elem_to_double(a->v_pool, a->kv_dtype,
                                                 pool_index(blk, h, off, d, a->Hkv, a->b, a->D)) * a->v_scale;
    }
}

static int check_args(const pkvo_args* a) {
    if (a->S < 0 || a->Hq <= 0 || a->Hkv <= 0 || a->Hq % a->Hkv || a->D <= 0 || a->b <= 0) return PKVO_EINVAL;
    for (int s = 0; s < a->S; ++s)
        if (a->seq_lens[s] < 0 || (int64_t)a->seq_lens[s] > (int64_t)a->MB * a->b) return PKVO_EINVAL;
    return PKVO_OK;
}

/* The plain definition [P3 4.4; P1 "逻辑块到物理块的映射转换" step 4]: for each
 * sequence s and query head i, gather token t's key and value through
 * block_tables[s][t / b] at offset t % b, then
 *     out[s][i] = sum_t softmax_t(scale * q.k_t) * v_t
 * over the seq_lens[s] tokens.  out is float64 [S][Hq][D].  Returns 0, or 1 on
 * an invalid argument or block id. */
int pkvo_paged_decode(const void* q, int q_dtype, int S, int Hq,
                      const void* k_pool, const void* v_pool, int kv_dtype,
                      int NB, int b, int Hkv, int D, double k_scale, double v_scale,
                      const int32_t* block_tables, int MB, const int32_t* seq_lens,
                      double scale, double* out) {
    pkvo_args a = {q, q_dtype, S, Hq, k_pool, v_pool, kv_dtype, NB, b, Hkv, D,
                   k_scale, v_scale, block_tables, MB, seq_lens, scale};
    if (check_args(&a)) return PKVO_EINVAL;
    int status = PKVO_OK;
    int64_t rows = (int64_t)S * Hq;
#pragma omp parallel for schedule(dynamic, 1)
    for (int64_t r = 0; r < rows; ++r) {
        int s = (int)(r / Hq), i = (int)(r % Hq);
        int L = seq_lens[s];
        double* o = out + r * D;
        for (int d = 0; d < D; ++d) o[d] = 0.0;
        if (L == 0) continue;
        double* sc = (double*)malloc(sizeof(double) * (size_t)L);
        if (scores_range(&a, s, i, 0, L, sc)) {
#pragma omp atomic write
            status = PKVO_EINVAL;
            free(sc);
            continue;
        }
        double m = -INFINITY;
        for (int t = 0; t < L; ++t) m = sc[t] > m ? sc[t] : m;
        double sum = 0.0;
        for (int t = 0; t < L; ++t) { sc[t] = exp(sc[t] - m); sum += sc[t]; }
        weighted_v(&a, s, i, 0, L, sc, o);
        for (int d = 0; d < D; ++d) o[d] /= sum;
        free(sc);
    }
    return status;
}

/* Paged prefill attention (causal, multi-query).  Prefill processes a
 * prompt's tokens and writes their KV into the blocks; chunked prefill splits
 * a long prompt into chunks of at most a token budget that run in successive
 * iterations ([P1] "PagedAttention 内存管理与核心数据结构": prefill then decode;
 * [P1] scheduling section on chunked prefill).  Each query token therefore
 * attends to every earlier token of its sequence -- the context already in
 * the pool from earlier chunks -- and to the tokens of its own chunk up to
 * and including itself.
 *
 * Sequence s owns the query rows [query_start[s], query_start[s+1]) of q
 * ([T][Hq][D]); n_s = query_start[s+1] - query_start[s] new tokens whose KV
 * is already in the pool, at the last n_s of its seq_lens[s] positions.  Row
 * j is at position p = seq_lens[s] - n_s + j and
 *     out[query_start[s] + j][i] = sum_{t <= p} softmax_t(scale * q.k_t) * v_t
 * with keys and values gathered through block_tables[s] as in decode.  Rows
 * outside every sequence's range are left at zero.  Returns 1 on an invalid
 * argument (n_s > seq_lens[s], a decreasing or out-of-range query_start, a
 * block id outside the pool). */
int pkvo_paged_prefill(const void* q, int q_dtype, int T, int Hq, int S, const int32_t* query_start,
                       const void* k_pool, const void* v_pool, int kv_dtype,
                       int NB, int b, int Hkv, int D, double k_scale, double v_scale,
                       const int32_t* block_tables, int MB, const int32_t* seq_lens,
                       double scale, double* out) {
    pkvo_args a = {q, q_dtype, S, Hq, k_pool, v_pool, kv_dtype, NB, b, Hkv, D,
                   k_scale, v_scale, block_tables, MB, seq_lens, scale};
    if (check_args(&a) || T < 0) return PKVO_EINVAL;
    if (S > 0 && query_start[0] < 0) return PKVO_EINVAL;
    for (int s = 0; s < S; ++s) {
        int n = query_start[s + 1] - query_start[s];
        if (n < 0 || query_start[s + 1] > T || n > seq_lens[s]) return PKVO_EINVAL;
    }
    memset(out, 0, sizeof(double) * (size_t)T * Hq * D);
    int G = Hq / Hkv;
    int status = PKVO_OK;
    int64_t rows = (int64_t)T * Hq;
#pragma omp parallel for schedule(dynamic, 4)
    for (int64_t r = 0; r < rows; ++r) {
        int tok = (int)(r / Hq), i = (int)(r % Hq), h = i / G;
        int s = -1;
        for (int c = 0; c < S; ++c)
            if (tok >= query_start[c] && tok < query_start[c + 1]) { s = c; break; }
        if (s < 0) continue;
        int n = query_start[s + 1] - query_start[s];
        int p = seq_lens[s] - n + (tok - query_start[s]);   /* this token's position */
        int nk = p + 1;                                      /* keys 0..p */
        double* qrow = (double*)malloc(sizeof(double) * (size_t)D);
        double* sc = (double*)malloc(sizeof(double) * (size_t)nk);
        for (int d = 0; d < D; ++d) qrow[d] = elem_to_double(q, q_dtype, r * D + d);
        int bad = 0;
        for (int t = 0; t < nk && !bad; ++t) {
            int32_t blk = block_tables[(int64_t)s * MB + t / b];
            if (blk < 0 || blk >= NB) { bad = 1; break; }
            double dot = 0.0;
            for (int d = 0; d < D; ++d)
                dot += qrow[d] * elem_to_double(k_pool, kv_dtype, pool_index(blk, h, t % b, d, Hkv, b, D)) * k_scale;
            sc[t] = scale * dot;
        }
        if (bad) {
#pragma omp atomic write
            status = PKVO_EINVAL;
            free(qrow); free(sc);
            continue;
        }
        double m = -INFINITY;
        for (int t = 0; t < nk; ++t) m = sc[t] > m ? sc[t] : m;
        double sum = 0.0;
        for (int t = 0; t < nk; ++t) { sc[t] = exp(sc[t] - m); sum += sc[t]; }
        double* o = out + r * D;
        for (int t = 0; t < nk; ++t) {
            int32_t blk = block_tables[(int64_t)s * MB + t / b];
            for (int d = 0; d < D; ++d)
                o[d] += sc[t] * elem_to_double(v_pool, kv_dtype, pool_index(blk, h, t % b, d, Hkv, b, D)) * v_scale;
        }
        for (int d = 0; d < D; ++d) o[d] /= sum;
        free(qrow); free(sc);
    }
    return status;
}

/* Split-K form of the same computation.  The pages give only the partition
 * axis of the launch grid (openEuler essay, section "PagedAttention：把操作系统的
 * 分页搬上 GPU": grid (num_heads, num_seqs, max_num_partitions)); the reduce is
 * the standard log-sum-exp identity.  Partition p covers tokens
 * [p*P, min(L, (p+1)*P)).  For each (s, i, p) it writes
 *     m[s][i][p] = max score,  l[s][i][p] = sum_t exp(score_t - m),
 *     o[s][i][p][:] = sum_t exp(score_t - m) v_t / l
 * and for a partition with no tokens m = -inf, l = 0, o = 0.  NP is the
 * partition count of the arrays. */
int pkvo_paged_decode_partials(const void* q, int q_dtype, int S, int Hq,
                               const void* k_pool, const void* v_pool, int kv_dtype,
                               int NB, int b, int Hkv, int D, double k_scale, double v_scale,
                               const int32_t* block_tables, int MB, const int32_t* seq_lens,
                               double scale, int P, int NP, double* m_out, double* l_out, double* o_out) {
    pkvo_args a = {q, q_dtype, S, Hq, k_pool, v_pool, kv_dtype, NB, b, Hkv, D,
                   k_scale, v_scale, block_tables, MB, seq_lens, scale};
    if (check_args(&a) || P <= 0) return PKVO_EINVAL;
    for (int s = 0; s < S; ++s)
        if ((seq_lens[s] + P - 1) / P > NP) return PKVO_EINVAL;
    int status = PKVO_OK;
    int64_t rows = (int64_t)S * Hq * NP;
#pragma omp parallel for schedule(dynamic, 1)
    for (int64_t r = 0; r < rows; ++r) {
        int p = (int)(r % NP);
        int64_t si = r / NP;
        int s = (int)(si / Hq), i = (int)(si % Hq);
        int L = seq_lens[s];
        int t0 = p * P, t1 = (p + 1) * P < L ? (p + 1) * P : L;
        double* o = o_out + r * D;
        for (int d = 0; d < D; ++d) o[d] = 0.0;
        m_out[r] = -INFINITY;
        l_out[r] = 0.0;
        if (t0 >= t1) continue;
        double* sc = (double*)malloc(sizeof(double) * (size_t)(t1 - t0));
        if (scores_range(&a, s, i, t0, t1, sc)) {
#pragma omp atomic write
            status = PKVO_EINVAL;
            free(sc);
            continue;
        }
        double m = -INFINITY;
        for (int t = 0; t < t1 - t0; ++t) m = sc[t] > m ? sc[t] : m;
        double sum = 0.0;
        for (int t = 0; t < t1 - t0; ++t) { sc[t] = exp(sc[t] - m); sum += sc[t]; }
        weighted_v(&a, s, i, t0, t1, sc, o);
        for (int d = 0; d < D; ++d) o[d] /= sum;
        m_out[r] = m;
        l_out[r] = sum;
        free(sc);
    }
    return status;
}

/* Log-sum-exp merge of R rows of NP partials each:
 *     M = max_p m_p,  w_p = l_p exp(m_p - M),  out = sum_p w_p o_p / sum_p w_p;
 * partitions with l_p = 0 are skipped; a row with no tokens gives zeros. */
void pkvo_lse_merge(int64_t R, int NP, int D, const double* m, const double* l,
                    const double* o, double* out) {
    for (int64_t r = 0; r < R; ++r) {
        double M = -INFINITY;
        for (int p = 0; p < NP; ++p)
            if (l[r * NP + p] > 0.0 && m[r * NP + p] > M) M = m[r * NP + p];
        double wsum = 0.0;
        double* dst = out + r * D;
        for (int d = 0; d < D; ++d) dst[d] = 0.0;
        for (int p = 0; p < NP; ++p) {
            double lp = l[r * NP + p];
            if (lp <= 0.0) continue;
            double w = lp * exp(m[r * NP + p] - M);
            wsum += w;
            for (int d = 0; d < D; ++d) dst[d] += w * o[(r * NP + p) * D + d];
        }
        if (wsum > 0.0)
            for (int d = 0; d < D; ++d) dst[d] /= wsum;
    }
}

/* ----------------------------------------------------------------- append */

/* Slot-mapped write of this step's new keys and values [P3 4.3 step 2: "allocate
 * a new block -> update the block table -> write the KV"; P1 prefill/decode
 * paragraph: each decode step appends its KV vector to GPU memory].  For token
 * t with slot = slot_mapping[t] >= 0: blk = slot / b, off = slot % b, and for
 * every KV head h, K[blk][h][off][:] = k[t][h][:] (same for V).  When the cache
 * is fp8 and the input is f16/bf16, each element is stored as
 * e4m3(binary32(x) / binary32(scale)).  A slot outside [0, NB*b) is an error
 * (returns 1, nothing written for that token).  Tokens are written in order. */
int pkvo_append(const void* k, const void* v, int in_dtype, int T, const int64_t* slot_mapping,
                void* k_pool, void* v_pool, int kv_dtype, int NB, int b, int Hkv, int D,
                float k_scale, float v_scale) {
    int status = PKVO_OK;
    if (kv_dtype != in_dtype && kv_dtype != PKVO_E4M3) return PKVO_EINVAL;
    int eb = elem_bytes(kv_dtype);
    for (int t = 0; t < T; ++t) {
        int64_t slot = slot_mapping[t];
        if (slot < 0) continue;
        if (slot >= (int64_t)NB * b) { status = PKVO_EINVAL; continue; }
        int64_t blk = slot / b;
        int off = (int)(slot % b);
        for (int h = 0; h < Hkv; ++h) {
            for (int d = 0; d < D; ++d) {
                int64_t src = ((int64_t)t * Hkv + h) * D + d;
                int64_t dst = pool_index(blk, h, off, d, Hkv, b, D);
                if (kv_dtype == in_dtype) {
                    memcpy((char*)k_pool + dst * eb, (const char*)k + src * eb, (size_t)eb);
                    memcpy((char*)v_pool + dst * eb, (const char*)v + src * eb, (size_t)eb);
                } else {
                    float kx = (float)elem_to_double(k, in_dtype, src);
                    float vx = (float)elem_to_double(v, in_dtype, src);
                    float kq = kx / k_scale;   /* binary32 division */
                    float vq = vx / v_scale;
                    ((uint8_t*)k_pool)[dst] = pkvo_e4m3_encode(kq);
                    ((uint8_t*)v_pool)[dst] = pkvo_e4m3_encode(vq);
                }
            }
        }
    }
    return status;
}

/* ------------------------------------------------------------ copy blocks */

/* Copy-on-write block copy [P4 "Prefix Caching 与 Copy-on-Write": a shared block
 * is copied only when it is about to be modified; P1 "append" primitive].  For
 * each pair (src, dst) every byte of K[src] and V[src] (all KV heads, all b
 * slots) is copied to K[dst] and V[dst], pairs in order.  An id outside
 * [0, NB) is an error (returns 1, that pair skipped). */
int pkvo_copy_blocks(void* k_pool, void* v_pool, int kv_dtype, int NB, int b, int Hkv, int D,
                     const int32_t* pairs, int num_pairs) {
    int status = PKVO_OK;
    int64_t block_bytes = (int64_t)Hkv * b * D * elem_bytes(kv_dtype);
    for (int p = 0; p < num_pairs; ++p) {
        int32_t src = pairs[2 * p], dst = pairs[2 * p + 1];
        if (src < 0 || src >= NB || dst < 0 || dst >= NB) { status = PKVO_EINVAL; continue; }
        memmove((char*)k_pool + dst * block_bytes, (char*)k_pool + src * block_bytes, (size_t)block_bytes);
        memmove((char*)v_pool + dst * block_bytes, (char*)v_pool + src * block_bytes, (size_t)block_bytes);
    }
    return status;
}

int pkvo_num_threads(void) {
#ifdef _OPENMP
    return omp_get_max_threads();
#else
    return 1;
#endif
}

/* Threads the OpenMP loops above use from now on (at least 1); timing aid
 * only, the results do not depend on it. */
void pkvo_set_num_threads(int n) {
#ifdef _OPENMP
    omp_set_num_threads(n > 0 ? n : 1);
#else
    (void)n;
#endif
}
