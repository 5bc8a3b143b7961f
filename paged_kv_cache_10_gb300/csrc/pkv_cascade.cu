// pkv_cascade.cu -- shared-prefix (cascade) decode attention.
//
// When several sequences share their leading physical blocks (prefix
// sharing and parallel sampling: "vLLM 深度解析：从 PagedAttention 到生产部署",
// "Prefix Caching 与 Copy-on-Write"; "vLLM 高性能大语言模型推理引擎深度技术评估
// 与分布式架构展望", "束搜索与并行采样的三大调度原语": fork shares the parent's
// physical blocks), plain decode reads the shared blocks once per sequence.
// Cascade decode splits every member's attention into the shared part and
// its own part, which are combined exactly by the log-sum-exp merge:
//
//   1. cascade_prefix_kernel: for each group, KV head and 256-token prefix
//      partition, the query heads of ALL members (members x G rows on the
//      MMA's M dimension) attend to the shared blocks, which are read once
//      per CTA of 64 rows; partials go to partition indices [0, NPP);
//   2. the regular decode kernel attends each sequence's own tokens (from
//      the end of its group's prefix), partials at indices NPP + p;
//   3. the merge kernel combines prefix and own partials of every row.
//
// The result is the same function as pkv_paged_attention_decode.
#include <cstdint>

#include "pkv_decode_mma.cuh"
#include "pkv_merge.cuh"

namespace pkv {

constexpr int kPrefixPartitionBlocks = 16;  // 256 tokens per prefix partition
constexpr int kCascadeWarps = 4;            // 4 x 16 rows per CTA
constexpr int kCascadeStages = 6;

struct CascadeParams {
    DecodeParams base;
    const int32_t* group_offsets;  // [num_groups + 1] into group_members
    const int32_t* group_members;  // batch rows, group by group
    int32_t G;
    int32_t row_chunks;  // CTAs per (group, KV head, prefix partition) along rows
    int32_t npp;         // prefix partitions (partition indices [0, npp))
};

__device__ __forceinline__ void mbar_arrive(uint64_t* bar) {
    asm volatile("mbarrier.arrive.release.cta.shared::cta.b64 _, [%0];" ::"r"(smem_addr(bar)) : "memory");
}

// 4 CTAs per SM (<= 128 registers): a group's (prefix partition, KV head,
// row chunk) tasks then fit one wave on the 152 SMs for typical groups
// instead of spilling a small second wave.
template <typename KT, typename QT, int NW, int NST>
__global__ void __launch_bounds__(NW * 32, 4)
    cascade_prefix_kernel(const CascadeParams cp, const __grid_constant__ CUtensorMap tmk,
                          const __grid_constant__ CUtensorMap tmv) {
    constexpr int D = 128;
    constexpr bool kBF = std::is_same<KT, BF16>::value;
    constexpr int TILE = kBlockSize * D * 2;  // 16-bit pools only
    constexpr int STAGE = 2 * TILE;
    const DecodeParams& p = cp.base;

    extern __shared__ unsigned char smem_raw[];
    unsigned char* smem = smem_raw + ((1024 - (smem_addr(smem_raw) & 1023)) & 1023);
    uint64_t* full = reinterpret_cast<uint64_t*>(smem + NST * STAGE);
    uint64_t* empty = full + NST;
    volatile int* stage_phys = reinterpret_cast<int*>(empty + NST);

    const int warp = threadIdx.x >> 5, lane = threadIdx.x & 31;
    const int r0 = lane >> 2, qd = lane & 3;
    const int pp = blockIdx.x, h = blockIdx.y;
    const int grp = blockIdx.z / cp.row_chunks, chunk = blockIdx.z % cp.row_chunks;
    const int G = cp.G;

    const int m0 = __ldg(cp.group_offsets + grp), m1 = __ldg(cp.group_offsets + grp + 1);
    const int rows = (m1 - m0) * G;
    const int r_cta = chunk * NW * 16;
    if (r_cta >= rows) return;
    int nb = __ldg(p.group_blocks + grp);
    if (nb < 0 || nb > p.MB) {
        if (threadIdx.x == 0 && pp == 0 && h == 0 && chunk == 0) report(p.err, PKV_DEVERR_SEQ_LEN);
        nb = nb < 0 ? 0 : p.MB;
    }
    const int b0 = pp * kPrefixPartitionBlocks;
    const int seq0 = __ldg(cp.group_members + m0);
    const bool bad_seq0 = seq0 < 0 || seq0 >= p.S;
    if (bad_seq0 && threadIdx.x == 0 && pp == 0 && h == 0 && chunk == 0) report(p.err, PKV_DEVERR_SEQ_LEN);
    if (b0 >= nb || bad_seq0) {
        // this partition lies past the group's prefix (another group's prefix
        // is longer): an empty partial for each row, so the merge reads no
        // stale workspace
        for (int r = r_cta + threadIdx.x / 32; r < min(rows, r_cta + NW * 16); r += NW) {
            const int mem = __ldg(cp.group_members + m0 + r / G);
            if (mem < 0 || mem >= p.S) continue;
            const int64_t prow = (static_cast<int64_t>(mem) * p.Hq + h * G + r % G) * p.NP + pp;
            if (lane == 0) {
                p.part_m[prow] = -INFINITY;
                p.part_l[prow] = 0.f;
            }
            for (int d = lane; d < D; d += 32) p.part_o[prow * D + d] = 0.f;
        }
        return;
    }
    const int nblk = min(nb, b0 + kPrefixPartitionBlocks) - b0;
    const int32_t* bt = p.block_tables + static_cast<int64_t>(seq0) * p.MB + b0;
    const uint64_t pol = policy_evict_last();  // the prefix is read by every row chunk

    if (threadIdx.x == 0) {
#pragma unroll
        for (int i = 0; i < NST; ++i) {
            mbar_init(&full[i], 1);
            mbar_init(&empty[i], NW);
        }
        mbar_init_fence();
    }
    __syncthreads();

    auto issue = [&](int k) {  // thread 0 only
        const int stage = k % NST;
        const int phys = __ldg(bt + k);
        stage_phys[stage] = phys;
        if (phys >= 0 && phys < p.NB) {
            const int y = (phys * p.Hkv + h) * kBlockSize;
            unsigned char* dst = smem + stage * STAGE;
            mbar_arrive_expect_tx(&full[stage], STAGE);
            tma_load_2d(dst, &tmk, 0, y, &full[stage], pol);
            tma_load_2d(dst + 2048, &tmk, 64, y, &full[stage], pol);
            tma_load_2d(dst + TILE, &tmv, 0, y, &full[stage], pol);
            tma_load_2d(dst + TILE + 2048, &tmv, 64, y, &full[stage], pol);
        } else {
            report(p.err, PKV_DEVERR_BLOCK_ID);
            mbar_arrive_expect_tx(&full[stage], 0);
        }
    };
    if (threadIdx.x == 0)
        for (int k = 0; k < NST && k < nblk; ++k) issue(k);

    // Rows of this lane: ra = (member, head) pair r_cta + 16 warp + r0, rb = ra + 8.
    const int ra = r_cta + warp * 16 + r0, rb = ra + 8;
    int64_t qrow[2] = {-1, -1};
#pragma unroll
    for (int i = 0; i < 2; ++i) {
        const int r = i ? rb : ra;
        if (r < rows) {
            const int mem = __ldg(cp.group_members + m0 + r / G);
            if (mem >= 0 && mem < p.S)
                qrow[i] = static_cast<int64_t>(mem) * p.Hq + h * G + r % G;
            else if (r % G == 0)
                report(p.err, PKV_DEVERR_SEQ_LEN);
        }
    }
    // A fragments of Q: a0 (ra, k lo), a1 (rb, k lo), a2 (ra, k hi), a3 (rb, k hi)
    uint32_t qa[8][4];
    {
        const unsigned char* qb = static_cast<const unsigned char*>(p.q);
#pragma unroll
        for (int kk = 0; kk < 8; ++kk) {
#pragma unroll
            for (int i = 0; i < 2; ++i) {
                uint32_t lo = 0u, hi = 0u;
                if (qrow[i] >= 0) {
                    const unsigned char* qr = qb + qrow[i] * D * 2;
                    lo = *reinterpret_cast<const uint32_t*>(qr + (16 * kk + 2 * qd) * 2);
                    hi = *reinterpret_cast<const uint32_t*>(qr + (16 * kk + 8 + 2 * qd) * 2);
                }
                qa[kk][i] = lo;
                qa[kk][2 + i] = hi;
            }
        }
    }

    float o[16][4];
#pragma unroll
    for (int j = 0; j < 16; ++j) o[j][0] = o[j][1] = o[j][2] = o[j][3] = 0.f;
    float m[2] = {-INFINITY, -INFINITY}, l[2] = {0.f, 0.f};

    bool aborted = false;
    for (int k = 0; k < nblk; ++k) {
        const int stage = k % NST;
        if (!mbar_wait(&full[stage], (k / NST) & 1)) {
            if (lane == 0) report(p.err, PKV_DEVERR_TIMEOUT);
            aborted = true;
            break;
        }
        const int phys = stage_phys[stage];
        if (phys >= 0 && phys < p.NB) {
            const uint32_t kts = smem_addr(smem + stage * STAGE), vts = kts + TILE;
            // ---- S = Q K^T for 16 rows x 16 tokens (n-tile j = tokens 8j..8j+7)
            // four independent accumulator chains (2 n-tiles x even/odd k-steps)
            float sa[2][4] = {{0.f, 0.f, 0.f, 0.f}, {0.f, 0.f, 0.f, 0.f}};
            {
                float sb[2][4] = {{0.f, 0.f, 0.f, 0.f}, {0.f, 0.f, 0.f, 0.f}};
                const int mat = lane >> 3, rr = lane & 7;
                const int tok = rr + 8 * (mat >> 1);
#pragma unroll
                for (int kk = 0; kk < 8; ++kk) {
                    const int ch = 2 * kk + (mat & 1);
                    uint32_t b0, b1, b2, b3;
                    ldsm_x4(kts + (ch >> 3) * 2048 + swz128(tok, ch & 7), b0, b1, b2, b3);
                    float(*acc)[4] = (kk & 1) ? sb : sa;
                    mma16816a<kBF>(acc[0], qa[kk][0], qa[kk][1], qa[kk][2], qa[kk][3], b0, b1);
                    mma16816a<kBF>(acc[1], qa[kk][0], qa[kk][1], qa[kk][2], qa[kk][3], b2, b3);
                }
#pragma unroll
                for (int j = 0; j < 2; ++j)
#pragma unroll
                    for (int c = 0; c < 4; ++c) sa[j][c] += sb[j][c];
            }
            // ---- online softmax for rows ra (c0, c1) and rb (c2, c3); prefix blocks are full
            float pr[2][4];
            float alpha[2];
#pragma unroll
            for (int i = 0; i < 2; ++i) {
                const float s0 = sa[0][2 * i] * p.qk_scale, s1 = sa[0][2 * i + 1] * p.qk_scale;
                const float s2 = sa[1][2 * i] * p.qk_scale, s3 = sa[1][2 * i + 1] * p.qk_scale;
                float bm = fmaxf(fmaxf(s0, s1), fmaxf(s2, s3));
                bm = fmaxf(bm, __shfl_xor_sync(kFull, bm, 1));
                bm = fmaxf(bm, __shfl_xor_sync(kFull, bm, 2));
                const float mn = fmaxf(m[i], bm);
                alpha[i] = mn == m[i] ? 1.f : ex2(m[i] - mn);
                m[i] = mn;
                pr[i][0] = ex2(s0 - mn);
                pr[i][1] = ex2(s1 - mn);
                pr[i][2] = ex2(s2 - mn);
                pr[i][3] = ex2(s3 - mn);
                l[i] = l[i] * alpha[i] + (pr[i][0] + pr[i][1]) + (pr[i][2] + pr[i][3]);
            }
            if (__any_sync(kFull, alpha[0] != 1.f || alpha[1] != 1.f)) {
#pragma unroll
                for (int j = 0; j < 16; ++j) {
                    o[j][0] *= alpha[0];
                    o[j][1] *= alpha[0];
                    o[j][2] *= alpha[1];
                    o[j][3] *= alpha[1];
                }
            }
            // A fragments of P straight from the S accumulators
            const uint32_t pa0 = pack2<kBF>(pr[0][0], pr[0][1]);  // ra, tokens 2qd, 2qd+1
            const uint32_t pa1 = pack2<kBF>(pr[1][0], pr[1][1]);  // rb
            const uint32_t pa2 = pack2<kBF>(pr[0][2], pr[0][3]);  // ra, tokens 8+2qd, 9+2qd
            const uint32_t pa3 = pack2<kBF>(pr[1][2], pr[1][3]);  // rb
            // ---- O += P V
            {
                const int mat = lane >> 3, rr = lane & 7;
                const int tok = rr + 8 * (mat & 1);
#pragma unroll
                for (int i = 0; i < 8; ++i) {
                    const int ch = 2 * i + (mat >> 1);
                    uint32_t b0, b1, b2, b3;
                    ldsm_x4_t(vts + (ch >> 3) * 2048 + swz128(tok, ch & 7), b0, b1, b2, b3);
                    mma16816a<kBF>(o[2 * i], pa0, pa1, pa2, pa3, b0, b1);
                    mma16816a<kBF>(o[2 * i + 1], pa0, pa1, pa2, pa3, b2, b3);
                }
            }
        }
        __syncwarp();
        if (lane == 0) mbar_arrive(&empty[stage]);
        if (threadIdx.x == 0 && k + NST < nblk) {
            if (!mbar_wait(&empty[stage], (k / NST) & 1)) {
                report(p.err, PKV_DEVERR_TIMEOUT);
                aborted = true;
            } else {
                issue(k + NST);
            }
        }
        __syncwarp();
        if (__shfl_sync(kFull, aborted ? 1 : 0, 0)) break;
    }
    if (aborted) {
        // let copies still in flight land before the CTA exits
        for (int k = 0; k < NST && k < nblk; ++k) (void)mbar_wait(&full[k], 0);
    }

    // ---- partials of this prefix partition for rows ra, rb
#pragma unroll
    for (int i = 0; i < 2; ++i) {
        l[i] += __shfl_xor_sync(kFull, l[i], 1);
        l[i] += __shfl_xor_sync(kFull, l[i], 2);
    }
#pragma unroll
    for (int i = 0; i < 2; ++i) {
        if (qrow[i] < 0) continue;
        const int64_t prow = qrow[i] * p.NP + pp;
        const bool ok = !aborted && l[i] > 0.f;
        const float inv = ok ? 1.f / l[i] : 0.f;
        if (qd == 0) {
            p.part_m[prow] = ok ? m[i] : -INFINITY;
            p.part_l[prow] = ok ? l[i] : 0.f;
        }
        float* po = p.part_o + prow * D;
#pragma unroll
        for (int j = 0; j < 16; ++j) {
            const float2 v = make_float2(o[j][2 * i] * inv * p.v_scale, o[j][2 * i + 1] * inv * p.v_scale);
            *reinterpret_cast<float2*>(po + 8 * j + 2 * qd) = v;
        }
    }
}

// Partition count of the prefix part for a group prefix of `blocks` blocks.
int prefix_partitions(int blocks) {
    return (blocks + kPrefixPartitionBlocks - 1) / kPrefixPartitionBlocks;
}

template <typename KT, typename QT>
cudaError_t launch_prefix_t(const CascadeParams& cp, int num_groups, const CUtensorMap& tk, const CUtensorMap& tv,
                            cudaStream_t st) {
    constexpr int NW = kCascadeWarps, NST = kCascadeStages;
    constexpr int SMEM = NST * 2 * (kBlockSize * 128 * 2) + NST * 20 + 1024;
    auto kern = cascade_prefix_kernel<KT, QT, NW, NST>;
    static bool configured[kMaxDevices] = {};
    int dev = 0;
    cudaError_t e = cudaGetDevice(&dev);
    if (e != cudaSuccess) return e;
    if (dev >= kMaxDevices) return cudaErrorInvalidDevice;
    if (!configured[dev]) {
        e = cudaFuncSetAttribute(kern, cudaFuncAttributeMaxDynamicSharedMemorySize, SMEM);
        if (e != cudaSuccess) return e;
        configured[dev] = true;
    }
    dim3 grid(cp.npp, cp.base.Hkv, num_groups * cp.row_chunks);
    kern<<<grid, NW * 32, SMEM, st>>>(cp, tk, tv);
    return cudaGetLastError();
}

cudaError_t launch_cascade_prefix(const CascadeParams& cp, int num_groups, int kv_dtype, const CUtensorMap& tk,
                                  const CUtensorMap& tv, cudaStream_t st) {
    if (kv_dtype == PKV_BF16) return launch_prefix_t<BF16, BF16>(cp, num_groups, tk, tv, st);
    return launch_prefix_t<F16, F16>(cp, num_groups, tk, tv, st);
}

namespace {
bool aligned16(const void* p) { return (reinterpret_cast<uintptr_t>(p) & 15u) == 0; }
int64_t cdiv(int64_t a, int64_t b) { return (a + b - 1) / b; }
}  // namespace

}  // namespace pkv

using namespace pkv;

extern "C" size_t pkv_decode_cascade_workspace_bytes(int32_t num_seqs, int32_t num_q_heads, int32_t head_size,
                                                     int32_t max_seq_len, int32_t partition_tokens,
                                                     int32_t max_group_blocks) {
    if (num_seqs < 0 || num_q_heads <= 0 || head_size <= 0 || max_seq_len < 0 || partition_tokens < 0 ||
        max_group_blocks < 0 || partition_tokens % kBlockSize)
        return 0;
    const int64_t P = partition_tokens > 0 ? partition_tokens : kAutoMinPartition;
    const int64_t NP = prefix_partitions(max_group_blocks) + (max_seq_len > 0 ? cdiv(max_seq_len, P) : 1);
    return partials_bytes(num_seqs, num_q_heads, head_size, NP);
}

extern "C" pkv_status pkv_paged_attention_decode_cascade(
    const void* q, int32_t q_dtype, int32_t num_seqs, int32_t num_q_heads, const void* k_cache, const void* v_cache,
    const pkv_cache_desc* d, const int32_t* block_tables, int32_t max_blocks_per_seq, const int32_t* seq_lens,
    int32_t max_seq_len, const int32_t* seq_group, const int32_t* group_blocks, const int32_t* group_offsets,
    const int32_t* group_members, int32_t num_groups, int32_t max_group_members, int32_t max_group_blocks, float scale,
    void* out, void* workspace, size_t ws_bytes, int32_t partition_tokens, void* stream) {
    // ---- validation (host, before any launch)
    if (!d || num_seqs < 0 || num_q_heads <= 0 || max_blocks_per_seq <= 0 || max_seq_len < 0 ||
        partition_tokens < 0 || num_groups < 0 || max_group_members < 0 || max_group_blocks < 0)
        return PKV_ERR_INVALID;
    if (d->num_blocks <= 0 || d->num_kv_heads <= 0 || d->head_size <= 0 || d->block_size <= 0)
        return PKV_ERR_INVALID;
    if (d->kv_dtype < PKV_F16 || d->kv_dtype > PKV_FP8_E4M3) return PKV_ERR_INVALID;
    if (q_dtype != PKV_F16 && q_dtype != PKV_BF16) return PKV_ERR_INVALID;
    if (num_q_heads % d->num_kv_heads || !(scale == scale)) return PKV_ERR_INVALID;
    if (static_cast<int64_t>(max_seq_len) > static_cast<int64_t>(max_blocks_per_seq) * d->block_size)
        return PKV_ERR_INVALID;
    if (max_group_blocks > max_blocks_per_seq || partition_tokens % kBlockSize) return PKV_ERR_INVALID;
    if (d->kv_dtype == PKV_FP8_E4M3 || q_dtype != d->kv_dtype) return PKV_ERR_UNSUPPORTED;
    if (d->block_size != kBlockSize || d->head_size != 128) return PKV_ERR_UNSUPPORTED;
    const int G = num_q_heads / d->num_kv_heads;
    if (G != 1 && G != 2 && G != 4 && G != 8) return PKV_ERR_UNSUPPORTED;
    if (num_seqs > 65535 || d->num_kv_heads > 65535) return PKV_ERR_UNSUPPORTED;
    if (num_seqs == 0) return PKV_OK;
    if (!q || !k_cache || !v_cache || !block_tables || !seq_lens || !out || !seq_group) return PKV_ERR_INVALID;
    if (num_groups > 0 && (!group_blocks || !group_offsets || !group_members)) return PKV_ERR_INVALID;
    if (!aligned16(q) || !aligned16(k_cache) || !aligned16(v_cache) || !aligned16(out)) return PKV_ERR_INVALID;
    const int64_t pool_rows = static_cast<int64_t>(d->num_blocks) * d->num_kv_heads * kBlockSize;
    if (pool_rows > 0x7fffffff) return PKV_ERR_UNSUPPORTED;

    const int P = partition_tokens > 0 ? partition_tokens : auto_partition(num_seqs, d->num_kv_heads, max_seq_len);
    const int npp = num_groups > 0 ? prefix_partitions(max_group_blocks) : 0;
    const int64_t nps = max_seq_len > 0 ? cdiv(max_seq_len, P) : 1;
    const int64_t NP = npp + nps;
    const int64_t row_chunks = cdiv(static_cast<int64_t>(max_group_members) * G, 16 * kCascadeWarps);
    if (NP > 0x7fffffff || static_cast<int64_t>(num_groups) * row_chunks > 65535) return PKV_ERR_UNSUPPORTED;
    const size_t need = partials_bytes(num_seqs, num_q_heads, d->head_size, NP);
    if (!workspace || ws_bytes < need || !aligned16(workspace)) return PKV_ERR_WORKSPACE;
    unsigned int* err = error_word();
    if (!err) return PKV_ERR_CUDA;

    DecodeParams p{};
    p.q = q;
    p.k_cache = k_cache;
    p.v_cache = v_cache;
    p.block_tables = block_tables;
    p.seq_lens = seq_lens;
    p.out = out;
    p.S = num_seqs;
    p.Hq = num_q_heads;
    p.Hkv = d->num_kv_heads;
    p.D = d->head_size;
    p.NB = d->num_blocks;
    p.MB = max_blocks_per_seq;
    p.P = P;
    p.NP = static_cast<int32_t>(NP);
    p.qk_scale = scale * 1.4426950408889634f;
    p.v_scale = 1.f;
    p.err = err;
    p.seq_group = seq_group;
    p.group_blocks = group_blocks;
    p.part_base = npp;
    p.cascade = 1;
    partials_layout(p, workspace);

    CUtensorMap tk, tv;
    if (!encode_pool_map(&tk, k_cache, 2, pool_rows, d->head_size) ||
        !encode_pool_map(&tv, v_cache, 2, pool_rows, d->head_size))
        return PKV_ERR_CUDA;
    cudaStream_t st = static_cast<cudaStream_t>(stream);
    cudaError_t e = cudaSuccess;
    // 1. shared prefixes
    if (npp > 0 && row_chunks > 0) {
        CascadeParams cp{p, group_offsets, group_members, G, static_cast<int32_t>(row_chunks), npp};
        e = launch_cascade_prefix(cp, num_groups, d->kv_dtype, tk, tv, st);
        if (e != cudaSuccess) return PKV_ERR_CUDA;
    }
    // 2. each sequence's own tokens
    if (G >= 2) {
        e = d->kv_dtype == PKV_BF16 ? launch_decode_mma_bf16(p, G, tk, tv, st) : launch_decode_mma_f16(p, G, tk, tv, st);
    } else {
        e = d->kv_dtype == PKV_BF16 ? launch_decode_bf16(p, G, st) : launch_decode_f16(p, G, st);
    }
    if (e != cudaSuccess) return PKV_ERR_CUDA;
    // 3. merge every row
    e = launch_merge(p, q_dtype, st);
    return e == cudaSuccess ? PKV_OK : PKV_ERR_CUDA;
}
