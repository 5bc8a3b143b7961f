// pkv_decode_impl.cuh -- paged decode attention kernels (included by one
// translation unit per element-type family).
//
// What is computed ("vLLM：大语言模型推理与服务库" section 4.4; "vLLM 高性能大语言
// 模型推理引擎深度技术评估与分布式架构展望", "逻辑块到物理块的映射转换" step 4):
// for each sequence and query head, the keys and values of the sequence's
// tokens are gathered in place through its block table, and
//     out = sum_t softmax_t(scale * q . k_t) v_t .
//
// GB300 design (replacing the pages' one-warp-per-block CUDA-core kernel
// over the [blocks, heads, head_size/x, block_size, x] key layout):
//  * pool layout [NB][Hkv][16][D]: the (block, kv head) tile of K (and of V)
//    is one contiguous run (4 KiB for bf16 at D = 128), moved into shared
//    memory by a single 1-D TMA bulk copy (cp.async.bulk) that completes on
//    an mbarrier; no per-thread address generation for the gather;
//  * one CTA per (partition, kv head, sequence); its NW warps take the
//    partition's blocks round-robin, each warp with a private NST-stage
//    copy pipeline and its own online softmax, merged across warps at the
//    end (no CTA-wide barrier inside the loop);
//  * GQA: the G = Hq / Hkv query heads that share a KV head are handled by
//    the same warp, so each KV tile is read from HBM once per KV head;
//  * inside a warp each half-warp takes one token of a pair, each lane a
//    D/16-element slice of the row (16-byte vector reads of shared memory
//    for bf16 D = 128); dot products are reduced with a shuffle
//    reduce-scatter (8G partial sums over 16 lanes cost 8G - 1 shuffles,
//    not 4 * 8G);
//  * scores are kept in the log2 domain (q pre-multiplied by
//    scale * log2(e) * k_scale) so the softmax uses exp2;
//  * long contexts are split into partitions of P tokens (the pages' third
//    grid axis); a partition writes (m, l, o/l) and a separate log-sum-exp
//    merge kernel combines them.
#pragma once

#include <cfloat>
#include <cstdint>

#include "pkv_append.cuh"
#include "pkv_device.cuh"

namespace pkv {

constexpr unsigned kFull = 0xffffffffu;

// Shuffle reduce-scatter over the 16 lanes of a half-warp (xor masks
// MASK, MASK/2, ..., 1).  While more than one value is held, each step sends
// half the values to the partner and keeps the other half, so lane li ends
// up holding the full sum for the original indices [off, off + N/16) with
// off = li * N / 16; once a single value is left the remaining steps are
// plain all-reduce steps.
template <int N, int MASK>
__device__ __forceinline__ void reduce_scatter(float* v, int li) {
    if constexpr (MASK > 0) {
        if constexpr (N > 1) {
            const bool upper = (li & MASK) != 0;
#pragma unroll
            for (int k = 0; k < N / 2; ++k) {
                const float send = upper ? v[k] : v[k + N / 2];
                const float keep = upper ? v[k + N / 2] : v[k];
                v[k] = keep + __shfl_xor_sync(kFull, send, MASK);
            }
            reduce_scatter<N / 2, MASK / 2>(v, li);
        } else {
            v[0] += __shfl_xor_sync(kFull, v[0], MASK);
            reduce_scatter<1, MASK / 2>(v, li);
        }
    }
}

template <int D, typename KT, int NW, int NST>
struct DecodeSmem {
    static constexpr int kTile = kBlockSize * D * KT::bytes;  // one (block, head) tile
    static constexpr int kStage = 2 * kTile;                  // K tile + V tile
    static constexpr int kStagesBytes = NW * NST * kStage;
    static constexpr int kBarOffset = kStagesBytes;
    static constexpr int kPhysOffset = kBarOffset + NW * NST * 8;
    static constexpr int kPOffset = kPhysOffset + NW * NST * 4;
    template <int G>
    static constexpr int bytes() {
        return kPOffset + NW * kBlockSize * G * 4;
    }
};

// This CTA's (partition, KV head, sequence): from the grid, or from the
// host's work list (unit = s * (NP - part_base) + partition, KV head
// fastest).  A unit outside the batch sets PKV_DEVERR_SEQ_LEN; false: skip.
// With join_primary the grid's extra z-layer holds no units: its CTA
// (0, 0, S) waits there for the programmatic primary grid to complete.
__device__ __forceinline__ bool decode_unit(const DecodeParams& p, int& part, int& h, int& s) {
    if (!p.work) {
        part = blockIdx.x;
        h = blockIdx.y;
        s = blockIdx.z;
        if (s < p.S) return true;
        if (part == 0 && h == 0) wait_primary_grid();
        return false;
    }
    const int64_t lin = blockIdx.x;
    const int u = __ldg(p.work + lin / p.Hkv);
    const int npl = p.NP - p.part_base;
    h = static_cast<int>(lin % p.Hkv);
    if (u < 0 || static_cast<int64_t>(u) >= static_cast<int64_t>(p.S) * npl) {
        if (threadIdx.x == 0) report(p.err, PKV_DEVERR_SEQ_LEN);
        return false;
    }
    s = u / npl;
    part = u % npl;
    return true;
}

template <int D, int G, typename KT, typename QT, int NW, int NST>
__global__ void __launch_bounds__(NW * 32) decode_kernel(const DecodeParams p) {
    constexpr int VEC = D / 16;               // elements of a row per lane
    constexpr int VBYTES = VEC * KT::bytes;   // bytes of a row slice per lane
    constexpr int N = 8 * G;                  // partial scores per lane per block
    constexpr int NR = N >= 16 ? N / 16 : 1;  // scores held after the reduce-scatter
    using SM = DecodeSmem<D, KT, NW, NST>;
    constexpr int TILE = SM::kTile;
    constexpr int STAGE = SM::kStage;
    static_assert(VBYTES == 4 || VBYTES == 8 || VBYTES == 16, "row slice must be 4, 8 or 16 bytes");

    extern __shared__ __align__(128) unsigned char smem[];

    const int warp = threadIdx.x >> 5, lane = threadIdx.x & 31;
    allow_dependent_launch();  // the merge may stage its CTAs behind this grid's last wave
    const int hf = lane >> 4, li = lane & 15;
    int part, h, s;
    if (!decode_unit(p, part, h, s)) return;

    // Sequence length, clamped to the block table's reach and to the
    // partitions this launch covers; the sequence's own range starts after
    // its shared prefix (cascade decode) or at 0.
    int L = __ldg(p.seq_lens + s);
    const int Lcap = p.MB * kBlockSize;
    bool bad = L < 0 || L > Lcap;
    L = L < 0 ? 0 : (L > Lcap ? Lcap : L);
    const int start = own_start(p.seq_group, p.group_blocks, s, L, &bad);
    int Lown = L - start;
    if (Lown > (p.NP - p.part_base) * p.P) {
        bad = true;
        Lown = (p.NP - p.part_base) * p.P;
        L = start + Lown;
    }
    if (bad && threadIdx.x == 0 && part == 0 && h == 0) report(p.err, PKV_DEVERR_SEQ_LEN);
    const int nparts = Lown > 0 ? (Lown + p.P - 1) / p.P : (p.cascade ? 0 : 1);
    if (part >= nparts) return;
    const int t0 = start + part * p.P;
    const int t1 = min(L, t0 + p.P);
    const int j0 = t0 / kBlockSize;
    const int nblk = (t1 + kBlockSize - 1) / kBlockSize - j0;
    const int nb_w = warp < nblk ? (nblk - warp + NW - 1) / NW : 0;
    // fused append: the warp that streams the partition's last block writes
    // the new token's row just before copying that block
    const bool append_here = p.slots && t1 == L && !bad && nblk > 0 && warp == (nblk - 1) % NW;
    const FusedRow frow = fused_prefetch(p, s, h, L, append_here);

    unsigned char* wbase = smem + warp * NST * STAGE;
    uint64_t* bars = reinterpret_cast<uint64_t*>(smem + SM::kBarOffset) + warp * NST;
    volatile int* stage_phys = reinterpret_cast<int*>(smem + SM::kPhysOffset) + warp * NST;
    float* pbuf = reinterpret_cast<float*>(smem + SM::kPOffset) + warp * kBlockSize * G;

    const int32_t* bt = p.block_tables + static_cast<int64_t>(s) * p.MB + j0 + warp;
    const unsigned char* kpool = static_cast<const unsigned char*>(p.k_cache);
    const unsigned char* vpool = static_cast<const unsigned char*>(p.v_cache);
    const uint64_t pol = policy_evict_first();

    if (lane == 0) {
#pragma unroll
        for (int i = 0; i < NST; ++i) mbar_init(&bars[i], 1);
        mbar_init_fence();
    }
    __syncwarp();

    // Lane k of `tbl` holds the block id of this warp's block (window + k).
    int tbl = -1;
    int k_issue = 0;
    auto issue_next = [&]() {  // warp-uniform call
        if ((k_issue & 31) == 0) {
            const int k = k_issue + lane;
            tbl = k < nb_w ? __ldg(bt + static_cast<int64_t>(k) * NW) : -1;
        }
        const int phys = __shfl_sync(kFull, tbl, k_issue & 31);
        const int stage = k_issue % NST;
        if (append_here && k_issue == nb_w - 1) {
            fused_commit<KT>(p, h, frow);
            __syncwarp();
        }
        if (lane == 0) {
            stage_phys[stage] = phys;
            if (phys >= 0 && phys < p.NB) {
                const int64_t off = (static_cast<int64_t>(phys) * p.Hkv + h) * TILE;
                mbar_arrive_expect_tx(&bars[stage], 2 * TILE);
                bulk_g2s(wbase + stage * STAGE, kpool + off, TILE, &bars[stage], pol);
                bulk_g2s(wbase + stage * STAGE + TILE, vpool + off, TILE, &bars[stage], pol);
            } else {
                report(p.err, PKV_DEVERR_BLOCK_ID);
                mbar_arrive_expect_tx(&bars[stage], 0);
            }
        }
        ++k_issue;
    };

    // Query rows of the G heads, this lane's slice, pre-scaled to log2 units.
    float qf[G][VEC];
    {
        const unsigned char* qb = static_cast<const unsigned char*>(p.q);
#pragma unroll
        for (int g = 0; g < G; ++g) {
            const int64_t row = static_cast<int64_t>(s) * p.Hq + h * G + g;
            uint32_t w[VEC / 2];
            load_words<VEC * 2>(qb + (row * D + li * VEC) * 2, w);
            Unpack<QT, VEC>::run(w, qf[g]);
#pragma unroll
            for (int e = 0; e < VEC; ++e) qf[g][e] *= p.qk_scale;
        }
    }

    for (int i = 0; i < NST && k_issue < nb_w; ++i) issue_next();

    float m[G], acc[G][VEC];
    float lsum = 0.f;  // this lane's share of the softmax denominator of head g_h
#pragma unroll
    for (int g = 0; g < G; ++g) {
        m[g] = -INFINITY;
#pragma unroll
        for (int e = 0; e < VEC; ++e) acc[g][e] = 0.f;
    }
    // Indices held after the reduce-scatter: one head, NR consecutive token pairs.
    const int off = N >= 16 ? li * (N / 16) : (li >> 1);
    const int g_h = off / 8;
    const bool owner = N >= 16 || (li & 1) == 0;  // G = 1: lanes li, li^1 hold the same score

    bool aborted = false;
    for (int k = 0; k < nb_w; ++k) {
        const int stage = k % NST;
        if (!mbar_wait(&bars[stage], (k / NST) & 1)) {
            if (lane == 0) report(p.err, PKV_DEVERR_TIMEOUT);
            aborted = true;
            break;
        }
        const int phys = stage_phys[stage];
        const int tok0 = (j0 + warp + k * NW) * kBlockSize;
        const int nvalid = min(kBlockSize, t1 - tok0);
        if (phys >= 0 && phys < p.NB) {
            const unsigned char* kt = wbase + stage * STAGE;
            const unsigned char* vt = kt + TILE;
            // ---- scores: half-warp hf takes tokens 2*jj + hf
            float sc[N];
#pragma unroll
            for (int jj = 0; jj < 8; ++jj) {
                const int t = 2 * jj + hf;
                uint32_t w[VBYTES / 4];
                load_words<VBYTES>(kt + (t * D + li * VEC) * KT::bytes, w);
                float kf[VEC];
                Unpack<KT, VEC>::run(w, kf);
#pragma unroll
                for (int g = 0; g < G; ++g) {
                    float a = 0.f;
#pragma unroll
                    for (int e = 0; e < VEC; ++e) a = fmaf(qf[g][e], kf[e], a);
                    sc[g * 8 + jj] = a;
                }
            }
            reduce_scatter<N, 8>(sc, li);
            if (nvalid < kBlockSize) {
#pragma unroll
                for (int r = 0; r < NR; ++r) {
                    const int t = 2 * ((off + r) & 7) + hf;
                    if (t >= nvalid) sc[r] = -INFINITY;
                }
            }
            // ---- block max per head, new running max
            float bm = sc[0];
#pragma unroll
            for (int r = 1; r < NR; ++r) bm = fmaxf(bm, sc[r]);
#pragma unroll
            for (int mask = 1; mask < 16 / G; mask <<= 1) bm = fmaxf(bm, __shfl_xor_sync(kFull, bm, mask));
            bm = fmaxf(bm, __shfl_xor_sync(kFull, bm, 16));
            float alpha[G];
#pragma unroll
            for (int g = 0; g < G; ++g) {
                const float bmg = __shfl_sync(kFull, bm, g * (16 / G));
                const float mn = fmaxf(m[g], bmg);
                alpha[g] = exp2f(m[g] - mn);
                m[g] = mn;
            }
            // ---- probabilities of the held scores -> per-warp buffer
            float m_h = m[0], a_h = alpha[0];
#pragma unroll
            for (int g = 1; g < G; ++g)
                if (g == g_h) {
                    m_h = m[g];
                    a_h = alpha[g];
                }
            float ps = 0.f;
#pragma unroll
            for (int r = 0; r < NR; ++r) {
                const float pr = exp2f(sc[r] - m_h);
                ps += pr;
                const int t = 2 * ((off + r) & 7) + hf;
                pbuf[t * G + g_h] = pr;
            }
            lsum = lsum * a_h + (owner ? ps : 0.f);
            __syncwarp();
            // ---- acc = alpha * acc + sum_t p_t v_t
#pragma unroll
            for (int g = 0; g < G; ++g)
#pragma unroll
                for (int e = 0; e < VEC; ++e) acc[g][e] *= alpha[g];
#pragma unroll
            for (int jj = 0; jj < 8; ++jj) {
                const int t = 2 * jj + hf;
                if (t < nvalid) {
                    uint32_t w[VBYTES / 4];
                    load_words<VBYTES>(vt + (t * D + li * VEC) * KT::bytes, w);
                    float vf[VEC];
                    Unpack<KT, VEC>::run(w, vf);
                    float pp[G];
#pragma unroll
                    for (int g = 0; g < G; ++g) pp[g] = pbuf[t * G + g];
#pragma unroll
                    for (int g = 0; g < G; ++g)
#pragma unroll
                        for (int e = 0; e < VEC; ++e) acc[g][e] = fmaf(pp[g], vf[e], acc[g][e]);
                }
            }
        }
        __syncwarp();
        if (k_issue < nb_w) issue_next();
    }

    if (aborted) {
        // Let copies still in flight land before the shared memory is reused.
        for (int k = 0; k < NST; ++k) {
            const int kk = k_issue - 1 - k;
            if (kk < 0) break;
            (void)mbar_wait(&bars[kk % NST], (kk / NST) & 1);
        }
    }

    // ---- warp state: combine half-warps, reduce the denominator per head
#pragma unroll
    for (int g = 0; g < G; ++g)
#pragma unroll
        for (int e = 0; e < VEC; ++e) acc[g][e] += __shfl_xor_sync(kFull, acc[g][e], 16);
#pragma unroll
    for (int mask = 1; mask < 16 / G; mask <<= 1) lsum += __shfl_xor_sync(kFull, lsum, mask);
    lsum += __shfl_xor_sync(kFull, lsum, 16);

    float* ws = reinterpret_cast<float*>(wbase);  // [G] m, [G] l, [G][D] acc
    __syncwarp();
#pragma unroll
    for (int g = 0; g < G; ++g) {
        const float lg = __shfl_sync(kFull, lsum, g * (16 / G));
        if (lane == 0) {
            ws[g] = aborted ? -INFINITY : m[g];
            ws[G + g] = aborted ? 0.f : lg;
        }
        if (hf == 0) {
#pragma unroll
            for (int e = 0; e < VEC; ++e) ws[2 * G + g * D + li * VEC + e] = aborted ? 0.f : acc[g][e];
        }
    }
    __syncthreads();

    // ---- merge the NW warp states; write the output row or the partials
    for (int idx = threadIdx.x; idx < G * D; idx += NW * 32) {
        const int g = idx / D, d = idx % D;
        float M = -INFINITY;
#pragma unroll
        for (int w = 0; w < NW; ++w) M = fmaxf(M, reinterpret_cast<float*>(smem + w * NST * STAGE)[g]);
        float num = 0.f, den = 0.f;
        if (M != -INFINITY) {
#pragma unroll
            for (int w = 0; w < NW; ++w) {
                const float* wsw = reinterpret_cast<float*>(smem + w * NST * STAGE);
                const float mw = wsw[g];
                if (mw != -INFINITY) {
                    const float sc = exp2f(mw - M);
                    den = fmaf(sc, wsw[G + g], den);
                    num = fmaf(sc, wsw[2 * G + g * D + d], num);
                }
            }
        }
        const float o = den > 0.f ? num / den * p.v_scale : 0.f;
        const int64_t row = static_cast<int64_t>(s) * p.Hq + h * G + g;
        if (nparts == 1 && !p.cascade) {
            reinterpret_cast<typename QT::storage*>(p.out)[row * D + d] = from_float<QT>(o);
        } else {
            const int64_t prow = row * p.NP + p.part_base + part;
            p.part_o[prow * D + d] = o;
            if (d == 0) {
                p.part_m[prow] = M;
                p.part_l[prow] = den;
            }
        }
    }
}

// ------------------------------------------------------------- launchers
constexpr int kDecodeWarps = 4;
// Shared-memory budget per CTA for the copy stages: two CTAs per SM.
constexpr int kStageBudget = 96 * 1024;

template <int D, typename KT>
constexpr int decode_stages() {
    constexpr int st = kStageBudget / (kDecodeWarps * 2 * kBlockSize * D * KT::bytes);
    return st < 2 ? 2 : (st > 8 ? 8 : st);
}

template <int D, int G, typename KT, typename QT>
cudaError_t launch_decode_t(const DecodeParams& p, cudaStream_t st) {
    constexpr int NW = kDecodeWarps;
    constexpr int NST = decode_stages<D, KT>();
    constexpr int SMEM = DecodeSmem<D, KT, NW, NST>::template bytes<G>();
    auto kern = decode_kernel<D, G, KT, QT, NW, NST>;
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
    const dim3 grid = p.work ? dim3(static_cast<unsigned>(static_cast<int64_t>(p.num_work) * p.Hkv))
                             : dim3(p.NP - p.part_base, p.Hkv, p.S + (p.join_primary ? 1 : 0));  // this launch's partitions
    return launch_maybe_pdl(p.join_primary != 0 && !p.work, kern, grid, dim3(NW * 32), SMEM, st, p);
}

template <typename KT, typename QT>
cudaError_t launch_decode_family(const DecodeParams& p, int G, cudaStream_t st) {
    if (p.D == 128) {
        switch (G) {
        case 1: return launch_decode_t<128, 1, KT, QT>(p, st);
        case 2: return launch_decode_t<128, 2, KT, QT>(p, st);
        case 4: return launch_decode_t<128, 4, KT, QT>(p, st);
        case 8: return launch_decode_t<128, 8, KT, QT>(p, st);
        }
    } else if (p.D == 64) {
        switch (G) {
        case 1: return launch_decode_t<64, 1, KT, QT>(p, st);
        case 2: return launch_decode_t<64, 2, KT, QT>(p, st);
        case 4: return launch_decode_t<64, 4, KT, QT>(p, st);
        case 8: return launch_decode_t<64, 8, KT, QT>(p, st);
        }
    }
    return cudaErrorInvalidValue;
}

}  // namespace pkv
