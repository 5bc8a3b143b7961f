// pkv_decode_mma.cuh -- tensor-core paged decode attention for grouped-query
// attention (G = Hq / Hkv in {2, 4, 8}, head_size 128).
//
// Same computation as decode_kernel ("vLLM：大语言模型推理与服务库" section 4.4:
// per query head, walk the block table, q . K -> softmax -> weighted V), same
// grid (partition, kv head, sequence) and per-warp copy pipelines, but the
// two products of a 16-token block run on the tensor cores:
//
//   S^T [16 x 16] = Q [16 x 128] . K^T [128 x 16]    (rows = query heads,
//                                                      G of 16 used)
//   O   [16 x 128] += P [16 x 16] . V [16 x 128]
//
// with mma.m16n8k16 (fp32 accumulate).  The GQA group gives an M = 16 tile
// (G real rows); the newer 5th-generation MMA needs M >= 64, i.e. >= 8x
// padding plus a tensor-memory round trip per block for the online
// softmax, while this path keeps scores, probabilities and the output
// accumulator in registers: the S^T accumulator fragment of the first
// product is exactly the A-operand fragment of the second.
//
// Tiles arrive through 2-D TMA tensor copies with the 128-byte swizzle
// (16-byte chunk c of smem row r stored at chunk c ^ (r & 7)), so the
// fragment loads below (ldmatrix for 16-bit pools; 16-byte loads for fp8)
// are free of shared-memory bank conflicts.
//
// fp8 E4M3 pools: the MMA runs in f16.  Key and value bytes are turned into
// f16 pairs in registers (hardware e4m3x2 -> f16x2 conversion, exact), with
// the contraction index permuted so that each lane reads whole 16-byte
// chunks: the k-th MMA column of lane quad member q covers head dimensions
// 32q + 4k .. 32q + 4k + 3 for keys, and output column n of n-tile j is
// head dimension 16n + j for values.  q is converted to f16 (exact in the
// normal range).
#pragma once

#include <cuda.h>

#include <type_traits>

#include "pkv_decode_impl.cuh"

namespace pkv {

// ------------------------------------------------------------ PTX wrappers
__device__ __forceinline__ void ldsm_x4(uint32_t addr, uint32_t& r0, uint32_t& r1, uint32_t& r2, uint32_t& r3) {
    asm volatile("ldmatrix.sync.aligned.m8n8.x4.shared.b16 {%0,%1,%2,%3}, [%4];"
                 : "=r"(r0), "=r"(r1), "=r"(r2), "=r"(r3)
                 : "r"(addr));
}

__device__ __forceinline__ void ldsm_x4_t(uint32_t addr, uint32_t& r0, uint32_t& r1, uint32_t& r2, uint32_t& r3) {
    asm volatile("ldmatrix.sync.aligned.m8n8.x4.trans.shared.b16 {%0,%1,%2,%3}, [%4];"
                 : "=r"(r0), "=r"(r1), "=r"(r2), "=r"(r3)
                 : "r"(addr));
}

// D = A . B + D in place, with A rows 8..15 zero (a1 = a3 = 0): rows 8..15
// of the accumulator start at zero and stay zero, so only d[0], d[1] carry
// data, but the four registers stay one in-place group (no moves).
template <bool BF>
__device__ __forceinline__ void mma16816(float* d, uint32_t a0, uint32_t a2, uint32_t b0, uint32_t b1) {
    if constexpr (BF) {
        asm volatile(
            "mma.sync.aligned.m16n8k16.row.col.f32.bf16.bf16.f32 {%0,%1,%2,%3}, {%4,%5,%6,%7}, {%8,%9}, "
            "{%0,%1,%2,%3};"
            : "+f"(d[0]), "+f"(d[1]), "+f"(d[2]), "+f"(d[3])
            : "r"(a0), "r"(0u), "r"(a2), "r"(0u), "r"(b0), "r"(b1));
    } else {
        asm volatile(
            "mma.sync.aligned.m16n8k16.row.col.f32.f16.f16.f32 {%0,%1,%2,%3}, {%4,%5,%6,%7}, {%8,%9}, "
            "{%0,%1,%2,%3};"
            : "+f"(d[0]), "+f"(d[1]), "+f"(d[2]), "+f"(d[3])
            : "r"(a0), "r"(0u), "r"(a2), "r"(0u), "r"(b0), "r"(b1));
    }
}

// 2^x with the hardware approximation (relative error ~2^-22; -inf -> 0).
__device__ __forceinline__ float ex2(float x) {
    float y;
    asm("ex2.approx.ftz.f32 %0, %1;" : "=f"(y) : "f"(x));
    return y;
}

// Splits a 32-bit word of four E4M3 bytes into two f16x2 words (bytes 0,1
// and bytes 2,3), with the hardware conversion.
__device__ __forceinline__ void e4m3x4_to_f16x4(uint32_t w, uint32_t& lo, uint32_t& hi) {
    asm("{\n\t.reg .b16 l, h;\n\tmov.b32 {l, h}, %2;\n\t"
        "cvt.rn.f16x2.e4m3x2 %0, l;\n\tcvt.rn.f16x2.e4m3x2 %1, h;\n\t}"
        : "=r"(lo), "=r"(hi)
        : "r"(w));
}

__device__ __forceinline__ void tma_load_2d(void* dst, const CUtensorMap* map, int x, int y, uint64_t* bar,
                                            uint64_t policy) {
    asm volatile(
        "cp.async.bulk.tensor.2d.shared::cluster.global.tile.mbarrier::complete_tx::bytes.L2::cache_hint"
        " [%0], [%1, {%2, %3}], [%4], %5;" ::"r"(smem_addr(dst)),
        "l"(reinterpret_cast<uint64_t>(map)), "r"(x), "r"(y), "r"(smem_addr(bar)), "l"(policy)
        : "memory");
}

// Orders this thread's generic-proxy shared-memory writes before later
// async-proxy (TMA) accesses of the same memory.
__device__ __forceinline__ void fence_proxy_async_smem() {
    asm volatile("fence.proxy.async.shared::cta;" ::: "memory");
}

__device__ __forceinline__ uint32_t e4m3x2_to_f16x2(uint32_t two_bytes) {
    __half2_raw h = __nv_cvt_fp8x2_to_halfraw2(static_cast<__nv_fp8x2_storage_t>(two_bytes & 0xffffu), __NV_E4M3);
    return static_cast<uint32_t>(h.x) | (static_cast<uint32_t>(h.y) << 16);
}

template <bool BF>
__device__ __forceinline__ uint32_t pack2(float lo, float hi) {
    if constexpr (BF) {
        __nv_bfloat162 v = __floats2bfloat162_rn(lo, hi);
        return *reinterpret_cast<uint32_t*>(&v);
    } else {
        __half2 v = __floats2half2_rn(lo, hi);
        return *reinterpret_cast<uint32_t*>(&v);
    }
}

// Byte offset of 16-byte chunk `c` of row `r` in a 128-byte-row tile landed
// with the 128-byte swizzle.
__device__ __forceinline__ uint32_t swz128(int r, int c) {
    return static_cast<uint32_t>(r * 128 + ((c ^ (r & 7)) << 4));
}

// Copy stages per warp and resident CTAs per SM: about 190 KB of tiles in
// flight per SM either way; fp8 tiles are half the size, so twice the warps
// share the same bytes (its per-block instruction count is higher).
template <typename KT>
struct MmaCfg {
    static constexpr int kStages = KT::bytes == 1 ? 4 : 2;
    static constexpr int kCtasPerSm = 3;
};

template <typename KT, int NW, int NST>
struct MmaSmem {
    static constexpr int kTile = kBlockSize * 128 * KT::bytes;  // 4096 (16-bit) or 2048 (fp8)
    static constexpr int kStage = 2 * kTile;
    static constexpr int kBarOffset = NW * NST * kStage;
    static constexpr int kPhysOffset = kBarOffset + NW * NST * 8;
    // merge weights: [NW][8] per-warp scale factors, [8] 1/denominator, [8] denominator
    static constexpr int kMergeOffset = kPhysOffset + NW * NST * 4;
    static constexpr int kBytes = kMergeOffset + (NW * 8 + 16) * 4 + 1024;  // + alignment slack
};

template <int G, typename KT, typename QT, int NW, int NST>
__global__ void __launch_bounds__(NW * 32, MmaCfg<KT>::kCtasPerSm)
    decode_mma_kernel(const DecodeParams p, const __grid_constant__ CUtensorMap tmk,
                      const __grid_constant__ CUtensorMap tmv) {
    constexpr int D = 128;
    constexpr bool kFP8 = KT::bytes == 1;
    constexpr bool kBF = std::is_same<KT, BF16>::value;
    using SM = MmaSmem<KT, NW, NST>;
    constexpr int TILE = SM::kTile;
    constexpr int STAGE = SM::kStage;
    static_assert(G == 2 || G == 4 || G == 8, "group size");

    extern __shared__ unsigned char smem_raw[];
    // SW128 TMA destinations must be 1024-byte aligned.
    unsigned char* smem = smem_raw + ((1024 - (smem_addr(smem_raw) & 1023)) & 1023);

    const int warp = threadIdx.x >> 5, lane = threadIdx.x & 31;
    const int r0 = lane >> 2, qd = lane & 3;
    const int part = blockIdx.x, h = blockIdx.y, s = blockIdx.z;

    int L = __ldg(p.seq_lens + s);
    const int Lmax = min(p.MB * kBlockSize, p.NP * p.P);
    if (L < 0 || L > Lmax) {
        if (threadIdx.x == 0 && part == 0 && h == 0) report(p.err, PKV_DEVERR_SEQ_LEN);
        L = L < 0 ? 0 : Lmax;
    }
    const int nparts = L > 0 ? (L + p.P - 1) / p.P : 1;
    if (part >= nparts) return;
    const int t0 = part * p.P;
    const int t1 = min(L, t0 + p.P);
    const int j0 = t0 / kBlockSize;
    const int nblk = (t1 + kBlockSize - 1) / kBlockSize - j0;
    const int nb_w = warp < nblk ? (nblk - warp + NW - 1) / NW : 0;

    unsigned char* wbase = smem + warp * NST * STAGE;
    uint64_t* bars = reinterpret_cast<uint64_t*>(smem + SM::kBarOffset) + warp * NST;
    volatile int* stage_phys = reinterpret_cast<int*>(smem + SM::kPhysOffset) + warp * NST;
    const int32_t* bt = p.block_tables + static_cast<int64_t>(s) * p.MB + j0 + warp;
    const uint64_t pol = policy_evict_first();

    if (lane == 0) {
#pragma unroll
        for (int i = 0; i < NST; ++i) mbar_init(&bars[i], 1);
        mbar_init_fence();
    }
    __syncwarp();

    int tbl = -1;
    int k_issue = 0;
    auto issue_next = [&]() {  // warp-uniform call
        if ((k_issue & 31) == 0) {
            const int k = k_issue + lane;
            tbl = k < nb_w ? __ldg(bt + static_cast<int64_t>(k) * NW) : -1;
        }
        const int phys = __shfl_sync(kFull, tbl, k_issue & 31);
        const int stage = k_issue % NST;
        if (lane == 0) {
            fence_proxy_async_smem();  // generic writes to this stage (row zeroing) before the TMA
            stage_phys[stage] = phys;
            if (phys >= 0 && phys < p.NB) {
                const int y = (phys * p.Hkv + h) * kBlockSize;
                unsigned char* dst = wbase + stage * STAGE;
                mbar_arrive_expect_tx(&bars[stage], 2 * TILE);
                if constexpr (kFP8) {
                    tma_load_2d(dst, &tmk, 0, y, &bars[stage], pol);
                    tma_load_2d(dst + TILE, &tmv, 0, y, &bars[stage], pol);
                } else {
                    tma_load_2d(dst, &tmk, 0, y, &bars[stage], pol);
                    tma_load_2d(dst + 2048, &tmk, 64, y, &bars[stage], pol);
                    tma_load_2d(dst + TILE, &tmv, 0, y, &bars[stage], pol);
                    tma_load_2d(dst + TILE + 2048, &tmv, 64, y, &bars[stage], pol);
                }
            } else {
                report(p.err, PKV_DEVERR_BLOCK_ID);
                mbar_arrive_expect_tx(&bars[stage], 0);
            }
        }
        ++k_issue;
    };

    // ---- A fragments of Q (rows = heads of the group; rows >= G are zero)
    uint32_t qa[8][2];
    {
        const int g = r0 < G ? r0 : 0;
        const int64_t row = static_cast<int64_t>(s) * p.Hq + h * G + g;
        const unsigned char* qrow = static_cast<const unsigned char*>(p.q) + row * D * 2;
#pragma unroll
        for (int kk = 0; kk < 8; ++kk) {
            if constexpr (!kFP8) {
                qa[kk][0] = *reinterpret_cast<const uint32_t*>(qrow + (16 * kk + 2 * qd) * 2);
                qa[kk][1] = *reinterpret_cast<const uint32_t*>(qrow + (16 * kk + 8 + 2 * qd) * 2);
            } else {
                uint32_t w[2];
                load_words<8>(qrow + (32 * qd + 4 * kk) * 2, w);
                float f[4];
                Unpack<QT, 4>::run(w, f);
                qa[kk][0] = pack2<false>(f[0], f[1]);
                qa[kk][1] = pack2<false>(f[2], f[3]);
            }
            if (r0 >= G) qa[kk][0] = qa[kk][1] = 0u;
        }
    }

    for (int i = 0; i < NST && k_issue < nb_w; ++i) issue_next();

    float o[16][4];
#pragma unroll
    for (int j = 0; j < 16; ++j) o[j][0] = o[j][1] = o[j][2] = o[j][3] = 0.f;
    float m = -INFINITY, lsum = 0.f;

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
            unsigned char* kt = wbase + stage * STAGE;
            unsigned char* vt = kt + TILE;
            const uint32_t kts = smem_addr(kt), vts = smem_addr(vt);
            if (nvalid < kBlockSize) {
                // zero the value rows past the sequence end (stale pool bytes
                // must not reach the MMA: 0 * NaN is NaN)
                constexpr int kChunksPerRow = kFP8 ? 8 : 16;
                const int nz = (kBlockSize - nvalid) * kChunksPerRow;
                for (int i = lane; i < nz; i += 32) {
                    const int row = nvalid + i / kChunksPerRow, c = i % kChunksPerRow;
                    *reinterpret_cast<uint4*>(vt + (c >> 3) * 2048 + row * 128 + (c & 7) * 16) =
                        make_uint4(0u, 0u, 0u, 0u);
                }
                __syncwarp();
            }
            // fp8: value fragments are loaded up front so their latency hides
            // behind Q K^T (chunk r0 of tokens 2qd, 2qd+1, 2qd+8, 2qd+9)
            uint4 va[4];
            if constexpr (kFP8) {
#pragma unroll
                for (int i = 0; i < 4; ++i) {
                    const int tok = 2 * qd + (i & 1) + 8 * (i >> 1);
                    va[i] = *reinterpret_cast<const uint4*>(vt + swz128(tok, r0));
                }
            }
            // ---- S^T = Q K^T  (n-tile j = tokens 8j .. 8j+7)
            float sa[2][4] = {{0.f, 0.f, 0.f, 0.f}, {0.f, 0.f, 0.f, 0.f}};
            if constexpr (!kFP8) {
                const int mat = lane >> 3, rr = lane & 7;
                const int tok = rr + 8 * (mat >> 1);
#pragma unroll
                for (int kk = 0; kk < 8; ++kk) {
                    const int chunk = 2 * kk + (mat & 1);
                    uint32_t b0, b1, b2, b3;
                    ldsm_x4(kts + (chunk >> 3) * 2048 + swz128(tok, chunk & 7), b0, b1, b2, b3);
                    mma16816<kBF>(sa[0], qa[kk][0], qa[kk][1], b0, b1);
                    mma16816<kBF>(sa[1], qa[kk][0], qa[kk][1], b2, b3);
                }
            } else {
                uint32_t w[2][8];
#pragma unroll
                for (int j = 0; j < 2; ++j) {
                    const int tok = 8 * j + r0;
                    const uint4 c0 = *reinterpret_cast<const uint4*>(kt + swz128(tok, 2 * qd));
                    const uint4 c1 = *reinterpret_cast<const uint4*>(kt + swz128(tok, 2 * qd + 1));
                    w[j][0] = c0.x; w[j][1] = c0.y; w[j][2] = c0.z; w[j][3] = c0.w;
                    w[j][4] = c1.x; w[j][5] = c1.y; w[j][6] = c1.z; w[j][7] = c1.w;
                }
#pragma unroll
                for (int kk = 0; kk < 8; ++kk) {
#pragma unroll
                    for (int j = 0; j < 2; ++j) {
                        uint32_t blo, bhi;
                        e4m3x4_to_f16x4(w[j][kk], blo, bhi);
                        mma16816<false>(sa[j], qa[kk][0], qa[kk][1], blo, bhi);
                    }
                }
            }
            // ---- online softmax on row r0 (tokens 2qd, 2qd+1, 8+2qd, 9+2qd)
            float sv[4] = {sa[0][0] * p.qk_scale, sa[0][1] * p.qk_scale, sa[1][0] * p.qk_scale,
                           sa[1][1] * p.qk_scale};
            if (nvalid < kBlockSize) {
                const int tk[4] = {2 * qd, 2 * qd + 1, 8 + 2 * qd, 9 + 2 * qd};
#pragma unroll
                for (int i = 0; i < 4; ++i)
                    if (tk[i] >= nvalid) sv[i] = -INFINITY;
            }
            float bm = fmaxf(fmaxf(sv[0], sv[1]), fmaxf(sv[2], sv[3]));
            bm = fmaxf(bm, __shfl_xor_sync(kFull, bm, 1));
            bm = fmaxf(bm, __shfl_xor_sync(kFull, bm, 2));
            const float mn = fmaxf(m, bm);
            const float alpha = mn == m ? 1.f : ex2(m - mn);
            m = mn;
            float pr[4];
#pragma unroll
            for (int i = 0; i < 4; ++i) pr[i] = ex2(sv[i] - mn);
            lsum = lsum * alpha + (pr[0] + pr[1]) + (pr[2] + pr[3]);
            const uint32_t pa0 = pack2<kBF>(pr[0], pr[1]);
            const uint32_t pa2 = pack2<kBF>(pr[2], pr[3]);
            if (__any_sync(kFull, alpha != 1.f)) {  // skip when no row's max moved
#pragma unroll
                for (int j = 0; j < 16; ++j) {
                    o[j][0] *= alpha;
                    o[j][1] *= alpha;
                }
            }
            // ---- O += P V
            if constexpr (!kFP8) {
                const int mat = lane >> 3, rr = lane & 7;
                const int tok = rr + 8 * (mat & 1);
#pragma unroll
                for (int i = 0; i < 8; ++i) {
                    const int chunk = 2 * i + (mat >> 1);
                    uint32_t b0, b1, b2, b3;
                    ldsm_x4_t(vts + (chunk >> 3) * 2048 + swz128(tok, chunk & 7), b0, b1, b2, b3);
                    mma16816<kBF>(o[2 * i], pa0, pa2, b0, b1);
                    mma16816<kBF>(o[2 * i + 1], pa0, pa2, b2, b3);
                }
            } else {
                const uint32_t wa[4] = {va[0].x, va[0].y, va[0].z, va[0].w};
                const uint32_t wb[4] = {va[1].x, va[1].y, va[1].z, va[1].w};
                const uint32_t wc[4] = {va[2].x, va[2].y, va[2].z, va[2].w};
                const uint32_t wd[4] = {va[3].x, va[3].y, va[3].z, va[3].w};
#pragma unroll
                for (int w = 0; w < 4; ++w) {
#pragma unroll
                    for (int i = 0; i < 4; i += 2) {
                        const int j = 4 * w + i;
                        const uint32_t sel = i == 0 ? 0x5140u : 0x7362u;
                        uint32_t ab0, ab1, cd0, cd1;
                        e4m3x4_to_f16x4(__byte_perm(wa[w], wb[w], sel), ab0, ab1);
                        e4m3x4_to_f16x4(__byte_perm(wc[w], wd[w], sel), cd0, cd1);
                        mma16816<false>(o[j], pa0, pa2, ab0, cd0);
                        mma16816<false>(o[j + 1], pa0, pa2, ab1, cd1);
                    }
                }
            }
        }
        __syncwarp();
        if (k_issue < nb_w) issue_next();
    }

    if (aborted) {
        for (int k = 0; k < NST; ++k) {
            const int kk = k_issue - 1 - k;
            if (kk < 0) break;
            (void)mbar_wait(&bars[kk % NST], (kk / NST) & 1);
        }
    }

    // ---- warp state -> shared memory: [G] m, [G] l, then the accumulators
    // in fragment order with a 33-word pitch (value (j, e) of lane l at
    // 2G + (2j + e) * 33 + l): stores cover 32 consecutive words and the
    // merge's reads of consecutive head dimensions fall in distinct banks.
    lsum += __shfl_xor_sync(kFull, lsum, 1);
    lsum += __shfl_xor_sync(kFull, lsum, 2);
    float* ws = reinterpret_cast<float*>(wbase);
    __syncwarp();
    if (r0 < G && qd == 0) {
        ws[r0] = aborted ? -INFINITY : m;
        ws[G + r0] = aborted ? 0.f : lsum;
    }
#pragma unroll
    for (int j = 0; j < 16; ++j)
#pragma unroll
        for (int e = 0; e < 2; ++e) ws[2 * G + (2 * j + e) * 33 + lane] = aborted ? 0.f : o[j][e];
    __syncthreads();

    // ---- cross-warp log-sum-exp weights, once per (warp, head)
    float* msc = reinterpret_cast<float*>(smem + SM::kMergeOffset);  // [NW][8]
    float* minv = msc + NW * 8;                                       // [8]
    float* mden = minv + 8;                                           // [8]
    if (threadIdx.x < G) {
        const int g = threadIdx.x;
        float M = -INFINITY;
#pragma unroll
        for (int w = 0; w < NW; ++w) M = fmaxf(M, reinterpret_cast<float*>(smem + w * NST * STAGE)[g]);
        float den = 0.f;
#pragma unroll
        for (int w = 0; w < NW; ++w) {
            const float* wsw = reinterpret_cast<float*>(smem + w * NST * STAGE);
            const float sc = (M != -INFINITY && wsw[g] != -INFINITY) ? exp2f(wsw[g] - M) : 0.f;
            msc[w * 8 + g] = sc;
            den = fmaf(sc, wsw[G + g], den);
        }
        minv[g] = den > 0.f ? 1.f / den : 0.f;
        mden[g] = den > 0.f ? den : 0.f;
    }
    __syncthreads();

    for (int idx = threadIdx.x; idx < G * D; idx += NW * 32) {
        const int g = idx / D, d = idx % D;
        // inverse of the fragment order: head dimension d of row g
        int j, e, q4;
        if constexpr (kFP8) {
            j = d & 15;
            e = (d >> 4) & 1;
            q4 = d >> 5;
        } else {
            j = d >> 3;
            e = d & 1;
            q4 = (d >> 1) & 3;
        }
        const int frag = 2 * G + (2 * j + e) * 33 + g * 4 + q4;
        float num = 0.f;
#pragma unroll
        for (int w = 0; w < NW; ++w)
            num = fmaf(msc[w * 8 + g], reinterpret_cast<float*>(smem + w * NST * STAGE)[frag], num);
        const float out = num * minv[g] * p.v_scale;
        const int64_t row = static_cast<int64_t>(s) * p.Hq + h * G + g;
        if (nparts == 1) {
            reinterpret_cast<typename QT::storage*>(p.out)[row * D + d] = from_float<QT>(out);
        } else {
            const int64_t prow = row * p.NP + part;
            p.part_o[prow * D + d] = out;
            if (d == 0) {
                float M = -INFINITY;
#pragma unroll
                for (int w = 0; w < NW; ++w) M = fmaxf(M, reinterpret_cast<float*>(smem + w * NST * STAGE)[g]);
                p.part_m[prow] = M;
                p.part_l[prow] = mden[g];
            }
        }
    }
}

// ------------------------------------------------------------- launchers
template <int G, typename KT, typename QT>
cudaError_t launch_decode_mma_t(const DecodeParams& p, const CUtensorMap& tk, const CUtensorMap& tv,
                                cudaStream_t st) {
    constexpr int NW = kDecodeWarps;
    constexpr int NST = MmaCfg<KT>::kStages;
    constexpr int SMEM = MmaSmem<KT, NW, NST>::kBytes;
    auto kern = decode_mma_kernel<G, KT, QT, NW, NST>;
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
    dim3 grid(p.NP, p.Hkv, p.S);
    kern<<<grid, NW * 32, SMEM, st>>>(p, tk, tv);
    return cudaGetLastError();
}

template <typename KT, typename QT>
cudaError_t launch_decode_mma_family(const DecodeParams& p, int G, const CUtensorMap& tk, const CUtensorMap& tv,
                                     cudaStream_t st) {
    switch (G) {
    case 2: return launch_decode_mma_t<2, KT, QT>(p, tk, tv, st);
    case 4: return launch_decode_mma_t<4, KT, QT>(p, tk, tv, st);
    case 8: return launch_decode_mma_t<8, KT, QT>(p, tk, tv, st);
    }
    return cudaErrorInvalidValue;
}

}  // namespace pkv
