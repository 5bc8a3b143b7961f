// pkv_decode_mma.cuh -- tensor-core paged decode attention for grouped-query
// attention (G = Hq / Hkv in {2, 4, 8}, head_size 128).
//
// Same computation as decode_kernel ("vLLM：大语言模型推理与服务库" section 4.4:
// per query head, walk the block table, q . K -> softmax -> weighted V), same
// grid (partition, kv head, sequence) and per-warp copy pipelines, but the
// two products of a 16-token block run on the tensor cores with the G query
// heads of the group on the MMA's N = 8 columns:
//
//   S   [16 tok x 8 heads]  = K   [16 x 128] . Q^T [128 x 8]   (8 MMAs)
//   O^T [128 d  x 8 heads] += V^T [128 x 16] . P^T [16 x 8]     (2 x 8 MMAs)
//
// with mma.m16n8k16 and fp32 accumulation.  P enters the second product as
// a 16-bit head and a 16-bit tail (its rounding error), one MMA each into the
// same accumulator, so the probabilities keep 16 (bf16) or 22 (f16)
// significant bits: rounded once to bf16 they alone could move an output by
// 2^-9 of max|V|.  For G = 8 every column is used
// (G = 4 / 2: half / a quarter).  The newer 5th-generation MMA needs M >= 64
// and would round-trip the scores through tensor memory for the online
// softmax every block; this path keeps scores, probabilities and output in
// registers.  P goes from the accumulator layout of S to the B-operand
// layout of P^T with two 8x8 register transposes (movmatrix).
//
// Tiles arrive through 2-D TMA tensor copies with the 128-byte swizzle
// (16-byte chunk c of smem row r stored at chunk c ^ (r & 7)), so the
// fragment loads (ldmatrix for 16-bit pools; 16-byte loads for fp8) are free
// of shared-memory bank conflicts.
//
// fp8 E4M3 pools: the MMA runs in f16.  Key and value bytes are turned into
// f16 pairs in registers (hardware e4m3x2 -> f16x2 conversion, exact), with
// index permutations chosen so each lane reads whole 16-byte chunks: for
// keys, contraction column k of lane quad member q covers head dimensions
// 32q + 4k .. 32q + 4k + 3; for values, row g / g + 8 of m-tile i is head
// dimension 16g + 2i / 16g + 2i + 1.  q is converted to f16 (exact in the
// normal range), and the CTA keeps one copy of its Q^T fragments in shared
// memory rather than one per warp in registers, which fits a fifth CTA per
// SM.
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

// D = A . B + D in place, all four A registers given.
template <bool BF>
__device__ __forceinline__ void mma16816a(float* d, uint32_t a0, uint32_t a1, uint32_t a2, uint32_t a3, uint32_t b0,
                                          uint32_t b1) {
    if constexpr (BF) {
        asm volatile(
            "mma.sync.aligned.m16n8k16.row.col.f32.bf16.bf16.f32 {%0,%1,%2,%3}, {%4,%5,%6,%7}, {%8,%9}, "
            "{%0,%1,%2,%3};"
            : "+f"(d[0]), "+f"(d[1]), "+f"(d[2]), "+f"(d[3])
            : "r"(a0), "r"(a1), "r"(a2), "r"(a3), "r"(b0), "r"(b1));
    } else {
        asm volatile(
            "mma.sync.aligned.m16n8k16.row.col.f32.f16.f16.f32 {%0,%1,%2,%3}, {%4,%5,%6,%7}, {%8,%9}, "
            "{%0,%1,%2,%3};"
            : "+f"(d[0]), "+f"(d[1]), "+f"(d[2]), "+f"(d[3])
            : "r"(a0), "r"(a1), "r"(a2), "r"(a3), "r"(b0), "r"(b1));
    }
}

// Transpose of an 8x8 matrix of 16-bit values held as one register per lane
// (lane l holds row l/4, columns 2(l%4), 2(l%4)+1).
__device__ __forceinline__ uint32_t movmatrix_t(uint32_t x) {
    uint32_t y;
    asm volatile("movmatrix.sync.aligned.m8n8.trans.b16 %0, %1;" : "=r"(y) : "r"(x));
    return y;
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

// Two floats as a 16-bit pair (head) and the rounding error of that pair as a
// second 16-bit pair (tail): head + tail carries 16 (bf16) or 22 (f16)
// significant bits of each value.  The difference x - head is exact in
// float32, so the tail is x - head rounded once.
template <bool BF>
__device__ __forceinline__ void pack2_split(float lo, float hi, uint32_t& head, uint32_t& tail) {
    head = pack2<BF>(lo, hi);
    float rl, rh;
    if constexpr (BF) {
        rl = __uint_as_float(head << 16);
        rh = __uint_as_float(head & 0xffff0000u);
    } else {
        const float2 r = __half22float2(*reinterpret_cast<const __half2*>(&head));
        rl = r.x;
        rh = r.y;
    }
    tail = pack2<BF>(lo - rl, hi - rh);
}

// Byte offset of 16-byte chunk `c` of row `r` in a 128-byte-row tile landed
// with the 128-byte swizzle.  For even r: swz128(r, c ^ 1) = swz128(r, c) ^ 16,
// swz128(r + 1, c) = (swz128(r, c) ^ 16) + 128, and swz128(r + 8, c) =
// swz128(r, c) + 1024.
__device__ __forceinline__ uint32_t swz128(int r, int c) {
    return static_cast<uint32_t>(r * 128 + ((c ^ (r & 7)) << 4));
}

__device__ __forceinline__ uint4 lds128(uint32_t addr) {
    uint4 v;
    asm volatile("ld.shared.v4.b32 {%0, %1, %2, %3}, [%4];" : "=r"(v.x), "=r"(v.y), "=r"(v.z), "=r"(v.w) : "r"(addr));
    return v;
}

// The online softmax's reference maximum is moved only when a block's
// maximum exceeds it by more than this many log2 units (probabilities <= 2^8).
constexpr float kRebaseLog2 = 8.0f;

// Copy stages per warp and resident CTAs per SM.  Two stages keep a block
// in flight while one is attended (a third measured no faster on either
// type).  A CTA's start (its first copies' latency) is a fixed cost of each
// short partition, so more resident CTAs hide more of it: fp8 CTAs keep
// their Q^T fragments in shared memory and load the value bytes late, which
// fits five of them per SM in the register file (longctx_fp8 decode call
// 104.5 -> 102.4 us against four; six spill and lose).
template <typename KT>
struct MmaCfg {
    static constexpr int kWarps = 4;
    static constexpr int kStages = 2;
    static constexpr int kCtasPerSm = KT::bytes == 1 ? 5 : 3;
};

template <typename KT, int NW, int NST>
struct MmaSmem {
    static constexpr int kTile = kBlockSize * 128 * KT::bytes;  // 4096 (16-bit) or 2048 (fp8)
    static constexpr int kStage = 2 * kTile;
    static constexpr int kBarOffset = NW * NST * kStage;
    static constexpr int kPhysOffset = kBarOffset + NW * NST * 8;
    // merge weights: [NW][8] per-warp scale factors, [8] 1/denominator, [8] denominator
    static constexpr int kMergeOffset = kPhysOffset + NW * NST * 4;
    // fp8: the Q^T B fragments, [8 k-steps][32 lanes] pairs (16-bit pools keep them in registers)
    static constexpr int kQOffset = kMergeOffset + (NW * 8 + 16) * 4;
    static constexpr int kBytes = kQOffset + (KT::bytes == 1 ? 8 * 32 * 8 : 0) + 1024;  // + alignment slack
};

// B fragments of Q^T for (sequence s, KV head h): column n = head g8 of the
// group (heads >= G zero); fp8 pools take q as f16 (exact in the normal range).
template <int G, typename KT, typename QT>
__device__ __forceinline__ void load_qb(const void* q, int Hq, int s, int h, uint32_t (&qb)[8][2]) {
    constexpr int D = 128;
    const int lane = threadIdx.x & 31;
    const int g8 = lane >> 2, qd = lane & 3;
    const int g = g8 < G ? g8 : 0;
    const int64_t row = static_cast<int64_t>(s) * Hq + h * G + g;
    const unsigned char* qrow = static_cast<const unsigned char*>(q) + row * D * 2;
#pragma unroll
    for (int kk = 0; kk < 8; ++kk) {
        if constexpr (KT::bytes != 1) {
            qb[kk][0] = *reinterpret_cast<const uint32_t*>(qrow + (16 * kk + 2 * qd) * 2);
            qb[kk][1] = *reinterpret_cast<const uint32_t*>(qrow + (16 * kk + 8 + 2 * qd) * 2);
        } else {
            uint32_t w[2];
            load_words<8>(qrow + (32 * qd + 4 * kk) * 2, w);
            float f[4];
            Unpack<QT, 4>::run(w, f);
            qb[kk][0] = pack2<false>(f[0], f[1]);
            qb[kk][1] = pack2<false>(f[2], f[3]);
        }
        if (g8 >= G) qb[kk][0] = qb[kk][1] = 0u;
    }
}

// One 16-token block of the decode: S = K Q^T for the G heads on the MMA's
// N columns, the online-softmax update of (m, l) per head with the lazy
// reference maximum, and O^T += V^T P^T.  kt: the block's K tile (V tile
// TILE bytes after it) in the 128-byte-swizzled layout the TMA lands;
// nvalid: tokens of the block inside the sequence (value rows past it are
// zeroed first).  Warp-uniform call.
template <int G, typename KT, typename QT>
__device__ __forceinline__ void mma_block(unsigned char* kt, int nvalid, const uint32_t (&qb)[8][2],
                                          const uint2* qsm, float (&o)[8][4], float& mA, float& mB, float& lA,
                                          float& lB, float qk_scale, uint32_t koff, uint32_t voff) {
    constexpr bool kFP8 = KT::bytes == 1;
    constexpr bool kBF = std::is_same<KT, BF16>::value;
    constexpr int TILE = kBlockSize * 128 * KT::bytes;
    const int lane = threadIdx.x & 31;
    const int g8 = lane >> 2;
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
    // ---- S = K Q^T, two accumulators (even / odd k-steps) to halve the chain
    float sa[2][4] = {{0.f, 0.f, 0.f, 0.f}, {0.f, 0.f, 0.f, 0.f}};
    if constexpr (!kFP8) {
        const int mat = lane >> 3, rr = lane & 7;
        const int tok = rr + 8 * (mat & 1);
#pragma unroll
        for (int kk = 0; kk < 8; ++kk) {
            const int chunk = 2 * kk + (mat >> 1);
            uint32_t a0, a1, a2, a3;
            ldsm_x4(kts + (chunk >> 3) * 2048 + swz128(tok, chunk & 7), a0, a1, a2, a3);
            mma16816a<kBF>(sa[kk & 1], a0, a1, a2, a3, qb[kk][0], qb[kk][1]);
        }
    } else {
        uint32_t w0[8], w1[8];
        {
            const uint4 c0 = lds128(kts + koff);
            const uint4 c1 = lds128(kts + (koff ^ 16u));
            const uint4 c2 = lds128(kts + koff + 1024u);
            const uint4 c3 = lds128(kts + (koff ^ 16u) + 1024u);
            w0[0] = c0.x; w0[1] = c0.y; w0[2] = c0.z; w0[3] = c0.w;
            w0[4] = c1.x; w0[5] = c1.y; w0[6] = c1.z; w0[7] = c1.w;
            w1[0] = c2.x; w1[1] = c2.y; w1[2] = c2.z; w1[3] = c2.w;
            w1[4] = c3.x; w1[5] = c3.y; w1[6] = c3.z; w1[7] = c3.w;
        }
#pragma unroll
        for (int kk = 0; kk < 8; ++kk) {
            uint32_t a01, a45, a23, a67;
            e4m3x4_to_f16x4(w0[kk], a01, a45);
            e4m3x4_to_f16x4(w1[kk], a23, a67);
            const uint2 qf = qsm[kk * 32 + lane];
            mma16816a<false>(sa[kk & 1], a01, a23, a45, a67, qf.x, qf.y);
        }
    }
    // ---- online softmax: s0 (tok g8, head A), s1 (tok g8, head B),
    //      s2 (tok g8+8, head A), s3 (tok g8+8, head B)
    float sv[4];
#pragma unroll
    for (int c = 0; c < 4; ++c) sv[c] = (sa[0][c] + sa[1][c]) * qk_scale;
    if (nvalid < kBlockSize) {
        if (g8 >= nvalid) sv[0] = sv[1] = -INFINITY;
        if (g8 + 8 >= nvalid) sv[2] = sv[3] = -INFINITY;
    }
    float bA = fmaxf(sv[0], sv[2]), bB = fmaxf(sv[1], sv[3]);
#pragma unroll
    for (int mask = 4; mask < 32; mask <<= 1) {
        bA = fmaxf(bA, __shfl_xor_sync(kFull, bA, mask));
        bB = fmaxf(bB, __shfl_xor_sync(kFull, bB, mask));
    }
    // Lazy reference maximum: the probabilities are taken against a
    // reference that moves only when a block's maximum exceeds it by
    // more than 2^kRebaseLog2, so every p stays <= 2^kRebaseLog2 (exact
    // range for f16 / bf16) and O is rescaled only on those rare
    // moves, not whenever one of the group's heads sees a new maximum.
    // The partials carry the reference, and the merges use it as the
    // row's maximum; the result is the same softmax.
    const bool rbA = bA > mA + kRebaseLog2, rbB = bB > mB + kRebaseLog2;
    const float nA = rbA ? bA : mA, nB = rbB ? bB : mB;
    const float alA = rbA ? ex2(mA - nA) : 1.f;  // 0 on the first block (mA = -inf)
    const float alB = rbB ? ex2(mB - nB) : 1.f;
    mA = nA;
    mB = nB;
    const float p0 = ex2(sv[0] - nA), p1 = ex2(sv[1] - nB), p2 = ex2(sv[2] - nA), p3 = ex2(sv[3] - nB);
    lA = lA * alA + (p0 + p2);
    lB = lB * alB + (p1 + p3);
    if (__builtin_expect(__any_sync(kFull, rbA || rbB), 0)) {  // skip when no head's reference moved
#pragma unroll
        for (int i = 0; i < 8; ++i) {
            o[i][0] *= alA;
            o[i][1] *= alB;
            o[i][2] *= alA;
            o[i][3] *= alB;
        }
    }
    // P^T fragments: transpose the (token, head) 8x8 tiles of P.  P
    // enters the product as a 16-bit head plus a 16-bit tail (two
    // MMAs into the same float32 accumulator), so the probabilities
    // keep 16 (bf16) or 22 (f16) significant bits, not 8 or 11.
    uint32_t h01, t01, h23, t23;
    pack2_split<kBF>(p0, p1, h01, t01);
    pack2_split<kBF>(p2, p3, h23, t23);
    const uint32_t pb0 = movmatrix_t(h01), pt0 = movmatrix_t(t01);  // tokens 0..7
    const uint32_t pb1 = movmatrix_t(h23), pt1 = movmatrix_t(t23);  // tokens 8..15
    // ---- O^T += V^T P^T
    if constexpr (!kFP8) {
        const int mat = lane >> 3, rr = lane & 7;
        const int tok = rr + 8 * (mat >> 1);
#pragma unroll
        for (int i = 0; i < 8; ++i) {
            const int chunk = 2 * i + (mat & 1);
            uint32_t a0, a1, a2, a3;
            ldsm_x4_t(vts + (chunk >> 3) * 2048 + swz128(tok, chunk & 7), a0, a1, a2, a3);
            mma16816a<kBF>(o[i], a0, a1, a2, a3, pb0, pb1);
            mma16816a<kBF>(o[i], a0, a1, a2, a3, pt0, pt1);
        }
    } else {
        // value bytes: chunk g8 of tokens 2qd, 2qd+1, 2qd+8, 2qd+9; the four
        // offsets follow from one lane constant (see swz128)
        uint4 va[4];
        {
            const uint32_t v1 = (voff ^ 16u) + 128u;
            va[0] = lds128(vts + voff);
            va[1] = lds128(vts + v1);
            va[2] = lds128(vts + voff + 1024u);
            va[3] = lds128(vts + v1 + 1024u);
        }
        const uint32_t wa[4] = {va[0].x, va[0].y, va[0].z, va[0].w};
        const uint32_t wb[4] = {va[1].x, va[1].y, va[1].z, va[1].w};
        const uint32_t wc[4] = {va[2].x, va[2].y, va[2].z, va[2].w};
        const uint32_t wd[4] = {va[3].x, va[3].y, va[3].z, va[3].w};
#pragma unroll
        for (int i = 0; i < 8; ++i) {
            const int w = i >> 1;
            const uint32_t sel = (i & 1) ? 0x7362u : 0x5140u;  // bytes 2i, 2i+1 of the chunk
            uint32_t a01, a23, a45, a67;
            e4m3x4_to_f16x4(__byte_perm(wa[w], wb[w], sel), a01, a23);
            e4m3x4_to_f16x4(__byte_perm(wc[w], wd[w], sel), a45, a67);
            mma16816a<false>(o[i], a01, a23, a45, a67, pb0, pb1);
            mma16816a<false>(o[i], a01, a23, a45, a67, pt0, pt1);
        }
    }
}

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
    allow_dependent_launch();  // the merge may stage its CTAs behind this grid's last wave
    const int g8 = lane >> 2, qd = lane & 3;  // fragment row group / quad member
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
    auto issue_next = [&](const int stage) {  // warp-uniform call; stage = k_issue % NST
        if ((k_issue & 31) == 0) {
            const int k = k_issue + lane;
            tbl = k < nb_w ? __ldg(bt + static_cast<int64_t>(k) * NW) : -1;
        }
        const int phys = __shfl_sync(kFull, tbl, k_issue & 31);
        if (append_here && k_issue == nb_w - 1) {
            fused_commit<KT>(p, h, frow);
            __syncwarp();
        }
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

    uint32_t qb[8][2];
    uint2* qsm = reinterpret_cast<uint2*>(smem + SM::kQOffset);
    if constexpr (!kFP8) load_qb<G, KT, QT>(p.q, p.Hq, s, h, qb);

#pragma unroll
    for (int i = 0; i < NST; ++i)
        if (k_issue < nb_w) issue_next(i);

    if constexpr (kFP8) {
        // the CTA's warps share one copy of the fragments (registers for a
        // fifth resident CTA); warp w of the four writes k-steps 2w, 2w + 1
        uint32_t qt[8][2];
        load_qb<G, KT, QT>(p.q, p.Hq, s, h, qt);
#pragma unroll
        for (int kk = 0; kk < 8; ++kk)
            if ((kk >> 1) == warp % 4) qsm[kk * 32 + lane] = make_uint2(qt[kk][0], qt[kk][1]);
        __syncthreads();
    }

    // O^T accumulators: m-tile i, c0/c1 = (row g8, heads 2qd, 2qd+1),
    // c2/c3 = (row g8 + 8, heads 2qd, 2qd+1).
    float o[8][4];
#pragma unroll
    for (int i = 0; i < 8; ++i) o[i][0] = o[i][1] = o[i][2] = o[i][3] = 0.f;
    float mA = -INFINITY, mB = -INFINITY, lA = 0.f, lB = 0.f;  // heads 2qd (A), 2qd+1 (B)

    // fp8 fragment offsets in a stage's tiles: K chunk 2qd of row g8, V chunk
    // g8 of row 2qd (the stage bases are 1024-byte aligned)
    const uint32_t koff = swz128(g8, 2 * qd), voff = swz128(2 * qd, g8);
    bool aborted = false;
    uint32_t phase = 0;  // (k / NST) & 1
    int tok0 = (j0 + warp) * kBlockSize;
    // unrolled by the ring depth: each stage's addresses are constants
    for (int k0 = 0; k0 < nb_w && !aborted; k0 += NST) {
#pragma unroll
        for (int st = 0; st < NST; ++st) {
            if (k0 + st >= nb_w) break;
            if (!mbar_wait(&bars[st], phase)) {
                if (lane == 0) report(p.err, PKV_DEVERR_TIMEOUT);
                aborted = true;
                break;
            }
            const int phys = stage_phys[st];
            const int nvalid = min(kBlockSize, t1 - tok0);
            tok0 += NW * kBlockSize;
            if (phys >= 0 && phys < p.NB) {
                mma_block<G, KT, QT>(wbase + st * STAGE, nvalid, qb, qsm, o, mA, mB, lA, lB, p.qk_scale, koff, voff);
            }
            __syncwarp();
            if (k_issue < nb_w) issue_next(st);
        }
        phase ^= 1u;
    }

    if (aborted) {
        for (int k = 0; k < NST; ++k) {
            const int kk = k_issue - 1 - k;
            if (kk < 0) break;
            (void)mbar_wait(&bars[kk % NST], (kk / NST) & 1);
        }
    }

    // ---- warp state -> shared memory: [8] m, [8] l, then the accumulators in
    // fragment order with a 33-word pitch (value c of m-tile i of lane l at
    // 16 + (4i + c) * 33 + l).
#pragma unroll
    for (int mask = 4; mask < 32; mask <<= 1) {
        lA += __shfl_xor_sync(kFull, lA, mask);
        lB += __shfl_xor_sync(kFull, lB, mask);
    }
    float* ws = reinterpret_cast<float*>(wbase);
    __syncwarp();
    if (g8 == 0) {
        ws[2 * qd] = aborted ? -INFINITY : mA;
        ws[2 * qd + 1] = aborted ? -INFINITY : mB;
        ws[8 + 2 * qd] = aborted ? 0.f : lA;
        ws[8 + 2 * qd + 1] = aborted ? 0.f : lB;
    }
#pragma unroll
    for (int i = 0; i < 8; ++i)
#pragma unroll
        for (int c = 0; c < 4; ++c) ws[16 + (4 * i + c) * 33 + lane] = aborted ? 0.f : o[i][c];
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
            den = fmaf(sc, wsw[8 + g], den);
        }
        minv[g] = den > 0.f ? 1.f / den : 0.f;
        mden[g] = den > 0.f ? den : 0.f;
    }
    __syncthreads();

    // ---- output: thread t writes head g = t / TPH, head dimensions
    // [DPT (t % TPH), DPT (t % TPH + 1)) in one vector store
    constexpr int TPH = NW * 32 / G;  // threads per head
    constexpr int DPT = D / TPH;      // head dimensions per thread (G)
    static_assert(TPH * G == NW * 32 && DPT * TPH == D, "output split");
    {
        const int g = threadIdx.x / TPH;
        const int d0 = (threadIdx.x % TPH) * DPT;
        float sc[NW];
#pragma unroll
        for (int w = 0; w < NW; ++w) sc[w] = msc[w * 8 + g];
        const float inv = minv[g];
        float r[DPT];
#pragma unroll
        for (int j = 0; j < DPT; ++j) {
            const int d = d0 + j;
            // inverse of the fragment layout: head g, head dimension d
            int i, upper, gl;
            if constexpr (kFP8) {
                gl = d >> 4;
                i = (d & 15) >> 1;
                upper = d & 1;
            } else {
                i = d >> 4;
                upper = (d >> 3) & 1;
                gl = d & 7;
            }
            const int frag = 16 + (4 * i + 2 * upper + (g & 1)) * 33 + 4 * gl + (g >> 1);
            float num = 0.f;
#pragma unroll
            for (int w = 0; w < NW; ++w) num = fmaf(sc[w], reinterpret_cast<float*>(smem + w * NST * STAGE)[frag], num);
            r[j] = num * inv * p.v_scale;
        }
        const int64_t row = static_cast<int64_t>(s) * p.Hq + h * G + g;
        if (nparts == 1 && !p.cascade) {
            constexpr bool kBFq = std::is_same<QT, BF16>::value;
            uint32_t w[DPT / 2];
#pragma unroll
            for (int j = 0; j < DPT / 2; ++j) w[j] = pack2<kBFq>(r[2 * j], r[2 * j + 1]);
            unsigned char* dst = static_cast<unsigned char*>(p.out) + (row * D + d0) * 2;
            if constexpr (DPT == 8) {
                *reinterpret_cast<uint4*>(dst) = make_uint4(w[0], w[1], w[2], w[3]);
            } else if constexpr (DPT == 4) {
                *reinterpret_cast<uint2*>(dst) = make_uint2(w[0], w[1]);
            } else {
                *reinterpret_cast<uint32_t*>(dst) = w[0];
            }
        } else {
            const int64_t prow = row * p.NP + p.part_base + part;
            float* dst = p.part_o + prow * D + d0;
#pragma unroll
            for (int j = 0; j + 4 <= DPT; j += 4)
                *reinterpret_cast<float4*>(dst + j) = make_float4(r[j], r[j + 1], r[j + 2], r[j + 3]);
            if constexpr (DPT == 2) *reinterpret_cast<float2*>(dst) = make_float2(r[0], r[1]);
            if (d0 == 0) {
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
    constexpr int NW = MmaCfg<KT>::kWarps;
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
    const dim3 grid = p.work ? dim3(static_cast<unsigned>(static_cast<int64_t>(p.num_work) * p.Hkv))
                             : dim3(p.NP - p.part_base, p.Hkv, p.S + (p.join_primary ? 1 : 0));  // this launch's partitions
    return launch_maybe_pdl(p.join_primary != 0 && !p.work, kern, grid, dim3(NW * 32), SMEM, st, p, tk, tv);
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
