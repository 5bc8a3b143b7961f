// pkv_append.cuh -- the slot-mapped KV write of one token row, shared by the
// append kernels and the decode kernels' fused append.
//
// A new token's K/V row goes to block slot / 16, offset slot % 16 of the
// [NB][Hkv][16][D] pools ("vLLM：大语言模型推理与服务库" section 4.3; "vLLM 高性能
// 大语言模型推理引擎深度技术评估与分布式架构展望": each decode step appends the
// new token's KV vector).  An fp8 E4M3 cache stores
// e4m3_rn_satfinite(x / scale), the division in IEEE binary32.
#pragma once

#include <cstdint>

#include "pkv_device.cuh"

namespace pkv {

// Eight 16-bit input elements (one 16-byte vector) to eight E4M3 codes.
template <typename IT>
__device__ __forceinline__ uint2 encode_e4m3x8(uint4 x, float scale) {
    float f[8];
    const uint32_t w[4] = {x.x, x.y, x.z, x.w};
    Unpack<IT, 8>::run(w, f);
    uint32_t out[2];
#pragma unroll
    for (int j = 0; j < 2; ++j) {
        uint32_t word = 0;
#pragma unroll
        for (int e = 0; e < 2; ++e) {
            const float2 pr = make_float2(__fdiv_rn(f[4 * j + 2 * e], scale), __fdiv_rn(f[4 * j + 2 * e + 1], scale));
            const __nv_fp8x2_storage_t c2 = __nv_cvt_float2_to_fp8x2(pr, __NV_SATFINITE, __NV_E4M3);
            word |= static_cast<uint32_t>(c2) << (16 * e);
        }
        out[j] = word;
    }
    return make_uint2(out[0], out[1]);
}

// Decode with a fused append (pkv_paged_attention_decode_append).  Of the
// CTA whose partition covers batch row s's last position L - 1, the warp
// that streams the block holding that position writes its KV head h's row of
// the step's new token (row s of k_new / v_new, [S][Hkv][D]) to
// slot_mapping[s] just before it copies that block, so no other warp waits.
// With copy-on-write (cow_src[s] >= 0: the row's last block is a fresh copy
// of a shared block, [P4] "Prefix Caching 与 Copy-on-Write"), the same warp
// first copies its head's tile of the source block into it.  The slot must
// be the one the block table maps position L - 1 to (else PKV_DEVERR_SLOT),
// the source block inside the pool (else PKV_DEVERR_COPY_PAIR); otherwise
// nothing is written for the row.
struct FusedRow {
    int64_t drow;  // destination row (token of one head) in the pool; -1: nothing to write
    int32_t src;   // copy-on-write source block, or -1
    int32_t blk;   // destination block
    uint4 x;       // this lane's 16-byte input chunk (lane < 2 * D / 8: K chunks, then V)
};

// Reads what the write needs at the start (the loads' latency passes while
// the warp streams its earlier blocks).  `on`: warp-uniform.
__device__ __forceinline__ FusedRow fused_prefetch(const DecodeParams& p, int s, int h, int L, bool on) {
    FusedRow r{-1, -1, -1, make_uint4(0u, 0u, 0u, 0u)};
    if (!on || L <= 0) return r;
    const int64_t slot = __ldg(p.slots + s);
    if (slot < 0) return r;
    const int32_t src = p.cow_src ? __ldg(p.cow_src + s) : -1;
    const int lane = threadIdx.x & 31, chunks = p.D / 8;
    if (lane < 2 * chunks) {
        const int which = lane / chunks, c = lane - which * chunks;
        r.x = __ldg(reinterpret_cast<const uint4*>(static_cast<const unsigned char*>(which ? p.v_new : p.k_new) +
                                                   (static_cast<int64_t>(s) * p.Hkv + h) * p.D * 2) + c);
    }
    const int pos = L - 1;
    const int32_t blk = __ldg(p.block_tables + static_cast<int64_t>(s) * p.MB + pos / kBlockSize);
    if (blk < 0 || blk >= p.NB || slot / kBlockSize != blk || slot % kBlockSize != pos % kBlockSize) {
        if (lane == 0) report(p.err, PKV_DEVERR_SLOT);
        return r;
    }
    if (src >= p.NB || (src >= 0 && src == blk)) {
        if (lane == 0) report(p.err, PKV_DEVERR_COPY_PAIR);
        return r;
    }
    r.src = src;
    r.blk = blk;
    r.drow = (static_cast<int64_t>(blk) * p.Hkv + h) * kBlockSize + pos % kBlockSize;
    return r;
}

// Writes the row (warp-uniform call) and orders it before the warp's
// following TMA copies (the caller's __syncwarp then the copy).
template <typename KT>
__device__ __forceinline__ void fused_commit(const DecodeParams& p, int h, const FusedRow& r) {
    if (r.drow < 0) return;
    const int lane = threadIdx.x & 31, chunks = p.D / 8;
    if (r.src >= 0) {
        // copy-on-write: this head's tile of the source block, except the
        // appended row (written below), for K and V
        const int row_chunks = p.D * KT::bytes / 16;  // 16-byte chunks of one token row
        const int tile_chunks = kBlockSize * row_chunks;
        const int skip = static_cast<int>(r.drow % kBlockSize);
        const int64_t src_tile = (static_cast<int64_t>(r.src) * p.Hkv + h) * tile_chunks;
        const int64_t dst_tile = (static_cast<int64_t>(r.blk) * p.Hkv + h) * tile_chunks;
        for (int which = 0; which < 2; ++which) {
            const uint4* sp = reinterpret_cast<const uint4*>(which ? p.v_cache : p.k_cache) + src_tile;
            uint4* dp = const_cast<uint4*>(reinterpret_cast<const uint4*>(which ? p.v_cache : p.k_cache)) + dst_tile;
            for (int i = lane; i < tile_chunks; i += 32)
                if (i / row_chunks != skip) dp[i] = __ldg(sp + i);
        }
    }
    if (lane < 2 * chunks) {
        const int which = lane / chunks, c = lane - which * chunks;
        unsigned char* pool = const_cast<unsigned char*>(static_cast<const unsigned char*>(which ? p.v_cache : p.k_cache));
        if constexpr (KT::bytes == 2) {
            reinterpret_cast<uint4*>(pool + r.drow * p.D * 2)[c] = r.x;
        } else {
            const float sc = which ? p.v_enc_scale : p.k_enc_scale;
            reinterpret_cast<uint2*>(pool + r.drow * p.D)[c] =
                p.in_dtype == PKV_BF16 ? encode_e4m3x8<BF16>(r.x, sc) : encode_e4m3x8<F16>(r.x, sc);
        }
    }
    asm volatile("fence.proxy.async.global;" ::: "memory");
}

}  // namespace pkv
