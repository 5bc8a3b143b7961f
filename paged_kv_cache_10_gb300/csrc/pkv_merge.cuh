// pkv_merge.cuh -- log-sum-exp merge of split-K decode partials.
//
// The pages give only the partition axis of the decode grid (openEuler essay
// on vLLM, "PagedAttention：把操作系统的分页搬上 GPU": grid (num_heads,
// num_seqs, max_num_partitions)); the reduce is the standard log-sum-exp
// identity over the partitions' (max, sum, normalised output).
#pragma once

#include "pkv_device.cuh"

namespace pkv {

constexpr unsigned kMergeFull = 0xffffffffu;

// Partition range [first, first + nparts) that the merge combines for one
// (sequence, query head) row, with the main kernels' clamping of the
// sequence length.  nparts <= 1 outside cascade decode means the main
// kernel wrote the row itself.
__device__ __forceinline__ void merge_row_range(const DecodeParams& p, int64_t row, int& first, int& nparts) {
    const int s = static_cast<int>(row / p.Hq);
    int L = __ldg(p.seq_lens + s);
    const int Lcap = p.MB * kBlockSize;
    L = L < 0 ? 0 : (L > Lcap ? Lcap : L);
    bool bad = false;
    const int start = own_start(p.seq_group, p.group_blocks, s, L, &bad);
    const int Lown = min(L - start, (p.NP - p.part_base) * p.P);
    const int nown = Lown > 0 ? (Lown + p.P - 1) / p.P : 0;
    if (!p.cascade) {
        first = 0;
        nparts = nown > 0 ? nown : 1;
    } else {
        first = start > 0 ? 0 : p.part_base;  // prefix partials only for group members
        nparts = p.part_base + nown - first;
    }
}

constexpr int kMergeChunk = 8;  // partitions whose loads one warp keeps in flight

// Log-sum-exp merge of the split-K partials of one (sequence, query head)
// row: M = max_p m_p, w_p = l_p 2^(m_p - M), out = sum_p w_p o_p / sum_p w_p,
// over the partials' (max, sum, normalised output).  WPR warps share a row
// (256-thread CTAs, 8 / WPR rows each); warp w of a row takes the row's
// partitions w, w + WPR, ... in chunks of kMergeChunk.  For a chunk, lane u
// loads (m, l) of its u-th partition while every lane loads its D / 32 head
// dimensions of all the chunk's partial outputs, so one round of independent
// loads covers the chunk; the weights are then broadcast by shuffles.  A
// warp keeps its own running maximum; the WPR warps of a row are combined
// through shared memory by the same identity.  Empty partials (l = 0) carry
// no data and are skipped, never multiplied (their output may be stale).
template <int D, typename QT, int WPR>
__global__ void __launch_bounds__(256) merge_kernel(const DecodeParams p) {
    constexpr int VD = D / 32;  // head dimensions per lane (4 or 2)
    constexpr int RPC = 8 / WPR;  // rows per CTA
    __shared__ float red_acc[WPR > 1 ? 8 : 1][D];
    __shared__ float red_m[8], red_den[8];
    const int warp = threadIdx.x >> 5, lane = threadIdx.x & 31;
    const int wr = warp % WPR;  // this warp's share of the row
    const int64_t rows = static_cast<int64_t>(p.S) * p.Hq;
    const int64_t row = static_cast<int64_t>(blockIdx.x) * RPC + warp / WPR;
    int first = 0, nparts = 0;
    if (row < rows) merge_row_range(p, row, first, nparts);
    const bool active = row < rows && (p.cascade || nparts > 1);
    wait_primary_grid();  // every CTA waits, so this grid never completes before its producer

    float acc[VD];
#pragma unroll
    for (int v = 0; v < VD; ++v) acc[v] = 0.f;
    float den = 0.f, M = -INFINITY;
    if (active) {
        const float* pm = p.part_m + row * p.NP + first;
        const float* pl = p.part_l + row * p.NP + first;
        const float* po = p.part_o + (row * p.NP + first) * D + lane * VD;
        const int mine = nparts > wr ? (nparts - wr + WPR - 1) / WPR : 0;  // this warp's partitions
        for (int c0 = 0; c0 < mine; c0 += kMergeChunk) {
            const int cnt = min(kMergeChunk, mine - c0);
            float m_u = -INFINITY, l_u = 0.f;
            if (lane < cnt) {
                const int j = wr + (c0 + lane) * WPR;
                l_u = __ldg(pl + j);
                m_u = __ldg(pm + j);
            }
            float o[kMergeChunk][VD];
#pragma unroll
            for (int u = 0; u < kMergeChunk; ++u) {
                if (u < cnt) {
                    const float* src = po + static_cast<int64_t>(wr + (c0 + u) * WPR) * D;
                    if constexpr (VD == 4) {
                        const float4 x = __ldg(reinterpret_cast<const float4*>(src));
                        o[u][0] = x.x; o[u][1] = x.y; o[u][2] = x.z; o[u][3] = x.w;
                    } else {
                        const float2 x = __ldg(reinterpret_cast<const float2*>(src));
                        o[u][0] = x.x; o[u][1] = x.y;
                    }
                } else {
#pragma unroll
                    for (int v = 0; v < VD; ++v) o[u][v] = 0.f;
                }
            }
            if (!(l_u > 0.f)) m_u = -INFINITY;
            float cm = m_u;
#pragma unroll
            for (int mask = 1; mask < kMergeChunk; mask <<= 1) cm = fmaxf(cm, __shfl_xor_sync(kMergeFull, cm, mask));
            cm = __shfl_sync(kMergeFull, cm, 0);
            const float Mn = fmaxf(M, cm);
            if (Mn == -INFINITY) continue;  // nothing but empty partials so far
            if (Mn != M) {  // rescale what was accumulated against the old maximum
                const float a = exp2f(M - Mn);  // M = -inf: 0, with nothing accumulated
#pragma unroll
                for (int v = 0; v < VD; ++v) acc[v] *= a;
                den *= a;
                M = Mn;
            }
            const float w_u = m_u == -INFINITY ? 0.f : l_u * exp2f(m_u - M);
#pragma unroll
            for (int u = 0; u < kMergeChunk; ++u) {
                const float w = __shfl_sync(kMergeFull, w_u, u);
                if (w > 0.f) {
#pragma unroll
                    for (int v = 0; v < VD; ++v) acc[v] = fmaf(w, o[u][v], acc[v]);
                    den += w;
                }
            }
        }
    }

    auto* out = reinterpret_cast<typename QT::storage*>(p.out) + row * D;
    if constexpr (WPR == 1) {
        if (active) {
#pragma unroll
            for (int v = 0; v < VD; ++v) out[lane * VD + v] = from_float<QT>(den > 0.f ? acc[v] / den : 0.f);
        }
    } else {
        // combine the row's warps: rescale each warp's sums to the row maximum
#pragma unroll
        for (int v = 0; v < VD; ++v) red_acc[warp][lane * VD + v] = acc[v];
        if (lane == 0) {
            red_m[warp] = M;
            red_den[warp] = den;
        }
        __syncthreads();
        if (active) {
            const int w0 = warp - wr;  // first warp of this row
            float Mr = -INFINITY;
#pragma unroll
            for (int w = 0; w < WPR; ++w) Mr = fmaxf(Mr, red_m[w0 + w]);
            float sc[WPR], dn = 0.f;
#pragma unroll
            for (int w = 0; w < WPR; ++w) {
                sc[w] = red_m[w0 + w] == -INFINITY ? 0.f : exp2f(red_m[w0 + w] - Mr);
                dn = fmaf(sc[w], red_den[w0 + w], dn);
            }
            // the row's warps split its D head dimensions for the output
            for (int d = wr * 32 + lane; d < D; d += WPR * 32) {
                float a = 0.f;
#pragma unroll
                for (int w = 0; w < WPR; ++w) a = fmaf(sc[w], red_acc[w0 + w][d], a);
                out[d] = from_float<QT>(dn > 0.f ? a / dn : 0.f);
            }
        }
    }
}

// Warps per row for a launch whose rows have at most NP partitions: enough
// that one round of loads covers a row of up to 64 partitions.
inline int merge_warps_per_row(int NP) { return NP <= 8 ? 1 : (NP <= 16 ? 2 : (NP <= 32 ? 4 : 8)); }

}  // namespace pkv
