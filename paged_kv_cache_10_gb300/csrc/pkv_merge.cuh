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

// Log-sum-exp merge of the split-K partials, one CTA of kMergeThreads per
// (sequence, query head) row: M = max_p m_p, w_p = l_p 2^(m_p - M),
// out = sum_p w_p o_p / sum_p w_p.  The weights of a chunk of partitions
// are computed once into shared memory; the kMergeThreads / D thread groups
// then each walk every (kMergeThreads / D)-th partition of the chunk for
// their head dimension d with 16 independent loads in flight (each load a
// coalesced row of partial outputs), and the groups' sums are added in
// shared memory.  Rows of single-partition sequences were written by the
// main kernel and are skipped.
template <int D, typename QT, int kMergeThreads>
__global__ void __launch_bounds__(kMergeThreads) merge_kernel(const DecodeParams p) {
    constexpr int NG = kMergeThreads / D;  // thread groups sharing one head dimension
    __shared__ float w_s[kMergeThreads];
    __shared__ float red[kMergeThreads / 32];
    __shared__ float part_acc[kMergeThreads];
    __shared__ float part_den[kMergeThreads];
    const int tid = threadIdx.x, lane = tid & 31, warp = tid >> 5;
    const int d = tid % D, grp = tid / D;
    const int64_t row = blockIdx.x;
    const int s = static_cast<int>(row / p.Hq);
    // same clamping as the main kernels
    int L = __ldg(p.seq_lens + s);
    const int Lcap = p.MB * kBlockSize;
    L = L < 0 ? 0 : (L > Lcap ? Lcap : L);
    bool bad = false;
    const int start = own_start(p.seq_group, p.group_blocks, s, L, &bad);
    const int Lown = min(L - start, (p.NP - p.part_base) * p.P);
    const int nown = Lown > 0 ? (Lown + p.P - 1) / p.P : 0;
    int first, nparts;  // partitions [first, first + nparts) of this row
    if (!p.cascade) {
        first = 0;
        nparts = nown > 0 ? nown : 1;
        if (nparts <= 1) return;  // written by the main kernel
    } else {
        first = start > 0 ? 0 : p.part_base;  // prefix partials only for group members
        nparts = p.part_base + nown - first;
    }
    const float* pm = p.part_m + row * p.NP + first;
    const float* pl = p.part_l + row * p.NP + first;
    const float* po = p.part_o + (row * p.NP + first) * D;

    float M = -INFINITY;
    for (int i = tid; i < nparts; i += kMergeThreads) M = fmaxf(M, pl[i] > 0.f ? pm[i] : -INFINITY);
#pragma unroll
    for (int mask = 16; mask > 0; mask >>= 1) M = fmaxf(M, __shfl_xor_sync(kMergeFull, M, mask));
    if (lane == 0) red[warp] = M;
    __syncthreads();
    M = red[0];
#pragma unroll
    for (int w = 1; w < kMergeThreads / 32; ++w) M = fmaxf(M, red[w]);

    float acc = 0.f, den = 0.f;
    if (M != -INFINITY && nparts > 0) {
        for (int base = 0; base < nparts; base += kMergeThreads) {
            const int cnt = min(kMergeThreads, nparts - base);
            __syncthreads();  // previous chunk's weights fully consumed
            if (tid < cnt) {
                const float l = pl[base + tid];
                w_s[tid] = l > 0.f ? l * exp2f(pm[base + tid] - M) : 0.f;
            }
            __syncthreads();
            const float* o = po + static_cast<int64_t>(base) * D + d;
            int j = grp;
            for (; j + 15 * NG < cnt; j += 16 * NG) {
                float v[16];
#pragma unroll
                for (int u = 0; u < 16; ++u) v[u] = o[(j + u * NG) * D];
#pragma unroll
                for (int u = 0; u < 16; ++u) {
                    const float w = w_s[j + u * NG];
                    acc = w > 0.f ? fmaf(w, v[u], acc) : acc;  // empty partials carry no data
                    den += w;
                }
            }
            for (; j < cnt; j += NG) {
                const float w = w_s[j];
                acc = w > 0.f ? fmaf(w, o[j * D], acc) : acc;
                den += w;
            }
        }
    }
    // combine the groups' partial sums for each head dimension
    part_acc[tid] = acc;
    part_den[tid] = den;
    __syncthreads();
    if (grp == 0) {
        float a = acc, dn = den;
#pragma unroll
        for (int q = 1; q < NG; ++q) {
            a += part_acc[q * D + d];
            dn += part_den[q * D + d];
        }
        auto* out = reinterpret_cast<typename QT::storage*>(p.out) + row * D;
        out[d] = from_float<QT>(dn > 0.f ? a / dn : 0.f);
    }
}

// The same merge with one warp per row, 8 rows per CTA, for rows with few
// partitions (latency-bound: a CTA per row spends its time on its own
// barriers).  Lanes hold the partitions' weights (computed once, broadcast
// by shuffles); each lane accumulates D / 32 consecutive head dimensions
// with vector loads, four partitions in flight.
template <int D, typename QT>
__global__ void __launch_bounds__(256) merge_warp_kernel(const DecodeParams p) {
    constexpr int VD = D / 32;  // head dimensions per lane (4 or 2)
    const int lane = threadIdx.x & 31;
    const int64_t row = static_cast<int64_t>(blockIdx.x) * 8 + (threadIdx.x >> 5);
    if (row >= static_cast<int64_t>(p.S) * p.Hq) return;
    const int s = static_cast<int>(row / p.Hq);
    // same clamping as the main kernels
    int L = __ldg(p.seq_lens + s);
    const int Lcap = p.MB * kBlockSize;
    L = L < 0 ? 0 : (L > Lcap ? Lcap : L);
    bool bad = false;
    const int start = own_start(p.seq_group, p.group_blocks, s, L, &bad);
    const int Lown = min(L - start, (p.NP - p.part_base) * p.P);
    const int nown = Lown > 0 ? (Lown + p.P - 1) / p.P : 0;
    int first, nparts;  // partitions [first, first + nparts) of this row
    if (!p.cascade) {
        first = 0;
        nparts = nown > 0 ? nown : 1;
        if (nparts <= 1) return;  // written by the main kernel
    } else {
        first = start > 0 ? 0 : p.part_base;  // prefix partials only for group members
        nparts = p.part_base + nown - first;
    }
    const float* pm = p.part_m + row * p.NP + first;
    const float* pl = p.part_l + row * p.NP + first;
    const float* po = p.part_o + (row * p.NP + first) * D + lane * VD;

    float acc[VD];
#pragma unroll
    for (int v = 0; v < VD; ++v) acc[v] = 0.f;
    float den = 0.f;
    // partitions in chunks of 32: lane i owns partition base + i
    float M = -INFINITY;
    for (int i = lane; i < nparts; i += 32) M = fmaxf(M, __ldg(pl + i) > 0.f ? __ldg(pm + i) : -INFINITY);
#pragma unroll
    for (int mask = 16; mask > 0; mask >>= 1) M = fmaxf(M, __shfl_xor_sync(kMergeFull, M, mask));
    if (M != -INFINITY) {
        for (int base = 0; base < nparts; base += 32) {
            const int cnt = min(32, nparts - base);
            float w = 0.f;
            if (lane < cnt) {
                const float l = __ldg(pl + base + lane);
                w = l > 0.f ? l * exp2f(__ldg(pm + base + lane) - M) : 0.f;
            }
            for (int j = 0; j < cnt; j += 4) {
                float wj[4];
                float o[4][VD];
#pragma unroll
                for (int u = 0; u < 4; ++u) {
                    wj[u] = __shfl_sync(kMergeFull, w, (j + u) & 31);
                    if (j + u < cnt && wj[u] > 0.f) {
                        const float* src = po + static_cast<int64_t>(base + j + u) * D;
                        if constexpr (VD == 4) {
                            const float4 x = __ldg(reinterpret_cast<const float4*>(src));
                            o[u][0] = x.x; o[u][1] = x.y; o[u][2] = x.z; o[u][3] = x.w;
                        } else {
                            const float2 x = __ldg(reinterpret_cast<const float2*>(src));
                            o[u][0] = x.x; o[u][1] = x.y;
                        }
                    } else {
                        wj[u] = 0.f;  // past the chunk or an empty partial: no data
#pragma unroll
                        for (int v = 0; v < VD; ++v) o[u][v] = 0.f;
                    }
                }
#pragma unroll
                for (int u = 0; u < 4; ++u) {
                    den += wj[u];
#pragma unroll
                    for (int v = 0; v < VD; ++v) acc[v] = fmaf(wj[u], o[u][v], acc[v]);
                }
            }
        }
    }
    auto* out = reinterpret_cast<typename QT::storage*>(p.out) + row * D + lane * VD;
#pragma unroll
    for (int v = 0; v < VD; ++v) out[v] = from_float<QT>(den > 0.f ? acc[v] / den : 0.f);
}

// Rows with at most this many partitions are merged a warp per row; more
// partitions get the CTA-per-row kernel with two thread groups per head
// dimension (more loads in flight per row).
constexpr int kMergeNarrowMaxParts = 16;

}  // namespace pkv
