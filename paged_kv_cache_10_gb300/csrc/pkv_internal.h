// pkv_internal.h -- host-side declarations shared by the library's
// translation units (not part of the public ABI).
#pragma once

#include <cstddef>
#include <cstdint>

#include <cuda.h>
#include <cuda_runtime.h>

#include "../../include/pagedkv.h"

namespace pkv {

constexpr int kBlockSize = 16;
constexpr int kMaxDevices = 64;
// Smallest partition the automatic choice uses (sizes the P = 0 workspace).
constexpr int kAutoMinPartition = 256;

// Arguments of one decode launch, already validated on the host.
struct DecodeParams {
    const void* q;
    const void* k_cache;
    const void* v_cache;
    const int32_t* block_tables;
    const int32_t* seq_lens;
    void* out;
    float* part_m;   // [S][Hq][NP]   running max, log2 domain
    float* part_l;   // [S][Hq][NP]   sum of exp2(score - m)
    float* part_o;   // [S][Hq][NP][D] normalised partial output
    int32_t S, Hq, Hkv, D, NB, MB;
    int32_t P;        // tokens per partition (multiple of kBlockSize)
    int32_t NP;       // partitions in the grid (ceil(max_seq_len / P), >= 1)
    float qk_scale;   // scale * log2(e) * k_scale
    float v_scale;    // 1 for f16/bf16 pools
    unsigned int* err;
    // Shared-prefix (cascade) decode: a sequence in group g >= 0 starts its
    // own attention at token group_blocks[g] * 16 (the prefix is attended by
    // the prefix kernel); partials of this launch go to partition index
    // part_base + p, and with cascade != 0 the output is never written
    // directly (the merge always runs).  All null / 0 for plain decode.
    const int32_t* seq_group = nullptr;
    const int32_t* group_blocks = nullptr;
    int32_t part_base = 0;
    int32_t cascade = 0;
    // Fused append (pkv_paged_attention_decode_append): one new token per
    // batch row, slots[s] < 0 for none.  All null for plain decode.
    const void* k_new = nullptr;  // [S][Hkv][D], in_dtype
    const void* v_new = nullptr;
    const int64_t* slots = nullptr;
    const int32_t* cow_src = nullptr;  // [S]: block copied into the row's last block first, or -1
    int32_t in_dtype = 0;
    float k_enc_scale = 1.f;  // fp8 caches: code = e4m3(x / scale)
    float v_enc_scale = 1.f;
    // Optional CTA order (host plan): CTA i takes unit work[i / Hkv] =
    // s * (NP - part_base) + partition and KV head i % Hkv; null: the grid
    // (partition, KV head, sequence).
    const int32_t* work = nullptr;
    int32_t num_work = 0;
    // Cascade decode: this launch is a programmatic dependent of the prefix
    // pass before it on the stream.  The grid gets one more z-layer; its CTA
    // (0, 0, S) waits for the prefix pass to complete, so this grid completes
    // after it and a programmatic dependent of this grid (the merge) sees both.
    int32_t join_primary = 0;
};

// Launches kern on st, as a programmatic dependent of the kernel before it
// when pdl is set (a plain launch where the driver refuses the attribute).
template <typename... Params, typename... Args>
cudaError_t launch_maybe_pdl(bool pdl, void (*kern)(Params...), dim3 grid, dim3 block, size_t smem, cudaStream_t st,
                             Args&&... args) {
    if (pdl) {
        cudaLaunchConfig_t cfg = {};
        cfg.gridDim = grid;
        cfg.blockDim = block;
        cfg.dynamicSmemBytes = smem;
        cfg.stream = st;
        cudaLaunchAttribute la[1];
        la[0].id = cudaLaunchAttributeProgrammaticStreamSerialization;
        la[0].val.programmaticStreamSerializationAllowed = 1;
        cfg.attrs = la;
        cfg.numAttrs = 1;
        const cudaError_t e = cudaLaunchKernelEx(&cfg, kern, args...);
        if (e != cudaErrorNotSupported && e != cudaErrorInvalidValue) return e;
        (void)cudaGetLastError();
    }
    kern<<<grid, block, smem, st>>>(args...);
    return cudaGetLastError();
}

// First token of a sequence's own (non-shared) attention range, clamped
// into [0, L] on whole blocks; out-of-range group data reports
// PKV_DEVERR_SEQ_LEN through the caller.
__host__ __device__ inline int own_start(const int32_t* seq_group, const int32_t* group_blocks, int s, int L,
                                         bool* bad) {
    if (!seq_group) return 0;
    const int g = seq_group[s];
    if (g < 0) return 0;
    int start = group_blocks[g] * kBlockSize;
    if (start < 0 || start > L) {
        *bad = true;
        start = start < 0 ? 0 : (L / kBlockSize) * kBlockSize;
    }
    return start;
}

// Device address of the error word on the current device (cached).
unsigned int* error_word();

// Launchers, one translation unit per element-type family.  They return a
// cudaError_t of the launch(es); PKV_ERR_UNSUPPORTED shapes never reach them.
cudaError_t launch_decode_f16(const DecodeParams& p, int G, cudaStream_t st);
cudaError_t launch_decode_bf16(const DecodeParams& p, int G, cudaStream_t st);
cudaError_t launch_decode_fp8_bf16q(const DecodeParams& p, int G, cudaStream_t st);
cudaError_t launch_decode_fp8_f16q(const DecodeParams& p, int G, cudaStream_t st);

// Tensor-core launchers for grouped-query attention (G in {2, 4, 8},
// head_size 128); tk / tv map the K / V pools as 2-D [NB*Hkv*16 rows][128]
// tensors with a 128-byte inner box and the 128-byte swizzle.
cudaError_t launch_decode_mma_f16(const DecodeParams& p, int G, const CUtensorMap& tk, const CUtensorMap& tv,
                                  cudaStream_t st);
cudaError_t launch_decode_mma_bf16(const DecodeParams& p, int G, const CUtensorMap& tk, const CUtensorMap& tv,
                                   cudaStream_t st);
cudaError_t launch_decode_mma_fp8_bf16q(const DecodeParams& p, int G, const CUtensorMap& tk, const CUtensorMap& tv,
                                        cudaStream_t st);
cudaError_t launch_decode_mma_fp8_f16q(const DecodeParams& p, int G, const CUtensorMap& tk, const CUtensorMap& tv,
                                       cudaStream_t st);
// Tensor-core decode of grouped heads at head_size 128 for the pool type
// (the warp-level MMA kernel).
cudaError_t launch_decode_gqa(const DecodeParams& p, int G, int kv_dtype, int q_dtype, const CUtensorMap& tk,
                              const CUtensorMap& tv, cudaStream_t st);

// Shared-prefix (cascade) decode: the prefix pass over each group's shared
// leading blocks, kPrefixPartitionBlocks blocks per prefix partition.  Wide
// partitions leave SMs to the own-token decode running beside the prefix
// pass (1024 tokens: graph step 48.8 -> 43.4 us against 512 on the
// 128-sequence, 2048-token-prefix batch; 256 tokens: 59.0 us).
constexpr int kPrefixPartitionBlocks = 64;  // 1024 tokens
int prefix_partitions(int blocks);
struct CascadeParams {
    DecodeParams base;
    const int32_t* group_offsets;  // [num_groups + 1] into group_members
    const int32_t* group_members;  // batch rows, group by group
    int32_t G;
    int32_t row_chunks;  // CTAs per (group, KV head, prefix partition) along rows (128 rows each)
    int32_t npp;         // prefix partitions (partition indices [0, npp))
    // The 16-bit pool the prefix pass reads (the caller's pool, or the
    // staged copy of an fp8 pool): its block table (rows of the groups'
    // first members), block count and scales.
    const int32_t* prefix_tables;
    int32_t prefix_nb;
    float prefix_qk_scale;  // scale * log2(e) (* k_scale for a staged copy)
    float prefix_o_scale;   // 1, or v_scale for a staged copy
};
// tq: q as [S][Hq][D] with a box of 64 x G x 1 (encode_token_head_map); tk,
// tv: the 16-bit pool the prefix pass reads, in q's type.
cudaError_t launch_cascade_prefix_tc(const CascadeParams& cp, int num_groups, int q_dtype, int D, const CUtensorMap& tq,
                                     const CUtensorMap& tk, const CUtensorMap& tv, cudaStream_t st);

// Cascade decode over an fp8 E4M3 pool: the tcgen05 prefix pass reads a
// 16-bit copy (q's type) of every group's shared blocks, made first by
// launch_cascade_stage_fp8: copy block g * MGB + j holds block j of group g's
// prefix, and the first member's row of the copy's [S][MB] table names it.
struct CascadeStage {
    int64_t table_off, k_off, v_off, bytes;  // from the start of the staging area
};
CascadeStage cascade_stage_layout(int64_t S, int64_t MB, int64_t num_groups, int64_t MGB, int64_t Hkv, int64_t D);
cudaError_t launch_cascade_stage_fp8(const CascadeParams& cp, int num_groups, int MGB, int q_dtype,
                                     const void* k_cache, const void* v_cache, void* staging, cudaStream_t st);

// Log-sum-exp merge of split-K partials into out (q dtype).
cudaError_t launch_merge(const DecodeParams& p, int q_dtype, cudaStream_t st);

// Host helpers shared by the entry points (pkv_api.cu).
int auto_partition(int S, int Hkv, int max_seq_len, bool planned);
bool encode_pool_map(CUtensorMap* map, const void* base, int elem_bytes, int64_t rows, int D);
// 3-D view of a 16-bit [T][H][D] tensor with a box of 64 elements x box_h x
// box_t and the 128-byte swizzle (a box lands as box_t * box_h rows of 128
// bytes, token-major).
bool encode_token_head_map(CUtensorMap* map, const void* base, int D, int H, int64_t T, int box_h, int box_t);
// Partials of S*Hq rows x NP partitions: m, l (256-byte aligned regions), o.
size_t partials_bytes(int64_t S, int64_t Hq, int64_t D, int64_t NP);
void partials_layout(DecodeParams& p, void* workspace);  // sets part_m/l/o from S, Hq, NP

int num_sms();

}  // namespace pkv
