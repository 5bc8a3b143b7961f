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
};

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

// Log-sum-exp merge of split-K partials into out (q dtype).
cudaError_t launch_merge(const DecodeParams& p, int q_dtype, cudaStream_t st);

int num_sms();

}  // namespace pkv
