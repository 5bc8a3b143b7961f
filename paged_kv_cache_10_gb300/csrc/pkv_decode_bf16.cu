// pkv_decode_bf16.cu -- decode attention instantiations for bf16 pools (bf16 q).
#include "pkv_decode_mma.cuh"

namespace pkv {
cudaError_t launch_decode_bf16(const DecodeParams& p, int G, cudaStream_t st) {
    return launch_decode_family<BF16, BF16>(p, G, st);
}
cudaError_t launch_decode_mma_bf16(const DecodeParams& p, int G, const CUtensorMap& tk, const CUtensorMap& tv,
                                  cudaStream_t st) {
    return launch_decode_mma_family<BF16, BF16>(p, G, tk, tv, st);
}
}  // namespace pkv
