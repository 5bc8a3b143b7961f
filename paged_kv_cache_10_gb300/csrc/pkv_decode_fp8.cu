// pkv_decode_fp8.cu -- decode attention instantiations for fp8 E4M3 pools
// (bf16 or f16 q).
#include "pkv_decode_mma.cuh"

namespace pkv {
cudaError_t launch_decode_fp8_bf16q(const DecodeParams& p, int G, cudaStream_t st) {
    return launch_decode_family<E4M3, BF16>(p, G, st);
}
cudaError_t launch_decode_fp8_f16q(const DecodeParams& p, int G, cudaStream_t st) {
    return launch_decode_family<E4M3, F16>(p, G, st);
}
cudaError_t launch_decode_mma_fp8_bf16q(const DecodeParams& p, int G, const CUtensorMap& tk, const CUtensorMap& tv,
                                        cudaStream_t st) {
    return launch_decode_mma_family<E4M3, BF16>(p, G, tk, tv, st);
}
cudaError_t launch_decode_mma_fp8_f16q(const DecodeParams& p, int G, const CUtensorMap& tk, const CUtensorMap& tv,
                                       cudaStream_t st) {
    return launch_decode_mma_family<E4M3, F16>(p, G, tk, tv, st);
}
}  // namespace pkv
