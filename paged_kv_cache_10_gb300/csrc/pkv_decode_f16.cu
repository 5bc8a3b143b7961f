// pkv_decode_f16.cu -- decode attention instantiations for f16 pools (f16 q).
#include "pkv_decode_mma.cuh"

namespace pkv {
cudaError_t launch_decode_f16(const DecodeParams& p, int G, cudaStream_t st) {
    return launch_decode_family<F16, F16>(p, G, st);
}
cudaError_t launch_decode_mma_f16(const DecodeParams& p, int G, const CUtensorMap& tk, const CUtensorMap& tv,
                                  cudaStream_t st) {
    return launch_decode_mma_family<F16, F16>(p, G, tk, tv, st);
}
}  // namespace pkv
