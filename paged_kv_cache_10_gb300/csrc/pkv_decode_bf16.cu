// pkv_decode_bf16.cu -- decode attention instantiations for bf16 pools (bf16 q).
#include "pkv_decode_impl.cuh"

namespace pkv {
cudaError_t launch_decode_bf16(const DecodeParams& p, int G, cudaStream_t st) {
    return launch_decode_family<BF16, BF16>(p, G, st);
}
}  // namespace pkv
