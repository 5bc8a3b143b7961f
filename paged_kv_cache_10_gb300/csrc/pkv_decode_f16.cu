// pkv_decode_f16.cu -- decode attention instantiations for f16 pools (f16 q).
#include "pkv_decode_impl.cuh"

namespace pkv {
cudaError_t launch_decode_f16(const DecodeParams& p, int G, cudaStream_t st) {
    return launch_decode_family<F16, F16>(p, G, st);
}
}  // namespace pkv
