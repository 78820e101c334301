// bf16 pool instantiations of the decode kernel (bf16 elements carried as raw 16-bit words).
#include "pa_decode_launch.cuh"

namespace pa {
cudaError_t launch_decode_bf16(const DecodeParams& p, int D, int B, int G, cudaStream_t s) {
    return launch_decode_typed<unsigned short>(p, D, B, G, s);
}
}  // namespace pa
