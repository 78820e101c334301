// fp32 pool instantiations of the decode kernel.
#include "pa_decode_launch.cuh"

namespace pa {
cudaError_t launch_decode_f32(const DecodeParams& p, int D, int B, int G, cudaStream_t s) {
    return launch_decode_typed<float>(p, D, B, G, s);
}
}  // namespace pa
