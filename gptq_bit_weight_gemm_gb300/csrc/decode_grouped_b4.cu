// decode_grouped_b4.cu -- 4-bit instantiations of the grouped (one weight per expert) decode
// kernel, in their own translation unit so that they compile in parallel with the rest.
#include "decode.cuh"
#include "decode_mma.cuh"

namespace gptq {
cudaError_t launch_decode_grouped_b4(const Problem& p, cudaStream_t stream) {
  return decode::launch_grouped_bits<4>(p, stream);
}
}  // namespace gptq
