// decode_b2.cu -- 2-bit instantiations of the decode kernel (kept in their own
// translation unit so the widths compile in parallel).
#include "decode.cuh"
#include "decode_mma.cuh"

namespace gptq {
cudaError_t launch_decode_b2(const Problem& p, cudaStream_t stream) {
  return decode::launch_bits<2>(p, stream);
}
}  // namespace gptq
