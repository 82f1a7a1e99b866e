// decode_b4.cu -- 4-bit instantiations of the decode kernel (kept in their own
// translation unit so the widths compile in parallel).
#include "decode.cuh"
#include "decode_mma.cuh"

namespace gptq {
cudaError_t launch_decode_b4(const Problem& p, cudaStream_t stream) {
  return decode::launch_bits<4>(p, stream);
}
}  // namespace gptq
