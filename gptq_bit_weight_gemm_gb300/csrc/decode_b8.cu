// decode_b8.cu -- 8-bit instantiations of the decode kernel (kept in their own
// translation unit so the widths compile in parallel).
#include "decode.cuh"
#include "decode_mma.cuh"

namespace gptq {
cudaError_t launch_decode_b8(const Problem& p, cudaStream_t stream) {
  return decode::launch_bits<8>(p, stream);
}
}  // namespace gptq
