// prefill.cu -- large-M path (interim): runs the decode kernel on 16-row slices of A.
#include "gptq_internal.h"

namespace gptq {

cudaError_t launch_decode(const Problem& p, cudaStream_t stream);

cudaError_t launch_prefill(const Problem& p, cudaStream_t stream) {
  const size_t es = 2;
  for (int m0 = 0; m0 < p.M; m0 += kDecodeMaxM) {
    Problem s = p;
    s.M = p.M - m0 < kDecodeMaxM ? p.M - m0 : kDecodeMaxM;
    s.A = static_cast<const char*>(p.A) + static_cast<size_t>(m0) * p.K * es;
    s.out = static_cast<char*>(p.out) + static_cast<size_t>(m0) * p.N * es;
    cudaError_t e = launch_decode(s, stream);
    if (e != cudaSuccess) return e;
  }
  return cudaSuccess;
}

}  // namespace gptq
