// act_order.cu -- activation column gather for act-order checkpoints whose rows were sorted by
// group (gptq_prepack_act_order): A'[m][k'] = A[m][perm[k']], written once into caller-provided
// workspace so that every column slab of the decode kernel then reads contiguous activations.
//
// The quantization groups of an act-order checkpoint are the row sets {k : g_idx[k] == g} (page
// "增强 vLLM 对 GPTQv2 格式的支持：分析与实现", section "LLM 的权重量化"); after sorting the rows
// by group, A @ W == A[:, perm] @ W_sorted.
#include <cuda_runtime.h>
#include <stdint.h>

#include "gptq_internal.h"

namespace gptq {
namespace {

// One element per thread-iteration, consecutive threads on consecutive k' of a row: the writes
// and the perm reads coalesce; the reads of A are a gather (A is small and stays in L2).  The
// kernel lets the dependent GEMM launch at once (its CTAs stream weights meanwhile) and waits
// for its own predecessor before reading A.
__global__ void __launch_bounds__(256) k_gather_cols(const uint16_t* __restrict__ A,
                                                     const int32_t* __restrict__ perm, int M, int K,
                                                     uint16_t* __restrict__ out) {
  asm volatile("griddepcontrol.launch_dependents;" ::: "memory");
  asm volatile("griddepcontrol.wait;" ::: "memory");
  const long long total = static_cast<long long>(M) * K;
  const long long step = static_cast<long long>(gridDim.x) * blockDim.x;
  for (long long i = static_cast<long long>(blockIdx.x) * blockDim.x + threadIdx.x; i < total; i += step) {
    const int m = static_cast<int>(i / K), k = static_cast<int>(i - static_cast<long long>(m) * K);
    int src = __ldg(perm + k);
    src = src < 0 ? 0 : (src >= K ? K - 1 : src);        // a bad entry never reads outside the row
    out[i] = __ldg(A + static_cast<long long>(m) * K + src);
  }
}

}  // namespace

cudaError_t launch_gather_cols(const void* A, const int32_t* perm, int M, int K, void* out,
                               cudaStream_t stream) {
  const long long total = static_cast<long long>(M) * K;
  long long blocks = (total + 255) / 256;
  const long long cap = static_cast<long long>(device_info().sm_count) * 8;
  if (blocks > cap) blocks = cap;
  cudaLaunchConfig_t cfg = {};
  cfg.gridDim = dim3(static_cast<unsigned>(blocks), 1, 1);
  cfg.blockDim = dim3(256, 1, 1);
  cfg.stream = stream;
  cudaLaunchAttribute attr[1];
  attr[0].id = cudaLaunchAttributeProgrammaticStreamSerialization;
  attr[0].val.programmaticStreamSerializationAllowed = 1;
  cfg.attrs = attr;
  cfg.numAttrs = 1;
  return cudaLaunchKernelEx(&cfg, k_gather_cols, static_cast<const uint16_t*>(A), perm, M, K,
                            static_cast<uint16_t*>(out));
}

}  // namespace gptq
