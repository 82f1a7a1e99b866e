// gptq_internal.h -- host-side launch interface between the C ABI (gptq_api.cu) and the
// kernels.  Not installed; the public interface is include/gptq.h.
#pragma once

#include <cuda_runtime.h>
#include <stddef.h>
#include <stdint.h>

namespace gptq {

// A validated problem: every field checked by the C ABI before a launcher sees it.
struct Problem {
  const void* A;             // [M, K] fp16/bf16 (gemm) or nullptr
  int M, K, N;
  int dtype;                 // 0 fp16, 1 bf16 (activations / outputs)
  const int32_t* qweight;    // [K*bits/32, N]
  const int32_t* qzeros;     // [G, N*bits/32]
  const void* scales;        // [G, N] fp16
  const int32_t* g_idx;      // [K] or nullptr
  const int32_t* perm;       // [K] or nullptr: A column of each weight row (prepacked act-order)
  int bits;
  int group;                 // K when the caller passed -1
  int G;
  int zero_offset;           // 1 for GPTQv1, 0 for GPTQv2
  void* out;                 // C [M, N] or W [K, N]
  unsigned* status;          // device status word of the current device
  // grouped GEMM (one weight per expert, stacked [E][...]): device row offsets [E + 1] into A
  // and C, E experts, `rows` rows in A and C; M is then the bound on any expert's rows
  const int32_t* offsets;
  int E;
  int rows;
  // caller workspace (the tensor-core kernel with bf16 activations: the fp16 copy of A and its
  // row scales, prefill_workspace_bytes)
  void* workspace;
  size_t workspace_bytes;
  // qweight is in the interleaved layout of gptq_prepack_interleave (decode kernels only)
  bool interleaved;
  // nullable: the kernels do nothing unless *run_flag == run_when (a device flag written by an
  // earlier kernel of the same stream)
  const int* run_flag;
  int run_when;
  // launch without programmatic dependent launch: the kernel starts once the previous kernel has
  // completed (needed when it reads weights that the previous kernels wrote)
  bool no_pdl;
  // decode kernels: the tokens in blocks of the kernel's token tile, one block per grid z (0/1:
  // one block), all reading the same weights
  int tok_split;
};

struct DeviceInfo {
  int device;
  int sm_count;
  int cc_major, cc_minor;
  size_t smem_optin;         // max dynamic shared memory per block (opt-in)
};

const DeviceInfo& device_info();   // current device, cached

cudaError_t launch_dequant(const Problem& p, cudaStream_t stream);
cudaError_t launch_decode(const Problem& p, cudaStream_t stream);
cudaError_t launch_decode_grouped(const Problem& p, cudaStream_t stream);
cudaError_t launch_prefill(const Problem& p, cudaStream_t stream);
// Workspace the tensor-core kernel needs for bf16 activations of M x K (0 for fp16).
size_t prefill_workspace_bytes(int M, int K);
cudaError_t launch_gather_cols(const void* A, const int32_t* perm, int M, int K, void* out,
                               cudaStream_t stream);
// Act-order on the device: the stable sort of the rows by g_idx (perm; src, the packed word and
// bit offset of each sorted row's code; flag = 1 when every group holds exactly `group` rows,
// else 0) and the packed weight rewritten in that order (only when the flag is 1; with flag 0 and
// a non-null status the repack raises kStatusGidxGroups there).  Shared memory per CTA is at most
// kMaxActOrderSmem; sort_groups_fits and repack_strip_width (0: no strip fits) say whether a
// shape qualifies.
constexpr size_t kMaxActOrderSmem = 200 * 1024;
bool sort_groups_fits(int K, int G, int group);
int repack_strip_width(int K, int bits);
cudaError_t launch_sort_groups(const int32_t* g_idx, int K, int G, int group, int bits, int32_t* perm,
                               uint32_t* src, int* flag, cudaStream_t stream);
cudaError_t launch_repack_rows(const int32_t* qweight, const uint32_t* src, const int* flag, int K, int N,
                               int bits, int32_t* out, unsigned* status, cudaStream_t stream);
cudaError_t launch_wait_selftest(unsigned* status, uint64_t limit_ns, int* flag, cudaStream_t stream);

struct QuantProblem {
  const float* W;
  int K, N, bits, group, G;
  const int32_t* g_idx;
  int sym, fmt;
  int32_t* qweight;
  int32_t* qzeros;
  void* scales;
  unsigned* status;
};
cudaError_t launch_quantize(const QuantProblem& q, cudaStream_t stream);
// An empty kernel launched without programmatic dependent launch: after it, a GEMM kernel that
// reads the checkpoint before its dependency wait sees everything the kernels before it wrote.
cudaError_t launch_writer_fence(cudaStream_t stream);

// cuTensorMapEncodeTiled through the runtime's driver entry point (no libcuda link); false if
// the driver refuses the map.  `dtype` is a CUtensorMapDataType, `swizzle` a CUtensorMapSwizzle.
bool encode_tensor_map(void* tmap, int dtype, void* base, const uint64_t* dims,
                       const uint64_t* strides, const uint32_t* box, const uint32_t* estr,
                       int swizzle);

// Largest M handled by the decode (split-K, weight-streaming) kernels; larger M goes to the
// tensor-core tile kernel.
constexpr int kDecodeMaxM = 32;

}  // namespace gptq
