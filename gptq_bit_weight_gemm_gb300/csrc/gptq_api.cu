// gptq_api.cu -- the C ABI (include/gptq.h): host-side validation, dispatch, the host v1 -> v2
// zero repack and the device status word.
#include <cuda.h>
#include <cudaTypedefs.h>
#include <cuda_runtime.h>

#include <mutex>
#include <vector>

#include "../../include/gptq.h"
#include "gptq_internal.h"

namespace gptq {

cudaError_t launch_decode_b2(const Problem& p, cudaStream_t stream);
cudaError_t launch_decode_b3(const Problem& p, cudaStream_t stream);
cudaError_t launch_decode_b4(const Problem& p, cudaStream_t stream);
cudaError_t launch_decode_b8(const Problem& p, cudaStream_t stream);

cudaError_t launch_decode(const Problem& p, cudaStream_t stream) {
  switch (p.bits) {
    case 2: return launch_decode_b2(p, stream);
    case 3: return launch_decode_b3(p, stream);
    case 4: return launch_decode_b4(p, stream);
    case 8: return launch_decode_b8(p, stream);
    default: return cudaErrorInvalidValue;
  }
}

cudaError_t launch_decode_grouped_b2(const Problem& p, cudaStream_t stream);
cudaError_t launch_decode_grouped_b3(const Problem& p, cudaStream_t stream);
cudaError_t launch_decode_grouped_b4(const Problem& p, cudaStream_t stream);
cudaError_t launch_decode_grouped_b8(const Problem& p, cudaStream_t stream);

cudaError_t launch_decode_grouped(const Problem& p, cudaStream_t stream) {
  switch (p.bits) {
    case 2: return launch_decode_grouped_b2(p, stream);
    case 3: return launch_decode_grouped_b3(p, stream);
    case 4: return launch_decode_grouped_b4(p, stream);
    case 8: return launch_decode_grouped_b8(p, stream);
    default: return cudaErrorInvalidValue;
  }
}

namespace {

constexpr int kMaxDevices = 64;

// One word per device; kernels OR error bits into it (GPTQ_DEV_*).
__device__ unsigned g_device_status;

struct DeviceState {
  std::once_flag once;
  DeviceInfo info;
  unsigned* status = nullptr;
  cudaError_t init_error = cudaSuccess;
};

DeviceState g_devices[kMaxDevices];

DeviceState* current_state(cudaError_t* err) {
  int dev = 0;
  cudaError_t e = cudaGetDevice(&dev);
  if (e != cudaSuccess || dev < 0 || dev >= kMaxDevices) {
    *err = e != cudaSuccess ? e : cudaErrorInvalidDevice;
    return nullptr;
  }
  DeviceState& st = g_devices[dev];
  std::call_once(st.once, [&st, dev]() {
    st.info.device = dev;
    cudaError_t r = cudaDeviceGetAttribute(&st.info.sm_count, cudaDevAttrMultiProcessorCount, dev);
    if (r == cudaSuccess)
      r = cudaDeviceGetAttribute(&st.info.cc_major, cudaDevAttrComputeCapabilityMajor, dev);
    if (r == cudaSuccess)
      r = cudaDeviceGetAttribute(&st.info.cc_minor, cudaDevAttrComputeCapabilityMinor, dev);
    int smem = 0;
    if (r == cudaSuccess)
      r = cudaDeviceGetAttribute(&smem, cudaDevAttrMaxSharedMemoryPerBlockOptin, dev);
    st.info.smem_optin = static_cast<size_t>(smem);
    if (r == cudaSuccess) r = cudaGetSymbolAddress(reinterpret_cast<void**>(&st.status), g_device_status);
    st.init_error = r;
  });
  *err = st.init_error;
  return st.init_error == cudaSuccess ? &st : nullptr;
}

bool aligned(const void* p, size_t a) { return (reinterpret_cast<uintptr_t>(p) % a) == 0; }

bool bits_ok(int bits) { return bits == 2 || bits == 3 || bits == 4 || bits == 8; }

// Shape/argument checks shared by every device entry point; fills p.G and p.group.
int check_common(const int32_t* qweight, const int32_t* qzeros, const void* scales,
                 const int32_t* g_idx, int K, int N, int bits, int group, Problem* p) {
  if (!bits_ok(bits)) return GPTQ_ERR_ARG;
  if (!qweight || !qzeros || !scales) return GPTQ_ERR_ARG;
  if (K <= 0 || N <= 0 || K % 32 || N % 32) return GPTQ_ERR_SHAPE;
  if (group == -1) {
    if (g_idx) return GPTQ_ERR_SHAPE;
    p->group = K;
    p->G = 1;
  } else {
    if (group <= 0 || K % group) return GPTQ_ERR_SHAPE;
    p->group = group;
    p->G = K / group;
  }
  if (!aligned(qweight, 16) || !aligned(qzeros, 16) || !aligned(scales, 16)) return GPTQ_ERR_ALIGN;
  if (g_idx && !aligned(g_idx, 4)) return GPTQ_ERR_ALIGN;
  p->qweight = qweight;
  p->qzeros = qzeros;
  p->scales = scales;
  p->g_idx = g_idx;
  p->K = K;
  p->N = N;
  p->bits = bits;
  return GPTQ_OK;
}

int device_ready(Problem* p) {
  cudaError_t err;
  DeviceState* st = current_state(&err);
  if (!st) return GPTQ_ERR_CUDA;
  if (st->info.cc_major != 10 || st->info.cc_minor != 3) return GPTQ_ERR_UNSUPPORTED;
  p->status = st->status;
  return GPTQ_OK;
}

int from_cuda(cudaError_t e) { return e == cudaSuccess ? GPTQ_OK : GPTQ_ERR_CUDA; }

// decode-only paths: a layout that fits no CTA (nothing was launched) is a shape the call refuses
int from_decode(cudaError_t e) { return e == cudaErrorInvalidConfiguration ? GPTQ_ERR_SHAPE : from_cuda(e); }

}  // namespace

bool encode_tensor_map(void* tmap, int dtype, void* base, const uint64_t* dims,
                       const uint64_t* strides, const uint32_t* box, const uint32_t* estr,
                       int swizzle) {
  static PFN_cuTensorMapEncodeTiled_v12000 fn = nullptr;
  static std::once_flag once;
  std::call_once(once, []() {
    void* p = nullptr;
    cudaDriverEntryPointQueryResult q;
    if (cudaGetDriverEntryPointByVersion("cuTensorMapEncodeTiled", &p, 12000, cudaEnableDefault,
                                         &q) == cudaSuccess &&
        q == cudaDriverEntryPointSuccess)
      fn = reinterpret_cast<PFN_cuTensorMapEncodeTiled_v12000>(p);
  });
  if (!fn) return false;
  return fn(static_cast<CUtensorMap*>(tmap), static_cast<CUtensorMapDataType>(dtype), 2, base,
            reinterpret_cast<const cuuint64_t*>(dims), reinterpret_cast<const cuuint64_t*>(strides),
            box, estr, CU_TENSOR_MAP_INTERLEAVE_NONE, static_cast<CUtensorMapSwizzle>(swizzle),
            CU_TENSOR_MAP_L2_PROMOTION_L2_256B, CU_TENSOR_MAP_FLOAT_OOB_FILL_NONE) == CUDA_SUCCESS;
}

const DeviceInfo& device_info() {
  cudaError_t err;
  DeviceState* st = current_state(&err);
  static DeviceInfo fallback{0, 1, 0, 0, 48 * 1024};
  return st ? st->info : fallback;
}

}  // namespace gptq

using gptq::Problem;

extern "C" int gptq_dequant(const int32_t* qweight, const int32_t* qzeros, const void* scales,
                            const int32_t* g_idx, int K, int N, int bits, int group, int fmt,
                            int out_dtype, void* W_out, void* stream) {
  Problem p = {};
  int rc = gptq::check_common(qweight, qzeros, scales, g_idx, K, N, bits, group, &p);
  if (rc) return rc;
  if (fmt != GPTQ_FMT_V1 && fmt != GPTQ_FMT_V2) return GPTQ_ERR_ARG;
  if (out_dtype != GPTQ_F16 && out_dtype != GPTQ_BF16) return GPTQ_ERR_ARG;
  if (!W_out) return GPTQ_ERR_ARG;
  if (!gptq::aligned(W_out, 16)) return GPTQ_ERR_ALIGN;
  rc = gptq::device_ready(&p);
  if (rc) return rc;
  p.dtype = out_dtype;
  p.zero_offset = fmt == GPTQ_FMT_V1 ? 1 : 0;
  p.out = W_out;
  return gptq::from_cuda(gptq::launch_dequant(p, static_cast<cudaStream_t>(stream)));
}

extern "C" size_t gptq_gemm_workspace_size(int M, int K, int N, int bits, int group) {
  (void)N; (void)bits; (void)group;
  return gptq::prefill_workspace_bytes(M, K);
}

namespace gptq {
namespace {

// Workspace of the act-order path of gptq_gemm: [flag | perm (K) | code sources (K) | sorted
// qweight | the tensor-core kernel's workspace for M x K (also the decode kernels' gathered
// activations)], each part starting on a 256-byte boundary.
struct ActOrderLayout {
  size_t perm, src, qweight, rest, total;
};

ActOrderLayout act_order_layout(int M, int K, int N, int bits) {
  auto up = [](size_t x) { return (x + 255) & ~static_cast<size_t>(255); };
  ActOrderLayout l;
  l.perm = 256;
  l.src = l.perm + up(static_cast<size_t>(K) * 4);
  l.qweight = l.src + up(static_cast<size_t>(K) * 4);
  l.rest = l.qweight + up(static_cast<size_t>(K) * bits / 32 * N * 4);
  l.total = l.rest + prefill_workspace_bytes(M > 0 ? M : 1, K);
  return l;
}

// Shapes whose rows the device sorts: the sort and repack fit their shared memory, and the sorted
// groups suit the group-wise (exact-difference) kernels: groups of whole k-tiles.
bool act_order_shape_ok(int K, int G, int group, int bits) {
  const int per = bits == 3 ? 32 : 32 / bits;
  return sort_groups_fits(K, G, group) && repack_strip_width(K, bits) > 0 && group % (4 * per) == 0;
}

// gptq_gemm with g_idx through sorted rows.  Launches, in stream order: the sort (perm, flag), the
// repack (flag 1 only), the group-wise GEMM on the sorted weight with A gathered through perm
// (flag 1 only), and the per-row-group GEMM on the original checkpoint (flag 0 only: g_idx with an
// entry out of range, or groups of unequal size).  The repack and the group-wise GEMM start only
// after their predecessor has completed (no programmatic dependent launch): they read what it
// wrote.  The per-row decode reads nothing the group-wise GEMM writes, and the flag is final once
// that GEMM has started (the sort had completed before the repack finished), so it is a
// programmatic dependent: with flag 1 its CTAs leave as slots free at the group-wise GEMM's tail
// instead of costing a launch after it.
int gemm_act_order(const Problem& p, cudaStream_t s) {
  const ActOrderLayout l = act_order_layout(p.M, p.K, p.N, p.bits);
  unsigned char* ws = static_cast<unsigned char*>(p.workspace);
  int* flag = reinterpret_cast<int*>(ws);
  int32_t* perm = reinterpret_cast<int32_t*>(ws + l.perm);
  uint32_t* src = reinterpret_cast<uint32_t*>(ws + l.src);
  int32_t* qw_sorted = reinterpret_cast<int32_t*>(ws + l.qweight);
  void* rest = ws + l.rest;
  const size_t rest_bytes = l.total - l.rest;
  cudaError_t e = launch_sort_groups(p.g_idx, p.K, p.G, p.group, p.bits, perm, src, flag, s);
  if (e != cudaSuccess) return from_cuda(e);
  e = launch_repack_rows(p.qweight, src, flag, p.K, p.N, p.bits, qw_sorted, nullptr, s);
  if (e != cudaSuccess) return from_cuda(e);

  Problem q = p;
  q.g_idx = nullptr;
  q.qweight = qw_sorted;
  q.run_flag = flag;
  q.run_when = 1;
  q.no_pdl = true;
  q.workspace = rest;
  q.workspace_bytes = rest_bytes;
  bool fast_done = false;
  if (p.M <= kDecodeMaxM) {
    Problem d = q;
    if (p.M > 1) {
      e = launch_gather_cols(p.A, perm, p.M, p.K, rest, s);
      if (e != cudaSuccess) return from_cuda(e);
      d.A = rest;
    } else {
      d.perm = perm;                            // one token: gathered while staging
    }
    e = launch_decode(d, s);
    if (e == cudaSuccess) fast_done = true;
    else if (e != cudaErrorInvalidConfiguration) return from_cuda(e);
  }
  if (!fast_done) {
    q.perm = perm;                              // the tensor-core kernel gathers A into `rest`
    e = launch_prefill(q, s);
    if (e != cudaSuccess) return from_cuda(e);
  }

  Problem f = p;
  f.run_flag = flag;
  f.run_when = 0;
  f.no_pdl = true;
  f.workspace = rest;
  f.workspace_bytes = rest_bytes;
  if (p.M <= kDecodeMaxM) {
    Problem fd = f;
    fd.no_pdl = false;
    e = launch_decode(fd, s);
    if (e != cudaErrorInvalidConfiguration) return from_cuda(e);
  }
  return from_cuda(launch_prefill(f, s));
}

}  // namespace
}  // namespace gptq

extern "C" size_t gptq_gemm_act_order_workspace_size(int M, int K, int N, int bits, int group) {
  if (M <= 0 || K <= 0 || N <= 0 || group <= 0 || K % group || !gptq::bits_ok(bits)) return 0;
  if (!gptq::act_order_shape_ok(K, K / group, group, bits)) return 0;
  return gptq::act_order_layout(M, K, N, bits).total;
}

namespace gptq {
namespace {

// gptq_gemm's argument validation: fills *p on success (p->M == 0: nothing to do).
int gemm_prepare(const void* A, int M, int K, int a_dtype, const int32_t* qweight, const int32_t* qzeros,
                 const void* scales, const int32_t* g_idx, int N, int bits, int group, int fmt, void* C,
                 void* workspace, size_t workspace_bytes, Problem* p) {
  *p = Problem{};
  int rc = check_common(qweight, qzeros, scales, g_idx, K, N, bits, group, p);
  if (rc) return rc;
  if (fmt != GPTQ_FMT_V1 && fmt != GPTQ_FMT_V2) return GPTQ_ERR_ARG;
  if (a_dtype != GPTQ_F16 && a_dtype != GPTQ_BF16) return GPTQ_ERR_ARG;
  if (M < 0) return GPTQ_ERR_SHAPE;
  if (M == 0) return GPTQ_OK;
  if (!A || !C) return GPTQ_ERR_ARG;
  if (!aligned(A, 16) || !aligned(C, 16)) return GPTQ_ERR_ALIGN;
  if (workspace && !aligned(workspace, 16)) return GPTQ_ERR_ALIGN;
  rc = device_ready(p);
  if (rc) return rc;
  p->A = A;
  p->M = M;
  p->dtype = a_dtype;
  p->zero_offset = fmt == GPTQ_FMT_V1 ? 1 : 0;
  p->out = C;
  p->workspace = workspace;
  p->workspace_bytes = workspace ? workspace_bytes : 0;
  return GPTQ_OK;
}

// gptq_gemm's routing of a validated problem.  decode_only: run only when the decode kernels take
// the problem (M <= 32, no g_idx, K within their reach); *declined is then set, with nothing
// launched, for a problem they do not take.
int gemm_run(const Problem& p, cudaStream_t s, bool decode_only, bool* declined) {
  if (decode_only) {
    cudaError_t e = cudaErrorInvalidConfiguration;
    if (p.M <= kDecodeMaxM && p.g_idx == nullptr) e = launch_decode(p, s);
    if (e == cudaErrorInvalidConfiguration) {
      *declined = true;
      return GPTQ_OK;
    }
    return from_cuda(e);
  }
  // act-order with room for the sorted copy: sort the rows on the device, then the group-wise
  // kernels (gptq_gemm_act_order_workspace_size is 0 for shapes that do not qualify)
  if (p.g_idx) {
    const size_t need = gptq_gemm_act_order_workspace_size(p.M, p.K, p.N, p.bits, p.group);
    if (need && p.workspace_bytes >= need) return gemm_act_order(p, s);
  }
  if (p.M <= kDecodeMaxM) {
    const cudaError_t e = launch_decode(p, s);
    // cudaErrorInvalidConfiguration: nothing launched, the decode layout does not fit this K at
    // this M even split 16 ways; the tensor-core kernel takes the problem (any M)
    if (e != cudaErrorInvalidConfiguration) return from_cuda(e);
  }
  // the tensor-core kernel multiplies bf16 activations as an fp16 copy in the workspace
  if (p.dtype == GPTQ_BF16 && p.workspace_bytes < prefill_workspace_bytes(p.M, p.K)) return GPTQ_ERR_WORKSPACE;
  return from_cuda(launch_prefill(p, s));
}

// The activations copied in by a kernel that reads page-locked host memory directly: it lets its
// dependents launch at once, so a decode kernel that follows with programmatic dependent launch
// streams its weights while A is still arriving, and reads A after its dependency wait.  n16:
// 16-byte pieces (M * K * 2 is a multiple of 64).
__global__ void __launch_bounds__(256) k_copy_in(const uint4* __restrict__ src, uint4* __restrict__ dst,
                                                 long long n16) {
  asm volatile("griddepcontrol.launch_dependents;" ::: "memory");
  const long long step = static_cast<long long>(gridDim.x) * blockDim.x;
  for (long long i = static_cast<long long>(blockIdx.x) * blockDim.x + threadIdx.x; i < n16; i += step)
    dst[i] = src[i];
}

// Page-locked host memory the device reaches at the same address (unified addressing).
bool device_mapped_host(const void* ptr) {
  cudaPointerAttributes at;
  if (cudaPointerGetAttributes(&at, ptr) != cudaSuccess) {
    cudaGetLastError();                        // an unknown pointer is not an error here
    return false;
  }
  return at.type == cudaMemoryTypeHost && at.devicePointer == ptr;
}

}  // namespace
}  // namespace gptq

extern "C" int gptq_gemm(const void* A, int M, int K, int a_dtype, const int32_t* qweight,
                         const int32_t* qzeros, const void* scales, const int32_t* g_idx, int N,
                         int bits, int group, int fmt, void* C, void* workspace,
                         size_t workspace_bytes, void* stream) {
  gptq::Problem p;
  const int rc = gptq::gemm_prepare(A, M, K, a_dtype, qweight, qzeros, scales, g_idx, N, bits, group, fmt, C,
                                    workspace, workspace_bytes, &p);
  if (rc != GPTQ_OK || p.M == 0) return rc;
  return gptq::gemm_run(p, static_cast<cudaStream_t>(stream), false, nullptr);
}

namespace gptq {
namespace {

// Where gptq_gemm_host moves A and C: page-locked host memory that the device reaches at the
// same address is read and written by kernels, anything else goes through DMA copies.  A takes
// the copy kernel only up to 32 KB: measured on llama-7B's [4096, 11008] (µs per call, direct
// call / captured plan), the kernel gave 20.8 / 16.9 at M = 1 and 24.0 / 20.3 at M = 4, but
// 31.8 / 41.5 at M = 16, where a DMA copy gives 32.5 / 30.5.
struct HostRoute {
  bool a_kernel;   // A copied in by k_copy_in
  bool c_direct;   // the decode kernels may write C straight into C_host
};

constexpr size_t kCopyKernelMaxBytes = 32 * 1024;

HostRoute host_route(const void* A_host, size_t a_bytes, const void* C_host) {
  return HostRoute{a_bytes <= kCopyKernelMaxBytes && aligned(A_host, 16) && device_mapped_host(A_host),
                   aligned(C_host, 16) && device_mapped_host(C_host)};
}

// gptq_gemm_host's stream work for a validated problem, without the final wait: A in, the GEMM,
// C out.  On an error the caller drains the stream before returning it.
int host_enqueue(const Problem& p, const HostRoute& r, const void* A_host, void* A_dev, void* C_dev, void* C_host,
                 cudaStream_t s) {
  const size_t a_bytes = static_cast<size_t>(p.M) * p.K * 2;
  if (r.a_kernel) {
    const long long n16 = static_cast<long long>(a_bytes / 16);
    long long blocks = (n16 + 255) / 256;
    if (blocks > 64) blocks = 64;
    k_copy_in<<<static_cast<unsigned>(blocks), 256, 0, s>>>(static_cast<const uint4*>(A_host),
                                                            static_cast<uint4*>(A_dev), n16);
    if (cudaGetLastError() != cudaSuccess) return GPTQ_ERR_CUDA;
  } else if (cudaMemcpyAsync(A_dev, A_host, a_bytes, cudaMemcpyHostToDevice, s) != cudaSuccess) {
    return GPTQ_ERR_CUDA;
  }
  // The decode kernels write C with plain stores: into page-locked host memory that the device
  // reaches directly, they write the result in place of a device buffer and a copy back.
  if (r.c_direct) {
    Problem d = p;
    d.out = C_host;
    bool declined = false;
    const int rc = gemm_run(d, s, true, &declined);
    if (rc != GPTQ_OK || !declined) return rc;
  }
  const int rc = gemm_run(p, s, false, nullptr);
  if (rc != GPTQ_OK) return rc;
  if (cudaMemcpyAsync(C_host, C_dev, static_cast<size_t>(p.M) * p.N * 2, cudaMemcpyDeviceToHost, s) != cudaSuccess)
    return GPTQ_ERR_CUDA;
  return GPTQ_OK;
}

}  // namespace
}  // namespace gptq

extern "C" int gptq_gemm_host(const void* A_host, void* A_dev, int M, int K, int a_dtype,
                              const int32_t* qweight, const int32_t* qzeros, const void* scales,
                              const int32_t* g_idx, int N, int bits, int group, int fmt, void* C_dev,
                              void* C_host, void* workspace, size_t workspace_bytes, void* stream) {
  if (M < 0 || K <= 0 || N <= 0) return GPTQ_ERR_SHAPE;
  if (M == 0) return GPTQ_OK;
  if (!A_host || !A_dev || !C_dev || !C_host) return GPTQ_ERR_ARG;
  gptq::Problem p;
  int rc = gptq::gemm_prepare(A_dev, M, K, a_dtype, qweight, qzeros, scales, g_idx, N, bits, group, fmt, C_dev,
                              workspace, workspace_bytes, &p);
  if (rc != GPTQ_OK) return rc;                // arguments are checked before anything is copied
  cudaStream_t s = static_cast<cudaStream_t>(stream);
  rc = gptq::host_enqueue(p, gptq::host_route(A_host, static_cast<size_t>(M) * K * 2, C_host), A_host, A_dev, C_dev, C_host, s);
  if (rc != GPTQ_OK) {
    cudaStreamSynchronize(s);                  // the copy of A has finished before the caller reuses it
    return rc;
  }
  return cudaStreamSynchronize(s) == cudaSuccess ? GPTQ_OK : GPTQ_ERR_CUDA;
}

// A prepared gptq_gemm_host: the stream work of one call captured into a CUDA graph.
struct gptq_host_plan {
  cudaGraphExec_t exec;
  cudaStream_t stream;
};

extern "C" int gptq_host_plan_create(gptq_host_plan** plan, const void* A_host, void* A_dev, int M, int K,
                                     int a_dtype, const int32_t* qweight, const int32_t* qzeros,
                                     const void* scales, const int32_t* g_idx, int N, int bits, int group,
                                     int fmt, void* C_dev, void* C_host, void* workspace,
                                     size_t workspace_bytes, void* stream) {
  if (!plan) return GPTQ_ERR_ARG;
  *plan = nullptr;
  if (!stream) return GPTQ_ERR_ARG;            // the legacy default stream cannot be captured
  // one call first: it checks the problem end to end and does every one-time setup (launch
  // attributes, occupancy queries) outside the capture
  int rc = gptq_gemm_host(A_host, A_dev, M, K, a_dtype, qweight, qzeros, scales, g_idx, N, bits, group, fmt, C_dev,
                          C_host, workspace, workspace_bytes, stream);
  if (rc != GPTQ_OK) return rc;
  gptq_host_plan* h = new gptq_host_plan{nullptr, static_cast<cudaStream_t>(stream)};
  if (M == 0) {
    *plan = h;
    return GPTQ_OK;
  }
  gptq::Problem p;
  rc = gptq::gemm_prepare(A_dev, M, K, a_dtype, qweight, qzeros, scales, g_idx, N, bits, group, fmt, C_dev,
                          workspace, workspace_bytes, &p);
  const gptq::HostRoute route = gptq::host_route(A_host, static_cast<size_t>(M) * K * 2, C_host);
  cudaGraph_t graph = nullptr;
  if (rc == GPTQ_OK && cudaStreamBeginCapture(h->stream, cudaStreamCaptureModeThreadLocal) != cudaSuccess)
    rc = GPTQ_ERR_CUDA;
  if (rc == GPTQ_OK) {
    rc = gptq::host_enqueue(p, route, A_host, A_dev, C_dev, C_host, h->stream);
    if (cudaStreamEndCapture(h->stream, &graph) != cudaSuccess && rc == GPTQ_OK) rc = GPTQ_ERR_CUDA;
  }
  if (rc == GPTQ_OK && cudaGraphInstantiate(&h->exec, graph, 0) != cudaSuccess) rc = GPTQ_ERR_CUDA;
  if (graph) cudaGraphDestroy(graph);
  if (rc != GPTQ_OK) {
    cudaGetLastError();
    delete h;
    return rc;
  }
  *plan = h;
  return GPTQ_OK;
}

extern "C" int gptq_host_plan_run(gptq_host_plan* plan) {
  if (!plan) return GPTQ_ERR_ARG;
  if (!plan->exec) return GPTQ_OK;             // M == 0
  if (cudaGraphLaunch(plan->exec, plan->stream) != cudaSuccess) return GPTQ_ERR_CUDA;
  return cudaStreamSynchronize(plan->stream) == cudaSuccess ? GPTQ_OK : GPTQ_ERR_CUDA;
}

extern "C" int gptq_host_plan_destroy(gptq_host_plan* plan) {
  if (!plan) return GPTQ_OK;
  if (plan->exec) cudaGraphExecDestroy(plan->exec);
  delete plan;
  return GPTQ_OK;
}

extern "C" int gptq_gemm_grouped(const void* A, int rows, int K, int a_dtype, const int32_t* offsets,
                                 int E, int max_m, const int32_t* qweight, const int32_t* qzeros,
                                 const void* scales, int N, int bits, int group, int fmt, void* C,
                                 void* stream) {
  Problem p = {};
  int rc = gptq::check_common(qweight, qzeros, scales, nullptr, K, N, bits, group, &p);
  if (rc) return rc;
  if (fmt != GPTQ_FMT_V1 && fmt != GPTQ_FMT_V2) return GPTQ_ERR_ARG;
  if (a_dtype != GPTQ_F16 && a_dtype != GPTQ_BF16) return GPTQ_ERR_ARG;
  if (rows < 0 || E < 0 || E > 65535 || max_m < 1 || max_m > gptq::kDecodeMaxM) return GPTQ_ERR_SHAPE;
  // the stacked weight is one tensor map of E * K * bits / 32 rows (32-bit coordinates)
  if (static_cast<long long>(E) * K * bits / 32 > 0x7FFFFFFFLL) return GPTQ_ERR_SHAPE;
  if (rows == 0 || E == 0) return GPTQ_OK;
  if (!A || !C || !offsets) return GPTQ_ERR_ARG;
  if (!gptq::aligned(A, 16) || !gptq::aligned(C, 16) || !gptq::aligned(offsets, 4)) return GPTQ_ERR_ALIGN;
  rc = gptq::device_ready(&p);
  if (rc) return rc;
  p.A = A;
  p.M = max_m;
  p.dtype = a_dtype;
  p.zero_offset = fmt == GPTQ_FMT_V1 ? 1 : 0;
  p.out = C;
  p.offsets = offsets;
  p.E = E;
  p.rows = rows;
  return gptq::from_decode(gptq::launch_decode_grouped(p, static_cast<cudaStream_t>(stream)));
}

extern "C" size_t gptq_gemm_perm_workspace_size(int M, int K) {
  if (M <= 1 || K <= 0) return 0;
  return (static_cast<size_t>(M) * K * 2 + 255) & ~static_cast<size_t>(255);
}

extern "C" int gptq_gemm_perm(const void* A, int M, int K, int a_dtype, const int32_t* perm,
                              const int32_t* qweight, const int32_t* qzeros, const void* scales,
                              int N, int bits, int group, int fmt, void* C, void* workspace,
                              size_t workspace_bytes, void* stream) {
  Problem p = {};
  if (group == -1) return GPTQ_ERR_SHAPE;                 // act-order always has real groups
  int rc = gptq::check_common(qweight, qzeros, scales, nullptr, K, N, bits, group, &p);
  if (rc) return rc;
  if (fmt != GPTQ_FMT_V1 && fmt != GPTQ_FMT_V2) return GPTQ_ERR_ARG;
  if (a_dtype != GPTQ_F16 && a_dtype != GPTQ_BF16) return GPTQ_ERR_ARG;
  if (M < 0 || M > gptq::kDecodeMaxM) return GPTQ_ERR_SHAPE;
  const size_t ws = gptq_gemm_perm_workspace_size(M, K);
  if (workspace_bytes < ws) return GPTQ_ERR_WORKSPACE;
  if (M == 0) return GPTQ_OK;
  if (!A || !C || !perm || (ws && !workspace)) return GPTQ_ERR_ARG;
  if (!gptq::aligned(A, 16) || !gptq::aligned(C, 16) || !gptq::aligned(perm, 16)) return GPTQ_ERR_ALIGN;
  if (ws && !gptq::aligned(workspace, 16)) return GPTQ_ERR_ALIGN;
  rc = gptq::device_ready(&p);
  if (rc) return rc;
  cudaStream_t s = static_cast<cudaStream_t>(stream);
  p.M = M;
  p.dtype = a_dtype;
  p.zero_offset = fmt == GPTQ_FMT_V1 ? 1 : 0;
  p.out = C;
  if (ws) {
    // several tokens: gather A[:, perm] once into the workspace, then a plain decode GEMM
    cudaError_t e = gptq::launch_gather_cols(A, perm, M, K, workspace, s);
    if (e != cudaSuccess) return gptq::from_cuda(e);
    p.A = workspace;
    p.perm = nullptr;
  } else {
    // one token: each CTA gathers its own k range while staging (no workspace)
    p.A = A;
    p.perm = perm;
  }
  return gptq::from_decode(gptq::launch_decode(p, s));
}

// ---------------------------------------------------------------------------------------------
// Allocation-free variant of gptq_gemm_perm.  Its only scratch (the gathered activations
// A[:, perm] for M > 1) is this file-scope device array; its device address is looked up once
// per device, with that device current, and handed to the gather kernel.
namespace {

constexpr size_t kNoAllocScratchBytes = static_cast<size_t>(1) << 20;   // 1 MiB per device
static __device__ __align__(256) unsigned char g_noalloc_scratch[kNoAllocScratchBytes];

struct ScratchState {
  std::once_flag once;
  void* ptr = nullptr;
  cudaError_t err = cudaSuccess;
};
ScratchState g_noalloc_state[gptq::kMaxDevices];

// Device address of g_noalloc_scratch on the current device (set up on first use), or nullptr.
void* noalloc_scratch() {
  int dev = 0;
  if (cudaGetDevice(&dev) != cudaSuccess || dev < 0 || dev >= gptq::kMaxDevices) return nullptr;
  ScratchState& st = g_noalloc_state[dev];
  std::call_once(st.once, [&st]() {
    void* ptr = nullptr;
    st.err = cudaGetSymbolAddress(&ptr, g_noalloc_scratch);
    st.ptr = st.err == cudaSuccess ? ptr : nullptr;
  });
  return st.ptr;
}

}  // namespace

extern "C" int gptq_gemm_perm_noalloc(const void* A, int M, int K, int a_dtype, const int32_t* perm,
                                      const int32_t* qweight, const int32_t* qzeros,
                                      const void* scales, int N, int bits, int group, int fmt,
                                      void* C, void* stream) {
  Problem p = {};
  if (group == -1) return GPTQ_ERR_SHAPE;
  int rc = gptq::check_common(qweight, qzeros, scales, nullptr, K, N, bits, group, &p);
  if (rc) return rc;
  if (fmt != GPTQ_FMT_V1 && fmt != GPTQ_FMT_V2) return GPTQ_ERR_ARG;
  if (a_dtype != GPTQ_F16 && a_dtype != GPTQ_BF16) return GPTQ_ERR_ARG;
  if (M < 0 || M > gptq::kDecodeMaxM) return GPTQ_ERR_SHAPE;
  const size_t need = gptq_gemm_perm_workspace_size(M, K);
  if (need > kNoAllocScratchBytes) return GPTQ_ERR_WORKSPACE;   // beyond the built-in scratch
  if (M == 0) return GPTQ_OK;
  if (!A || !C || !perm) return GPTQ_ERR_ARG;
  if (!gptq::aligned(A, 16) || !gptq::aligned(C, 16) || !gptq::aligned(perm, 16)) return GPTQ_ERR_ALIGN;
  rc = gptq::device_ready(&p);
  if (rc) return rc;
  cudaStream_t s = static_cast<cudaStream_t>(stream);
  p.M = M;
  p.dtype = a_dtype;
  p.zero_offset = fmt == GPTQ_FMT_V1 ? 1 : 0;
  p.out = C;
  if (need) {
    void* scratch = noalloc_scratch();
    if (!scratch) return GPTQ_ERR_CUDA;
    cudaError_t e = gptq::launch_gather_cols(A, perm, M, K, scratch, s);
    if (e != cudaSuccess) return gptq::from_cuda(e);
    p.A = scratch;
    p.perm = nullptr;
  } else {
    p.A = A;
    p.perm = perm;
  }
  return gptq::from_decode(gptq::launch_decode(p, s));
}

extern "C" int gptq_prepack_interleave(const int32_t* qweight, int K, int N, int bits, int32_t* qweight_il) {
  if (!gptq::bits_ok(bits) || !qweight || !qweight_il) return GPTQ_ERR_ARG;
  const int per = bits == 3 ? 32 : 32 / bits, rows = bits == 3 ? 3 : 1;
  if (K <= 0 || N <= 0 || N % 32 || K % (4 * per)) return GPTQ_ERR_SHAPE;
  const int tiles = K / per / 4, blocks = N / 32;
  // word ((((cb * tiles + kt) * rows + r) * 32 + lane) * 4 + c) holds row (4 kt + t) * rows + r and
  // column 32 cb + 4 quad(g) + c of the checkpoint, for lane = 4 g + t: the 16 bytes that lane of
  // the decode kernel's warp loads for unit t of k-tile kt, columns quad(g) of its 32-column block
  std::vector<int32_t> out(static_cast<size_t>(K / per) * rows * N);
  size_t i = 0;
  for (int cb = 0; cb < blocks; ++cb)
    for (int kt = 0; kt < tiles; ++kt)
      for (int r = 0; r < rows; ++r)
        for (int lane = 0; lane < 32; ++lane) {
          const int g = lane >> 2, t = lane & 3;
          const int quad = ((g & 1) << 2) | (g >> 1);
          const size_t src = (static_cast<size_t>(kt * 4 + t) * rows + r) * N + cb * 32 + quad * 4;
          for (int c = 0; c < 4; ++c) out[i++] = qweight[src + c];
        }
  for (size_t j = 0; j < out.size(); ++j) qweight_il[j] = out[j];
  return GPTQ_OK;
}

extern "C" int gptq_gemm_interleaved(const void* A, int M, int K, int a_dtype, const int32_t* perm,
                                     const int32_t* qweight_il, const int32_t* qzeros, const void* scales, int N,
                                     int bits, int group, int fmt, void* C, void* workspace,
                                     size_t workspace_bytes, void* stream) {
  Problem p = {};
  int rc = gptq::check_common(qweight_il, qzeros, scales, nullptr, K, N, bits, group, &p);
  if (rc) return rc;
  if (fmt != GPTQ_FMT_V1 && fmt != GPTQ_FMT_V2) return GPTQ_ERR_ARG;
  if (a_dtype != GPTQ_F16 && a_dtype != GPTQ_BF16) return GPTQ_ERR_ARG;
  const int per = bits == 3 ? 32 : 32 / bits;
  // whole k-tiles of 4 units, and groups made of whole k-tiles (the scale folds per group)
  if (K % (4 * per) || p.group % (4 * per)) return GPTQ_ERR_SHAPE;
  if (M < 0 || M > gptq::kDecodeMaxM) return GPTQ_ERR_SHAPE;
  const size_t ws = perm ? gptq_gemm_perm_workspace_size(M, K) : 0;
  if (workspace_bytes < ws) return GPTQ_ERR_WORKSPACE;
  if (M == 0) return GPTQ_OK;
  if (!A || !C || (ws && !workspace)) return GPTQ_ERR_ARG;
  if (!gptq::aligned(A, 16) || !gptq::aligned(C, 16) || (perm && !gptq::aligned(perm, 16))) return GPTQ_ERR_ALIGN;
  if (ws && !gptq::aligned(workspace, 16)) return GPTQ_ERR_ALIGN;
  rc = gptq::device_ready(&p);
  if (rc) return rc;
  cudaStream_t s = static_cast<cudaStream_t>(stream);
  p.M = M;
  p.dtype = a_dtype;
  p.zero_offset = fmt == GPTQ_FMT_V1 ? 1 : 0;
  p.out = C;
  p.interleaved = true;
  p.A = A;
  p.perm = perm;
  if (ws) {
    cudaError_t e = gptq::launch_gather_cols(A, perm, M, K, workspace, s);
    if (e != cudaSuccess) return gptq::from_cuda(e);
    p.A = workspace;
    p.perm = nullptr;
  }
  return gptq::from_decode(gptq::launch_decode(p, s));
}

extern "C" int gptq_prepack_act_order(const int32_t* qweight, const int32_t* g_idx, int K, int N,
                                      int bits, int group, int32_t* qweight_out, int32_t* perm) {
  if (!gptq::bits_ok(bits) || !qweight || !g_idx || !qweight_out || !perm) return GPTQ_ERR_ARG;
  if (K <= 0 || N <= 0 || K % 32 || N % 32 || group <= 0 || K % group) return GPTQ_ERR_SHAPE;
  const int G = K / group;
  // stable counting sort of the rows by group; every group must hold exactly `group` rows
  std::vector<int> next(G, 0);
  for (int k = 0; k < K; ++k) {
    const int g = g_idx[k];
    if (g < 0 || g >= G) return GPTQ_ERR_SHAPE;
    if (++next[g] > group) return GPTQ_ERR_SHAPE;
  }
  for (int g = 0; g < G; ++g) next[g] = g * group;
  std::vector<int32_t> order(K);
  for (int k = 0; k < K; ++k) order[next[g_idx[k]]++] = k;
  // rewrite every column's LSB-first code stream in the new row order
  const int rows = K * bits / 32;
  const uint32_t mask = (1u << bits) - 1u;
  const uint32_t* in = reinterpret_cast<const uint32_t*>(qweight);
  std::vector<uint32_t> out(static_cast<size_t>(rows) * N, 0u);
  for (int n = 0; n < N; ++n) {
    auto code = [&](int k) {
      const int bit = bits * k, w = bit >> 5, sh = bit & 31;
      uint64_t v = in[static_cast<size_t>(w) * N + n];
      if (sh + bits > 32) v |= static_cast<uint64_t>(in[static_cast<size_t>(w + 1) * N + n]) << 32;
      return static_cast<uint32_t>(v >> sh) & mask;
    };
    for (int k = 0; k < K; ++k) {
      const uint64_t v = static_cast<uint64_t>(code(order[k])) << ((bits * k) & 31);
      const int w = (bits * k) >> 5;
      out[static_cast<size_t>(w) * N + n] |= static_cast<uint32_t>(v);
      if (((bits * k) & 31) + bits > 32) out[static_cast<size_t>(w + 1) * N + n] |= static_cast<uint32_t>(v >> 32);
    }
  }
  for (size_t i = 0; i < out.size(); ++i) qweight_out[i] = static_cast<int32_t>(out[i]);
  for (int k = 0; k < K; ++k) perm[k] = order[k];
  return GPTQ_OK;
}

// The device prepack's workspace: the sort's flag (256 bytes), then each sorted row's code
// position (K words, rounded up to 256 bytes).
extern "C" size_t gptq_prepack_act_order_device_workspace_size(int K, int bits, int group) {
  if (K <= 0 || K % 32 || group <= 0 || K % group || !gptq::bits_ok(bits)) return 0;
  if (!gptq::sort_groups_fits(K, K / group, group) || gptq::repack_strip_width(K, bits) == 0) return 0;
  return 256 + ((static_cast<size_t>(K) * 4 + 255) & ~static_cast<size_t>(255));
}

// gptq_prepack_act_order on the device: the same kernels gptq_gemm's act-order path runs per
// call (the stable sort, then the repack, which writes only when every group holds `group` rows
// and otherwise raises GPTQ_DEV_GIDX_GROUPS), then the ordering kernel, so that a GEMM issued
// right after may read qweight_out before its own dependency wait.
extern "C" int gptq_prepack_act_order_device(const int32_t* qweight, const int32_t* g_idx, int K, int N,
                                             int bits, int group, int32_t* qweight_out, int32_t* perm,
                                             void* workspace, size_t workspace_bytes, void* stream) {
  if (!gptq::bits_ok(bits) || !qweight || !g_idx || !qweight_out || !perm || !workspace) return GPTQ_ERR_ARG;
  if (K <= 0 || N <= 0 || K % 32 || N % 32 || group <= 0 || K % group) return GPTQ_ERR_SHAPE;
  const size_t need = gptq_prepack_act_order_device_workspace_size(K, bits, group);
  if (need == 0) return GPTQ_ERR_SHAPE;
  if (workspace_bytes < need) return GPTQ_ERR_WORKSPACE;
  if (!gptq::aligned(qweight, 16) || !gptq::aligned(qweight_out, 16) || !gptq::aligned(perm, 16) ||
      !gptq::aligned(workspace, 16) || !gptq::aligned(g_idx, 4))
    return GPTQ_ERR_ALIGN;
  const uintptr_t in0 = reinterpret_cast<uintptr_t>(qweight), out0 = reinterpret_cast<uintptr_t>(qweight_out);
  const uintptr_t bytes = static_cast<uintptr_t>(K) / 32 * bits * static_cast<uintptr_t>(N) * 4;
  if (in0 < out0 + bytes && out0 < in0 + bytes) return GPTQ_ERR_ARG;   // the copy must not overlap
  gptq::Problem p;
  const int rc = gptq::device_ready(&p);
  if (rc) return rc;
  cudaStream_t s = static_cast<cudaStream_t>(stream);
  unsigned char* ws = static_cast<unsigned char*>(workspace);
  int* flag = reinterpret_cast<int*>(ws);
  uint32_t* src = reinterpret_cast<uint32_t*>(ws + 256);
  cudaError_t e = gptq::launch_sort_groups(g_idx, K, K / group, group, bits, perm, src, flag, s);
  if (e == cudaSuccess) e = gptq::launch_repack_rows(qweight, src, flag, K, N, bits, qweight_out, p.status, s);
  if (e == cudaSuccess) e = gptq::launch_writer_fence(s);
  return gptq::from_cuda(e);
}

extern "C" int gptq_quantize_rtn(const float* W, int K, int N, int bits, int group,
                                 const int32_t* g_idx, int sym, int fmt, int32_t* qweight,
                                 int32_t* qzeros, void* scales, void* stream) {
  Problem p = {};
  int rc = gptq::check_common(qweight, qzeros, scales, g_idx, K, N, bits, group, &p);
  if (rc) return rc;
  if (!W) return GPTQ_ERR_ARG;
  if (fmt != GPTQ_FMT_V1 && fmt != GPTQ_FMT_V2) return GPTQ_ERR_ARG;
  if (sym != 0 && sym != 1) return GPTQ_ERR_ARG;
  if (!gptq::aligned(W, 16)) return GPTQ_ERR_ALIGN;
  rc = gptq::device_ready(&p);
  if (rc) return rc;
  gptq::QuantProblem q;
  q.W = W; q.K = K; q.N = N; q.bits = bits; q.group = p.group; q.G = p.G;
  q.g_idx = g_idx; q.sym = sym; q.fmt = fmt;
  q.qweight = qweight; q.qzeros = qzeros; q.scales = scales; q.status = p.status;
  return gptq::from_cuda(gptq::launch_quantize(q, static_cast<cudaStream_t>(stream)));
}

// Host repack: reads every field of a row's LSB-first stream, adds one, writes it back.
extern "C" int gptq_repack_zeros_v1_to_v2(const int32_t* qz_v1, int32_t* qz_v2, int G, int N,
                                          int bits) {
  if (!gptq::bits_ok(bits) || !qz_v1 || !qz_v2) return GPTQ_ERR_ARG;
  if (G <= 0 || N <= 0 || N % 32) return GPTQ_ERR_SHAPE;
  const int words = N * bits / 32;
  const uint32_t mask = (1u << bits) - 1u;
  std::vector<uint32_t> out(static_cast<size_t>(G) * words, 0u);
  for (int g = 0; g < G; ++g) {
    const uint32_t* in = reinterpret_cast<const uint32_t*>(qz_v1) + static_cast<size_t>(g) * words;
    uint32_t* o = out.data() + static_cast<size_t>(g) * words;
    for (int n = 0; n < N; ++n) {
      const int bit = bits * n, w = bit >> 5, s = bit & 31;
      uint64_t pair = in[w];
      if (s + bits > 32) pair |= static_cast<uint64_t>(in[w + 1]) << 32;
      const uint32_t f = static_cast<uint32_t>(pair >> s) & mask;
      if (f == mask) return GPTQ_ERR_ZERO_OVERFLOW;
      const uint64_t v = static_cast<uint64_t>(f + 1) << s;
      o[w] |= static_cast<uint32_t>(v);
      if (s + bits > 32) o[w + 1] |= static_cast<uint32_t>(v >> 32);
    }
  }
  for (size_t i = 0; i < out.size(); ++i) qz_v2[i] = static_cast<int32_t>(out[i]);
  return GPTQ_OK;
}

extern "C" int gptq_get_device_status(void* stream, unsigned int* out) {
  if (!out) return GPTQ_ERR_ARG;
  cudaError_t err;
  gptq::DeviceState* st = gptq::current_state(&err);
  if (!st) return GPTQ_ERR_CUDA;
  cudaStream_t s = static_cast<cudaStream_t>(stream);
  err = cudaStreamSynchronize(s);
  if (err == cudaSuccess) err = cudaMemcpy(out, st->status, sizeof(unsigned), cudaMemcpyDeviceToHost);
  if (err == cudaSuccess) err = cudaMemset(st->status, 0, sizeof(unsigned));
  if (err == cudaSuccess) err = cudaDeviceSynchronize();
  return gptq::from_cuda(err);
}

extern "C" int gptq_selftest_wait_timeout(unsigned long long limit_ns, int* waited_out, void* stream) {
  if (!waited_out || limit_ns == 0 || limit_ns > 10000000000ull) return GPTQ_ERR_ARG;
  if (!gptq::aligned(waited_out, 4)) return GPTQ_ERR_ALIGN;
  Problem p = {};
  int rc = gptq::device_ready(&p);
  if (rc) return rc;
  return gptq::from_cuda(gptq::launch_wait_selftest(p.status, limit_ns, waited_out,
                                                    static_cast<cudaStream_t>(stream)));
}

extern "C" const char* gptq_strerror(int code) {
  switch (code) {
    case GPTQ_OK: return "GPTQ_OK";
    case GPTQ_ERR_ARG: return "GPTQ_ERR_ARG: invalid argument (NULL pointer or bits/fmt/dtype/sym)";
    case GPTQ_ERR_SHAPE: return "GPTQ_ERR_SHAPE: unsupported shape (K, N multiples of 32; group divides K)";
    case GPTQ_ERR_ALIGN: return "GPTQ_ERR_ALIGN: pointer not 16-byte aligned";
    case GPTQ_ERR_WORKSPACE: return "GPTQ_ERR_WORKSPACE: workspace too small";
    case GPTQ_ERR_ZERO_OVERFLOW: return "GPTQ_ERR_ZERO_OVERFLOW: v1 zero of 2^bits-1 has no v2 encoding";
    case GPTQ_ERR_CUDA: return "GPTQ_ERR_CUDA: CUDA call or launch failed";
    case GPTQ_ERR_UNSUPPORTED: return "GPTQ_ERR_UNSUPPORTED: device is not sm_103 (GB300)";
    case GPTQ_ERR_DEVICE: return "GPTQ_ERR_DEVICE: device status word reported an error";
    default: return "unknown gptq status";
  }
}
