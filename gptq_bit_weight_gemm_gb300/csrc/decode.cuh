// decode.cuh -- shared pieces of the few-token (M <= 32) GPTQ GEMM: arguments, split-K
// ranges, scale/zero access, activation staging, cluster barriers, and the dispatch on
// (bits, token count, dtype).  The kernel itself is in decode_mma.cuh.
//
// This is the decode case of vLLM's gptq_gemm (page "增强 vLLM 对 GPTQv2 格式的支持：分析与实
// 现", section "调整细节：根据格式选择处理方式": zeros[i] + zero_offset, zero_offset =
// use_v2_format ? 0 : 1); the same page notes that the 2-bit GEMV case is slower than the
// GEMM case and lists "improve gptq_gemm decode speed" as follow-up work.  Every weight is read
// from HBM exactly once; the grid is (cluster of CS CTAs splitting K) x (slabs of 128 columns)
// (x experts, for the grouped mixture-of-experts GEMM of page "4.3 Weight-only INT4 量化：GPTQ、
// AWQ 与 Marlin Kernel", section 7),
// partial sums meet through distributed shared memory in a fixed order (deterministic, no
// workspace, no atomics), and launches use programmatic dependent launch so a kernel's prologue
// overlaps the previous kernel's tail.
#pragma once

#include <cooperative_groups.h>

#include "gptq_device.cuh"
#include "gptq_internal.h"

namespace gptq {
namespace decode {

namespace cg = cooperative_groups;

constexpr int kWarps = 4;
constexpr int kThreads = kWarps * 32;
constexpr int kSlab = 128;    // columns per CTA (4 per lane)

struct Args {
  const void* A;
  int M, K, N;
  const int32_t* qweight;
  const int32_t* qzeros;
  const __half* scales;
  const int32_t* g_idx;
  const int32_t* perm;       // nullable: activation column of each (prepacked) weight row
  int group, G, zero_offset, zwords, units;
  void* C;
  unsigned* status;
  // grouped (one weight per expert): rows [offsets[e], offsets[e + 1]) of A and C belong to
  // expert e of `experts`; `rows` bounds them.  The grid has min(experts, rows) expert slots
  // (blockIdx.z): slot z takes the z-th expert that holds rows.  nullptr for a single weight.
  const int32_t* offsets;
  int rows;
  int experts;
  // interleaved weights (gptq_prepack_interleave): k-tiles per 32-column block, else 0 (the
  // checkpoint's own row-major layout, read through the tensor map)
  int il_tiles;
  // nullable: the kernel does nothing unless *run_flag == run_when (set by a kernel that completed
  // before the kernel ahead of this launch started, so the flag is final at entry, PDL or not)
  const int* run_flag;
  int run_when;
};

__device__ __forceinline__ void split(int total, int parts, int idx, int& b, int& e) {
  b = static_cast<int>(static_cast<long long>(total) * idx / parts);
  e = static_cast<int>(static_cast<long long>(total) * (idx + 1) / parts);
}

// Scales (as fp32) and runtime zeros of columns n0..n0+3 for group g.
template <int BITS>
__device__ __forceinline__ void load_sz(const Args& a, int g, int n0, float (&s)[4],
                                        int (&z)[4]) {
  const uint2 sv = __ldg(reinterpret_cast<const uint2*>(a.scales + static_cast<long long>(g) * a.N + n0));
  s[0] = __half2float(__ushort_as_half(static_cast<uint16_t>(sv.x & 0xFFFFu)));
  s[1] = __half2float(__ushort_as_half(static_cast<uint16_t>(sv.x >> 16)));
  s[2] = __half2float(__ushort_as_half(static_cast<uint16_t>(sv.y & 0xFFFFu)));
  s[3] = __half2float(__ushort_as_half(static_cast<uint16_t>(sv.y >> 16)));
  const uint32_t zf = zeros4<BITS>(a.qzeros + static_cast<long long>(g) * a.zwords, n0);
#pragma unroll
  for (int c = 0; c < 4; ++c)
    z[c] = static_cast<int>((zf >> (BITS * c)) & Pack<BITS>::kMask) + a.zero_offset;
}

__device__ __forceinline__ int checked_group(const Args& a, int k) {
  int g = __ldg(a.g_idx + k);
  if (g < 0 || g >= a.G) {
    atomicOr(a.status, kStatusGidxRange);
    g = g < 0 ? 0 : a.G - 1;
  }
  return g;
}

// Code j of column c within a loaded unit (ROWS x uint4, one word per column per row).
template <int BITS>
__device__ __forceinline__ uint32_t unit_code(const uint4 (&u)[Pack<BITS>::kRowsPerUnit], int c,
                                              int j) {
  if constexpr (BITS == 3) {
    const uint32_t w0 = (&u[0].x)[c], w1 = (&u[1].x)[c], w2 = (&u[2].x)[c];
    return code3(w0, w1, w2, j);
  } else {
    return ((&u[0].x)[c] >> (BITS * j)) & Pack<BITS>::kMask;
  }
}

__device__ __forceinline__ void pdl_launch_dependents() {
  asm volatile("griddepcontrol.launch_dependents;" ::: "memory");
}
__device__ __forceinline__ void pdl_wait() { asm volatile("griddepcontrol.wait;" ::: "memory"); }

__device__ __forceinline__ void prefetch_l2(const void* p) {
  asm volatile("prefetch.global.L2 [%0];" ::"l"(p));
}

__device__ __forceinline__ void cluster_arrive_relaxed() {
  asm volatile("barrier.cluster.arrive.relaxed.aligned;" ::: "memory");
}
__device__ __forceinline__ void cluster_wait() {
  asm volatile("barrier.cluster.wait.aligned;" ::: "memory");
}

// Stage activation pairs into shared memory.  Work item = (unit u, real token m < M): one
// thread reads the unit's PER consecutive activations of row m with 16-byte loads (8-byte for
// 8-bit units) and writes the NP pairs (lo_k(p), hi_k(p)) through `put(u, m, p, value)`.  A
// thread's loads for up to stage_batch(PER) items are all issued before any of them is used, so
// the staging costs one L2 round trip per batch.  (Batches of 8 units measured slower at 1 to 8
// tokens -- 8.3 -> 8.5 us at one token on llama-7B -- and no faster at 16.)  Rows m >= M and units
// past the last one are written as zero by the caller.
__host__ __device__ constexpr int stage_batch(int per) { return per >= 32 ? 2 : 4; }

template <int PER>
struct UnitVec {   // a unit's activations: PER 16-bit values
  static constexpr int kWords = PER / 2;
  uint32_t w[kWords];
  __device__ __forceinline__ void load(const uint16_t* p) {
    if constexpr (kWords >= 4) {
#pragma unroll
      for (int i = 0; i < kWords / 4; ++i) {
        const uint4 v = __ldg(reinterpret_cast<const uint4*>(p) + i);
        w[4 * i] = v.x; w[4 * i + 1] = v.y; w[4 * i + 2] = v.z; w[4 * i + 3] = v.w;
      }
    } else {
      const uint2 v = __ldg(reinterpret_cast<const uint2*>(p));
      w[0] = v.x; w[1] = v.y;
    }
  }
  // the same, gathered: value i is row[pk[i]] (prepacked act-order rows); an index outside
  // [0, K) is clamped so that a bad permutation cannot read outside the row
  __device__ __forceinline__ void load_perm(const uint16_t* row, const int32_t* pk, int K) {
    int idx[PER];
#pragma unroll
    for (int i = 0; i < PER / 4; ++i) {
      const int4 v = __ldg(reinterpret_cast<const int4*>(pk) + i);
      idx[4 * i] = v.x; idx[4 * i + 1] = v.y; idx[4 * i + 2] = v.z; idx[4 * i + 3] = v.w;
    }
#pragma unroll
    for (int i = 0; i < PER; ++i) idx[i] = idx[i] < 0 ? 0 : (idx[i] >= K ? K - 1 : idx[i]);
#pragma unroll
    for (int i = 0; i < kWords; ++i)
      w[i] = static_cast<uint32_t>(__ldg(row + idx[2 * i])) | (static_cast<uint32_t>(__ldg(row + idx[2 * i + 1])) << 16);
  }
  __device__ __forceinline__ uint32_t half(int k) const {
    return (w[k >> 1] >> (16 * (k & 1))) & 0xFFFFu;
  }
};

// tid / nthr: this thread's index among the nthr threads that stage.
template <int PER, int NP, class LoK, class HiK, class Put>
__device__ __forceinline__ void stage_pairs(const uint16_t* A, const int32_t* perm, int M, int K,
                                            int ufirst, int nunits, int units, LoK lo_k, HiK hi_k,
                                            Put put, int tid, int nthr) {
  const int items = nunits * M;
  constexpr int kStageBatch = stage_batch(PER);
  for (int base = 0; base < items; base += kStageBatch * nthr) {
    UnitVec<PER> v[kStageBatch];
#pragma unroll
    for (int j = 0; j < kStageBatch; ++j) {
      const int it = base + j * nthr + tid;
      const int uu = M == 1 ? it : it / M, m = it - uu * M;
      if (it < items && ufirst + uu < units) {
        if (perm)
          v[j].load_perm(A + static_cast<long long>(m) * K, perm + static_cast<long long>(ufirst + uu) * PER, K);
        else
          v[j].load(A + static_cast<long long>(m) * K + static_cast<long long>(ufirst + uu) * PER);
      }
    }
#pragma unroll
    for (int j = 0; j < kStageBatch; ++j) {
      const int it = base + j * nthr + tid;
      const int uu = M == 1 ? it : it / M, m = it - uu * M;
      if (it < items) {
        const bool live = ufirst + uu < units;
#pragma unroll
        for (int p = 0; p < NP; ++p)
          put(uu, m, p, live ? (v[j].half(lo_k(p)) | (v[j].half(hi_k(p)) << 16)) : 0u);
      }
    }
  }
}

// Cluster size: enough warps to fill the GPU (about 24 per SM), at least one k-tile per warp
// and CTA.  Up to 16 (a non-portable cluster size, opted into at launch) for narrow matrices;
// the launcher may halve it again to keep the grid within one wave.
inline int choose_cluster(const Problem& p, int per_unit) {
  const int slabs = (p.N + kSlab - 1) / kSlab;
  const int units = p.K / per_unit;
  const int target = device_info().sm_count * 24;
  // Grouped launches split K as for one expert and run the experts as extra waves: counting
  // every expert's slabs would shrink the split, and each CTA would then stage activations for a
  // K range so long that no room is left for weight buffers (measured 1.7x slower for 8 experts).
  int cs = 1;
  while (cs < 16 && slabs * cs * kWarps < target && units >= 4 * cs * kWarps) cs *= 2;
  return cs;
}

template <int BITS, int MT, int MX, typename T, bool FOLD, bool GROUPED>
cudaError_t launch_mma(const Problem& p, cudaStream_t stream);

// MT: token block bound (1, 8, 16, 32); MX: the exact token count when it is MT (0 = read at run
// time), so the common batch sizes run with every token loop sized at compile time.  GROUPED:
// one weight per expert (blockIdx.z), each with its own rows of A and C.
template <int BITS, int MT, int MX, typename T, bool GROUPED = false>
cudaError_t launch_mt(const Problem& p, cudaStream_t stream) {
  // the scale folds per group when groups align with k-tiles (4 units)
  const bool fold = p.g_idx == nullptr && (p.group % (4 * Pack<BITS>::kPerUnit)) == 0;
  if (fold) return launch_mma<BITS, MT, MX, T, true, GROUPED>(p, stream);
  return launch_mma<BITS, MT, MX, T, false, GROUPED>(p, stream);
}

// Whether 17..32 tokens run as two 16-token blocks side by side (each CTA with the 16-token
// kernel's registers and staging, the weights read twice) rather than one 32-token block.
// Measured (CUDA-graph replay): faster on small matrices (2-bit [4096, 4096]: M=32 17.3 -> 14.5 us,
// M=24 15.3 -> 14.4) and for 3-bit at exactly 32 tokens (act-order [5120, 13824] prepacked: 74.8 ->
// 55.6 us); slower on large 4-bit ones (llama-7B [4096, 11008] M=32: 30.2 -> 34.5 us) and for
// 3-bit at 20 tokens (44.3 -> 49.3 us).  Where the 32-token layout fits no CTA, the split is
// tried before giving up.
inline bool token_split_pays(const Problem& p) {
  return static_cast<long long>(p.K) * p.N <= (1ll << 24) || (p.bits == 3 && p.M == 32);
}

// Every M <= 32 runs the tensor-core decode kernel (token blocks of 8; one token has an
// instantiation of its own, where the token count is a compile-time constant): even at one token,
// handing the multiply-accumulate to the tensor core leaves the SM with only the unpack to issue.
template <int BITS, typename T>
cudaError_t launch_tokens(const Problem& p, cudaStream_t stream) {
  // 17..32 tokens as two 16-token blocks side by side (grid z), both reading the same weights
  auto split = [&]() {
    Problem q = p;
    q.tok_split = 2;
    return p.M == 32 ? launch_mt<BITS, 16, 16, T>(q, stream) : launch_mt<BITS, 16, 0, T>(q, stream);
  };
  if (p.M > 16 && token_split_pays(p)) return split();
  switch (p.M) {
    case 1: return launch_mt<BITS, 1, 1, T>(p, stream);
    case 8: return launch_mt<BITS, 8, 8, T>(p, stream);
    case 16: return launch_mt<BITS, 16, 16, T>(p, stream);
    default: break;
  }
  if (p.M <= 8) return launch_mt<BITS, 8, 0, T>(p, stream);
  if (p.M <= 16) return launch_mt<BITS, 16, 0, T>(p, stream);
  const cudaError_t e = p.M == 32 ? launch_mt<BITS, 32, 32, T>(p, stream) : launch_mt<BITS, 32, 0, T>(p, stream);
  return e == cudaErrorInvalidConfiguration ? split() : e;
}

template <int BITS>
cudaError_t launch_bits(const Problem& p, cudaStream_t stream) {
  if (p.dtype == 0) return launch_tokens<BITS, __half>(p, stream);
  return launch_tokens<BITS, __nv_bfloat16>(p, stream);
}

// Grouped: p.M is the bound on any expert's rows (the per-expert counts live on the device);
// one token keeps its compile-time instantiation, more take the run-time token count.
template <int BITS, typename T>
cudaError_t launch_grouped_tokens(const Problem& p, cudaStream_t stream) {
  if (p.M == 1) return launch_mt<BITS, 1, 1, T, true>(p, stream);
  if (p.M <= 8) return launch_mt<BITS, 8, 0, T, true>(p, stream);
  if (p.M <= 16) return launch_mt<BITS, 16, 0, T, true>(p, stream);
  return launch_mt<BITS, 32, 0, T, true>(p, stream);
}

template <int BITS>
cudaError_t launch_grouped_bits(const Problem& p, cudaStream_t stream) {
  if (p.dtype == 0) return launch_grouped_tokens<BITS, __half>(p, stream);
  return launch_grouped_tokens<BITS, __nv_bfloat16>(p, stream);
}

}  // namespace decode
}  // namespace gptq
