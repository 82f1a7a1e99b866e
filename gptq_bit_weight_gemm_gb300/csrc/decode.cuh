// decode.cuh -- memory-bound GPTQ GEMM for few tokens (M <= 32): C = A @ dequant(W).
//
// This is the decode case of vLLM's gptq_gemm (page "增强 vLLM 对 GPTQv2 格式的支持：分析与实
// 现", section "调整细节：根据格式选择处理方式": zeros[i] + zero_offset, zero_offset =
// use_v2_format ? 0 : 1); the same page notes that the 2-bit GEMV case is slower than the
// GEMM case and lists "improve gptq_gemm decode speed" as follow-up work.  Every weight is read
// from HBM exactly once, so the kernel is built to stream qweight at full bandwidth:
//
//  * grid = (cluster of CS CTAs along K) x (slabs of 128 columns), 4 warps per CTA.  Each lane
//    owns 4 adjacent columns, so one 16-byte load brings in one packed unit row for all of them
//    and a warp reads 512 contiguous bytes per row.  The CTAs of a cluster and the warps of a
//    CTA split the K units (split-K) into contiguous ranges; loads are double-buffered in
//    registers and the first ones are issued before the activations are staged.
//  * 16-bit path (M <= 4, fp16 any of 2/4/8 bits, bf16 2/4 bits, no act-order): q - zero is
//    built exactly as a pair of 16-bit floats (magic-number unpack, one sub/fma with a per-group
//    constant), multiplied by the activation pair and summed with one fp16x2/bf16x2 fma per pair;
//    the 16-bit partial sums are flushed into fp32 after every unit (bf16) or every 4 units
//    (fp16), and the scale is applied once per group: acc += scale * sum_k a_k (q_k - zero).
//  * fp32 path (M <= 4 with act-order, 3-bit or bf16 8-bit): w = (q - zero) * scale in fp32
//    (exact) and fp32 fmas.  4 < M <= 32 runs the tensor-core variant in decode_mma.cuh.
//  * partial sums are reduced across warps in shared memory and across the cluster through
//    distributed shared memory, in a fixed order (deterministic), then rounded once to the
//    output dtype.  No global workspace and no atomics.
//  * programmatic dependent launch: each CTA lets the next kernel in the stream start launching
//    at once, and waits (griddepcontrol.wait) for the previous kernel before touching global
//    memory, so launch latency overlaps the previous kernel's tail.
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
constexpr int kBatch = 4;     // units per load stage

struct Args {
  const void* A;
  int M, K, N;
  const int32_t* qweight;
  const int32_t* qzeros;
  const __half* scales;
  const int32_t* g_idx;
  int group, G, zero_offset, zwords, units;
  void* C;
  unsigned* status;
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
// thread's loads for up to kStageBatch items are all issued before any of them is used, so the
// staging costs about one L2 round trip, not one per item.  Rows m >= M and units past the last
// one are written as zero by the caller.
constexpr int kStageBatch = 4;

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
  __device__ __forceinline__ uint32_t half(int k) const {
    return (w[k >> 1] >> (16 * (k & 1))) & 0xFFFFu;
  }
};

template <int PER, int NP, class LoK, class HiK, class Put>
__device__ __forceinline__ void stage_pairs(const uint16_t* A, int M, int K, int ufirst, int nunits,
                                            int units, LoK lo_k, HiK hi_k, Put put) {
  const int items = nunits * M;
  for (int base = 0; base < items; base += kStageBatch * static_cast<int>(blockDim.x)) {
    UnitVec<PER> v[kStageBatch];
#pragma unroll
    for (int j = 0; j < kStageBatch; ++j) {
      const int it = base + j * static_cast<int>(blockDim.x) + static_cast<int>(threadIdx.x);
      const int uu = it / M, m = it - uu * M;
      if (it < items && ufirst + uu < units)
        v[j].load(A + static_cast<long long>(m) * K + static_cast<long long>(ufirst + uu) * PER);
    }
#pragma unroll
    for (int j = 0; j < kStageBatch; ++j) {
      const int it = base + j * static_cast<int>(blockDim.x) + static_cast<int>(threadIdx.x);
      const int uu = it / M, m = it - uu * M;
      if (it < items) {
        const bool live = ufirst + uu < units;
#pragma unroll
        for (int p = 0; p < NP; ++p)
          put(uu, m, p, live ? (v[j].half(lo_k(p)) | (v[j].half(hi_k(p)) << 16)) : 0u);
      }
    }
  }
}

// Raw scale/zero words of columns n0..n0+3 for group g (loads only; decoded later so the
// loads overlap the activation staging).
template <int BITS>
struct SZRaw {
  uint2 sv;
  uint32_t zf;
  __device__ __forceinline__ void load(const Args& a, int g, int n0) {
    sv = __ldg(reinterpret_cast<const uint2*>(a.scales + static_cast<long long>(g) * a.N + n0));
    zf = zeros4<BITS>(a.qzeros + static_cast<long long>(g) * a.zwords, n0);
  }
  __device__ __forceinline__ void decode(int zero_offset, float (&s)[4], int (&z)[4]) const {
    s[0] = __half2float(__ushort_as_half(static_cast<uint16_t>(sv.x & 0xFFFFu)));
    s[1] = __half2float(__ushort_as_half(static_cast<uint16_t>(sv.x >> 16)));
    s[2] = __half2float(__ushort_as_half(static_cast<uint16_t>(sv.y & 0xFFFFu)));
    s[3] = __half2float(__ushort_as_half(static_cast<uint16_t>(sv.y >> 16)));
#pragma unroll
    for (int c = 0; c < 4; ++c)
      z[c] = static_cast<int>((zf >> (BITS * c)) & Pack<BITS>::kMask) + zero_offset;
  }
};

// Shared memory of one CTA: [staged activations | per-warp partials] (aliased, one after the
// other in time), then the receive slots of the cluster reduce-scatter (never aliased).
template <int BITS, int MT, typename T, bool HALF>
__host__ __device__ constexpr size_t recv_offset(int units, int cs) {
  const size_t upc = static_cast<size_t>((units + cs - 1) / cs);
  const size_t stage = HALF ? upc * DiffPairs<T, (HALF ? BITS : 4)>::kPairs * MT * 4
                            : upc * Pack<BITS>::kPerUnit * MT * 4;
  const size_t red = static_cast<size_t>(kWarps) * MT * kSlab * 4;
  const size_t m = stage > red ? stage : red;
  return (m + 15) & ~static_cast<size_t>(15);
}
template <int BITS, int MT, typename T, bool HALF>
size_t smem_bytes(int units, int cs) {
  return recv_offset<BITS, MT, T, HALF>(units, cs) + static_cast<size_t>(MT) * kSlab * 4;
}

// Few-token instantiations are capped at 102 registers so five CTAs (20 warps) fit on an SM
// and the whole grid is resident in one wave.
template <int BITS, int MT, typename T, bool HALF, bool ACT>
__global__ void __launch_bounds__(kThreads, (MT <= 2 ? 5 : 1)) k_decode(const Args a) {
  using P = Pack<BITS>;
  constexpr int PER = P::kPerUnit;
  constexpr int ROWS = P::kRowsPerUnit;
  constexpr int CH = ROWS == 3 ? 2 : 4;          // register ring: units in flight per warp
  extern __shared__ __align__(16) unsigned char smem[];

  pdl_launch_dependents();
  cluster_arrive_relaxed();                      // matched by cluster_wait() before the reduction
  cg::cluster_group cluster = cg::this_cluster();
  const int cs = static_cast<int>(gridDim.x);   // grid x == cluster x
  const int rank = static_cast<int>(blockIdx.x);
  const int n_base = static_cast<int>(blockIdx.y) * kSlab;
  const int warp = threadIdx.x >> 5, lane = threadIdx.x & 31;
  const int n0 = n_base + lane * 4;
  // Lanes past the last column read the last valid columns (N % 4 == 0) and store nothing:
  // the hot loop needs no per-lane predicate.
  const int n0c = n0 < a.N ? n0 : a.N - 4;

  int cu0, cu1;
  split(a.units, cs, rank, cu0, cu1);
  int wu0, wu1;
  split(cu1 - cu0, kWarps, warp, wu0, wu1);
  wu0 += cu0;
  wu1 += cu0;

  const long long ustride = static_cast<long long>(ROWS) * a.N;   // words between units
  const int32_t* qw = a.qweight + n0c;
  auto unit_ptr = [&](int u, int r) { return qw + u * ustride + static_cast<long long>(r) * a.N; };
  auto load_unit = [&](uint4 (&dst)[ROWS], int u) {
#pragma unroll
    for (int r = 0; r < ROWS; ++r) dst[r] = ld_stream_v4(unit_ptr(u, r));
  };

  // The whole weight range of this warp is requested into L2 up front: the prefetches need no
  // registers, keep HBM busy, and the register ring below then mostly hits L2.  They are issued
  // before griddepcontrol.wait; that is safe because L2 is the point of coherence (a line written
  // by the previous kernel is never served stale from L2) and every real load comes after the
  // wait.
  for (int u = wu0; u < wu1; ++u)
#pragma unroll
    for (int r = 0; r < ROWS; ++r) prefetch_l2(unit_ptr(u, r));
  pdl_wait();            // the previous kernel's writes are visible from here on
  // Rolling ring: slot b holds unit ub + b; it is refilled with unit ub + b + CH right after
  // use, so CH units per warp stay in flight for the whole loop.
  uint4 ring[CH][ROWS];
#pragma unroll
  for (int b = 0; b < CH; ++b)
    if (wu0 + b < wu1) load_unit(ring[b], wu0 + b);

  const T* A = static_cast<const T*>(a.A);
  const int kbase = cu0 * PER;
  const int ucount = cu1 - cu0;

  float acc[MT][4];
#pragma unroll
  for (int m = 0; m < MT; ++m)
#pragma unroll
    for (int c = 0; c < 4; ++c) acc[m][c] = 0.f;

  if constexpr (HALF) {
    // ---------------------------------------------------------------- 16-bit path
    using DP = DiffPairs<T, BITS>;
    constexpr int NP = DP::kPairs;
    constexpr bool kFlushEveryUnit = std::is_same<T, __nv_bfloat16>::value;
    const int upg = a.group / PER;                 // units per group (group % PER == 0 here)
    int g = wu0 / upg;
    int left = upg - (wu0 - g * upg);              // units left in group g
    // Scale/zero words of the current group and, one group ahead, of the next: no global load
    // sits on the critical path at a group boundary.
    SZRaw<BITS> raw, raw_next;
    const int g_last = (wu1 - 1) / upg;
    if (wu0 < wu1) raw.load(a, g, n0c);            // in flight during the staging below
    if (wu0 < wu1 && g < g_last) raw_next.load(a, g + 1, n0c);

    // activation pairs: sAP[(unit * NP + p) * MT + m] = (a[m][k0 + lo_k(p)], a[m][k0 + hi_k(p)])
    uint32_t* sAP = reinterpret_cast<uint32_t*>(smem);
    const uint16_t* A16 = reinterpret_cast<const uint16_t*>(A);
    if (a.M < MT)
      for (int i = threadIdx.x; i < ucount * NP * MT; i += kThreads)
        if (i % MT >= a.M) sAP[i] = 0u;
    stage_pairs<PER, NP>(A16, a.M, a.K, cu0, ucount, a.units,
                         [](int p) { return DP::lo_k(p); }, [](int p) { return DP::hi_k(p); },
                         [&](int uu, int m, int p, uint32_t v) { sAP[(uu * NP + p) * MT + m] = v; });
    __syncthreads();

    float accg[MT][4];
    uint32_t acch[MT][4];
#pragma unroll
    for (int m = 0; m < MT; ++m)
#pragma unroll
      for (int c = 0; c < 4; ++c) { accg[m][c] = 0.f; acch[m][c] = 0u; }
    float s[4];
    uint32_t kz[4][DP::kConsts];
    auto set_group = [&]() {
      int z[4];
      raw.decode(a.zero_offset, s, z);
#pragma unroll
      for (int c = 0; c < 4; ++c) DP::consts(z[c], kz[c]);
    };
    auto flush = [&]() {
#pragma unroll
      for (int m = 0; m < MT; ++m)
#pragma unroll
        for (int c = 0; c < 4; ++c) {
          accg[m][c] += sum2_f32(acch[m][c], T());
          acch[m][c] = 0u;
        }
    };
    auto fold = [&]() {
#pragma unroll
      for (int m = 0; m < MT; ++m)
#pragma unroll
        for (int c = 0; c < 4; ++c) {
          acc[m][c] = fmaf(s[c], accg[m][c], acc[m][c]);
          accg[m][c] = 0.f;
        }
    };
    auto process = [&](int ub) {
#pragma unroll
      for (int b = 0; b < CH; ++b) {
        const int u = ub + b;
        if (u >= wu1) break;
        uint32_t ap[NP * MT];
        const uint32_t* src = sAP + (u - cu0) * NP * MT;
        if constexpr ((NP * MT) % 4 == 0) {
#pragma unroll
          for (int i = 0; i < NP * MT / 4; ++i) {
            const uint4 v = reinterpret_cast<const uint4*>(src)[i];
            ap[4 * i] = v.x; ap[4 * i + 1] = v.y; ap[4 * i + 2] = v.z; ap[4 * i + 3] = v.w;
          }
        } else {
#pragma unroll
          for (int i = 0; i < NP * MT / 2; ++i) {
            const uint2 v = reinterpret_cast<const uint2*>(src)[i];
            ap[2 * i] = v.x; ap[2 * i + 1] = v.y;
          }
        }
        const uint4 wv = ring[b][0];
        if (u + CH < wu1) load_unit(ring[b], u + CH);
#pragma unroll
        for (int c = 0; c < 4; ++c) {
          uint32_t d[NP];
          DP::run((&wv.x)[c], kz[c], d);
#pragma unroll
          for (int p = 0; p < NP; ++p)
#pragma unroll
            for (int m = 0; m < MT; ++m) acch[m][c] = fma2(ap[p * MT + m], d[p], acch[m][c], T());
        }
        if (kFlushEveryUnit || (b & 3) == 3) flush();
        if (--left == 0) {                         // group boundary (warp-uniform)
          if (!kFlushEveryUnit) flush();
          fold();
          left = upg;
          if (u + 1 < wu1) {
            ++g;
            raw = raw_next;
            set_group();
            if (g < g_last) raw_next.load(a, g + 1, n0c);
          }
        }
      }
      if (!kFlushEveryUnit) flush();
    };

    if (wu0 < wu1) set_group();
    for (int ub = wu0; ub < wu1; ub += CH) process(ub);
    if (wu0 < wu1 && left != upg) fold();          // range ended inside a group
  } else {
    // ---------------------------------------------------------------- fp32 path
    float* sA = reinterpret_cast<float*>(smem);   // sA[(k - kbase) * MT + m]
    const int kcount = ucount * PER;
    for (int i = threadIdx.x; i < kcount * MT; i += kThreads) {
      const int m = i / kcount, kk = i - m * kcount;
      sA[kk * MT + m] =
          m < a.M ? F16Traits<T>::to_f32(A[static_cast<long long>(m) * a.K + kbase + kk]) : 0.f;
    }
    __syncthreads();
    float s[4];
    int z[4];
    int cur_g = -1;
    auto process = [&](int ub) {
#pragma unroll
      for (int b = 0; b < CH; ++b) {
        const int u = ub + b;
        if (u >= wu1) break;
        const int k0 = u * PER;
        const int kk0 = k0 - kbase;
        uint4 wv[ROWS];
#pragma unroll
        for (int r = 0; r < ROWS; ++r) wv[r] = ring[b][r];
        if (u + CH < wu1) load_unit(ring[b], u + CH);
#pragma unroll 4
        for (int j = 0; j < PER; ++j) {
          const int k = k0 + j;
          const int g = ACT ? checked_group(a, k) : k / a.group;
          if (ACT || g != cur_g) {
            load_sz<BITS>(a, g, n0c, s, z);
            cur_g = g;
          }
          float w[4];
#pragma unroll
          for (int c = 0; c < 4; ++c) w[c] = diff_f32(unit_code<BITS>(wv, c, j), z[c]) * s[c];
          const float* ak = sA + (kk0 + j) * MT;
#pragma unroll
          for (int m = 0; m < MT; ++m) {
            const float av = ak[m];
#pragma unroll
            for (int c = 0; c < 4; ++c) acc[m][c] = fmaf(av, w[c], acc[m][c]);
          }
        }
      }
    };
    for (int ub = wu0; ub < wu1; ub += CH) process(ub);
  }

  // ---- reduction: warps (shared memory), then a reduce-scatter over the cluster: every CTA
  // pushes each column's partial sum into the shared memory of the CTA that owns the column
  // (distributed shared memory), one cluster barrier, and each owner sums its slots in rank
  // order (deterministic) and writes C.
  __syncthreads();   // every warp is done reading the staged activations
  float* red = reinterpret_cast<float*>(smem);                        // [kWarps][MT][kSlab]
  // [cs][MT][kSlab / cs]: a region of its own -- peers may push into it while this CTA is
  // still reading its staged activations.
  float* recv = reinterpret_cast<float*>(smem + recv_offset<BITS, MT, T, HALF>(a.units, cs));
#pragma unroll
  for (int m = 0; m < MT; ++m)
    *reinterpret_cast<float4*>(red + (warp * MT + m) * kSlab + lane * 4) =
        make_float4(acc[m][0], acc[m][1], acc[m][2], acc[m][3]);
  __syncthreads();
  const int per_rank = kSlab / cs;
  cluster_wait();    // every CTA of the cluster is running: remote stores are safe
  for (int i = threadIdx.x; i < MT * kSlab; i += kThreads) {
    float v = red[i];
#pragma unroll
    for (int w = 1; w < kWarps; ++w) v += red[w * MT * kSlab + i];
    const int m = i / kSlab, col = i - m * kSlab;
    const int owner = col / per_rank;
    float* dst = cluster.map_shared_rank(recv, owner);
    dst[(rank * MT + m) * per_rank + (col - owner * per_rank)] = v;
  }
  cluster.sync();    // all pushes visible to their owners
  T* C = static_cast<T*>(a.C);
  for (int i = threadIdx.x; i < MT * per_rank; i += kThreads) {
    const int m = i / per_rank, c = i - m * per_rank;
    const int n = n_base + rank * per_rank + c;
    if (m < a.M && n < a.N) {
      float v = 0.f;
      for (int q = 0; q < cs; ++q) v += recv[(q * MT + m) * per_rank + c];
      C[static_cast<long long>(m) * a.N + n] = F16Traits<T>::from_f32(v);
    }
  }
}

template <int BITS, int MT, typename T, bool HALF, bool ACT>
cudaError_t launch_one(const Problem& p, int cs, cudaStream_t stream) {
  Args a;
  a.A = p.A; a.M = p.M; a.K = p.K; a.N = p.N;
  a.qweight = p.qweight; a.qzeros = p.qzeros;
  a.scales = static_cast<const __half*>(p.scales);
  a.g_idx = p.g_idx; a.group = p.group; a.G = p.G; a.zero_offset = p.zero_offset;
  a.zwords = p.N * BITS / 32;
  a.units = p.K / Pack<BITS>::kPerUnit;
  a.C = p.out; a.status = p.status;
  const int slabs = (p.N + kSlab - 1) / kSlab;
  const size_t smem = smem_bytes<BITS, MT, T, HALF>(a.units, cs);
  auto kern = k_decode<BITS, MT, T, HALF, ACT>;
  if (smem > 48 * 1024) {
    cudaError_t e = cudaFuncSetAttribute(kern, cudaFuncAttributeMaxDynamicSharedMemorySize,
                                         static_cast<int>(smem));
    if (e != cudaSuccess) return e;
  }
  cudaLaunchConfig_t cfg = {};
  cfg.gridDim = dim3(cs, slabs, 1);
  cfg.blockDim = dim3(kThreads, 1, 1);
  cfg.dynamicSmemBytes = smem;
  cfg.stream = stream;
  cudaLaunchAttribute attr[2];
  attr[0].id = cudaLaunchAttributeClusterDimension;
  attr[0].val.clusterDim.x = cs;
  attr[0].val.clusterDim.y = 1;
  attr[0].val.clusterDim.z = 1;
  attr[1].id = cudaLaunchAttributeProgrammaticStreamSerialization;
  attr[1].val.programmaticStreamSerializationAllowed = 1;
  cfg.attrs = attr;
  cfg.numAttrs = 2;
  return cudaLaunchKernelEx(&cfg, kern, a);
}

// Cluster size: enough warps to fill the GPU (about 24 per SM), at least two units per warp.
inline int choose_cluster(const Problem& p, int per_unit) {
  const int slabs = (p.N + kSlab - 1) / kSlab;
  const int units = p.K / per_unit;
  const int target = device_info().sm_count * 24;
  int cs = 1;
  while (cs < 8 && slabs * cs * kWarps < target && units >= 4 * cs * kWarps) cs *= 2;
  return cs;
}

template <int BITS, int MT, typename T, bool FOLD>
cudaError_t launch_mma(const Problem& p, int cs, cudaStream_t stream);

template <int BITS, int MT, typename T>
cudaError_t launch_mt(const Problem& p, cudaStream_t stream) {
  const int cs = choose_cluster(p, Pack<BITS>::kPerUnit);
  constexpr bool kHas16 = (BITS == 2 || BITS == 4 || (BITS == 8 && std::is_same<T, __half>::value));
  if constexpr (MT >= 8) {
    // tensor cores from registers; the scale folds per group when groups align with k-tiles
    const bool fold = kHas16 && p.g_idx == nullptr && (p.group % (4 * Pack<BITS>::kPerUnit)) == 0;
    if constexpr (kHas16) {
      if (fold) return launch_mma<BITS, MT, T, true>(p, cs, stream);
    }
    return launch_mma<BITS, MT, T, false>(p, cs, stream);
  } else {
    const bool factorable = p.g_idx == nullptr && (p.group % Pack<BITS>::kPerUnit) == 0;
    if constexpr (kHas16) {
      if (factorable) return launch_one<BITS, MT, T, true, false>(p, cs, stream);
    }
    if (p.g_idx) return launch_one<BITS, MT, T, false, true>(p, cs, stream);
    return launch_one<BITS, MT, T, false, false>(p, cs, stream);
  }
}

// Every M <= 32 runs the register-MMA kernel (token blocks of 8): even at one token, handing
// the multiply-accumulate to the tensor core leaves the SM with only the unpack to issue.
template <int BITS>
cudaError_t launch_bits(const Problem& p, cudaStream_t stream) {
  if (p.dtype == 0) {
    if (p.M <= 8) return launch_mt<BITS, 8, __half>(p, stream);
    if (p.M <= 16) return launch_mt<BITS, 16, __half>(p, stream);
    return launch_mt<BITS, 32, __half>(p, stream);
  }
  if (p.M <= 8) return launch_mt<BITS, 8, __nv_bfloat16>(p, stream);
  if (p.M <= 16) return launch_mt<BITS, 16, __nv_bfloat16>(p, stream);
  return launch_mt<BITS, 32, __nv_bfloat16>(p, stream);
}

}  // namespace decode
}  // namespace gptq
