// act_order.cu -- act-order checkpoints (page "增强 vLLM 对 GPTQv2 格式的支持：分析与实现", section
// "LLM 的权重量化": the quantization groups are the row sets {k : g_idx[k] == g}).  Sorting the
// rows by group makes every group a contiguous row range, and A @ W == A[:, perm] @ W_sorted with
// perm[k'] the original row now at row k'.  Three kernels serve that:
//  * k_sort_groups: the stable sort of the rows by g_idx on the device (perm, and where each
//    sorted row's code sits in a packed column) and a flag saying whether every group holds
//    exactly `group` rows (the layout the group-wise kernels need);
//  * k_repack_rows: the packed weight rewritten in that row order (the device counterpart of the
//    host function gptq_prepack_act_order), when the flag allows;
//  * k_gather_cols: the activation columns in that order, A'[m][k'] = A[m][perm[k']], written once
//    into caller-provided workspace so that every column slab of the decode kernel then reads
//    contiguous activations.
#include <cuda_runtime.h>
#include <stdint.h>

#include <atomic>

#include "gptq_device.cuh"
#include "gptq_internal.h"

namespace gptq {
namespace {

constexpr int kSortThreads = 1024;   // one CTA: 32 warps, each owning a contiguous K/32 rows
// status bit GPTQ_DEV_GIDX_GROUPS: the stand-alone device prepack found g_idx it cannot sort
constexpr unsigned kStatusGidxGroups = 0x10u;

// Where sorted row k' finds its code in a column: the packed word (row of qweight) and the bit
// offset of the code of original row k inside it (LSB-first; a 3-bit code may run into the next
// word).  Entry = word << 5 | bit offset.
template <int BITS>
__device__ __forceinline__ uint32_t code_source(int k) {
  if constexpr (BITS == 3) {
    const int bit = 3 * (k & 31);
    return static_cast<uint32_t>(((k >> 5) * 3 + (bit >> 5)) << 5 | (bit & 31));
  } else {
    constexpr int PER = 32 / BITS;
    return static_cast<uint32_t>((k / PER) << 5 | (k % PER) * BITS);
  }
}

// Stable sort of the K rows by group.  The keys are staged in shared memory first (all loads in
// flight at once).  Warp w owns rows [w K/32, (w + 1) K/32): pass 1 counts each group's rows per
// warp (hist[w][g], shared-memory atomics), pass 2 turns the counts into each warp's first slot
// inside each group (one warp per group, a shuffle scan over the 32 warps' counts) and checks that
// every group holds `group` rows, pass 3 walks the warp's rows in order, 32 at a time: equal keys
// among the 32 are found with one warp ballot per key bit (their order is the lane order; a
// ballot per bit measured faster than match.any here), and the lowest lane of each key takes
// the key's next slots with one atomic add that returns the slot before it.  A warp's atomics
// execute in its program order, so slots follow the row order; batches of eight such steps issue
// their atomics back to back.  Ties keep their row order, so the result is the one ordering the
// host prepack also produces: perm[g * group + slot] = k, src[g * group + slot] = code_source(k).
// flag: 1 when every entry is in [0, G) and every group holds exactly `group` rows (perm and src
// are then complete), else 0 (both left unwritten).  The repack that follows may start its
// weight copies at once (programmatic dependent launch); it waits for this grid before reading
// what it wrote.
template <int BITS>
__global__ void __launch_bounds__(kSortThreads) k_sort_groups(const int32_t* __restrict__ g_idx, int K, int G,
                                                              int group, int32_t* __restrict__ perm,
                                                              uint32_t* __restrict__ src, int* __restrict__ flag,
                                                              int staged) {
  // [32][G] counts; then, when `staged`, perm and src of all K rows; then the keys [K] (16-bit)
  extern __shared__ uint32_t hist[];
  int32_t* sperm = reinterpret_cast<int32_t*>(hist + 32 * G);
  uint32_t* ssrc = hist + 32 * G + (staged ? K : 0);
  uint16_t* keys = reinterpret_cast<uint16_t*>(hist + 32 * G + (staged ? 2 * K : 0));
  __shared__ int bad;
  asm volatile("griddepcontrol.launch_dependents;" ::: "memory");
  const int warp = threadIdx.x >> 5, lane = threadIdx.x & 31;
  if (threadIdx.x == 0) bad = 0;
  for (int i = threadIdx.x; i < 32 * G; i += kSortThreads) hist[i] = 0u;
  __syncthreads();
  constexpr int kBatch = 8;                    // loads in flight per thread
  for (int base = 0; base < K; base += kSortThreads * kBatch) {
    int v[kBatch];
#pragma unroll
    for (int b = 0; b < kBatch; ++b) {
      const int k = base + b * kSortThreads + static_cast<int>(threadIdx.x);
      v[b] = k < K ? __ldg(g_idx + k) : 0;
    }
#pragma unroll
    for (int b = 0; b < kBatch; ++b) {
      const int k = base + b * kSortThreads + static_cast<int>(threadIdx.x);
      if (k < K) {
        const bool valid = v[b] >= 0 && v[b] < G;
        if (!valid) bad = 1;
        keys[k] = valid ? static_cast<uint16_t>(v[b]) : static_cast<uint16_t>(0xFFFFu);
      }
    }
  }
  __syncthreads();
  if (bad) {                                   // an entry out of range: the per-row kernels run
    if (threadIdx.x == 0) *flag = 0;
    return;
  }
  const int chunk = K / 32;
  const int k_lo = warp * chunk, k_hi = k_lo + chunk;
  uint32_t* h = hist + warp * G;
  for (int k = k_lo + lane; k < k_hi; k += 32) atomicAdd(&h[keys[k]], 1u);
  __syncthreads();
  for (int g = warp; g < G; g += 32) {
    const uint32_t c = hist[lane * G + g];
    uint32_t incl = c;
#pragma unroll
    for (int o = 1; o < 32; o <<= 1) {
      const uint32_t t = __shfl_up_sync(0xFFFFFFFFu, incl, o);
      if (lane >= o) incl += t;
    }
    hist[lane * G + g] = incl - c;
    if (lane == 31 && incl != static_cast<uint32_t>(group)) bad = 1;
  }
  __syncthreads();
  if (bad) {
    if (threadIdx.x == 0) *flag = 0;
    return;
  }
  constexpr int kSteps = 8;
  const int nbits = 32 - __clz(G - 1);         // keys below G (no bit at all when G == 1)
  for (int k0 = k_lo; k0 < k_hi; k0 += 32 * kSteps) {
    int g[kSteps];
    unsigned peers[kSteps];
    uint32_t old[kSteps];
    bool in[kSteps];
#pragma unroll
    for (int i = 0; i < kSteps; ++i) {
      const int k = k0 + 32 * i + lane;
      in[i] = k < k_hi;
      g[i] = in[i] ? static_cast<int>(keys[k]) : 0;
      peers[i] = __ballot_sync(0xFFFFFFFFu, in[i]);   // lanes past the chunk match no lane
    }
    // lanes with equal keys: one ballot per key bit (up to eight independent steps side by side;
    // a step past the chunk, the same for the whole warp, takes no ballot)
    for (int b = 0; b < nbits; ++b) {
#pragma unroll
      for (int i = 0; i < kSteps; ++i) {
        if (k0 + 32 * i >= k_hi) continue;
        const bool v = (g[i] >> b) & 1;
        const unsigned bal = __ballot_sync(0xFFFFFFFFu, v);
        peers[i] &= v ? bal : ~bal;
      }
    }
#pragma unroll
    for (int i = 0; i < kSteps; ++i) {
      old[i] = 0u;
      if (in[i] && lane == __ffs(peers[i]) - 1) old[i] = atomicAdd(&h[g[i]], static_cast<uint32_t>(__popc(peers[i])));
    }
#pragma unroll
    for (int i = 0; i < kSteps; ++i) {
      const uint32_t slot = __shfl_sync(0xFFFFFFFFu, old[i], in[i] ? __ffs(peers[i]) - 1 : lane);
      if (in[i]) {
        const int k = k0 + 32 * i + lane;
        const int dst = g[i] * group + static_cast<int>(slot) + __popc(peers[i] & ((1u << lane) - 1u));
        if (staged) {
          sperm[dst] = k;
          ssrc[dst] = code_source<BITS>(k);
        } else {
          perm[dst] = k;
          src[dst] = code_source<BITS>(k);
        }
      }
    }
  }
  __syncthreads();
  if (staged) {
    // scattered stores stay in shared memory; global memory gets 16-byte coalesced ones (one SM
    // issuing K scattered 4-byte global stores took most of the kernel's time)
    for (int i = threadIdx.x; i < K / 4; i += kSortThreads) {
      reinterpret_cast<int4*>(perm)[i] = reinterpret_cast<const int4*>(sperm)[i];
      reinterpret_cast<uint4*>(src)[i] = reinterpret_cast<const uint4*>(ssrc)[i];
    }
    __syncthreads();
  }
  if (threadIdx.x == 0) *flag = 1;
}

// The packed weight in sorted row order: output row k' holds the code of input row perm[k'] in
// each column (every width, LSB-first, 3-bit units of 32 codes over 3 words).  One CTA per strip
// of sw columns (32, 16, 8 or 4: the widest whose packed column fits) holds the strip's whole
// packed column in shared memory (asynchronous 16-byte copies of each row segment, all in flight
// at once, plus one zero row so that a 3-bit code's two-word read never leaves the strip).  Each
// thread then assembles one output unit for four adjacent columns: per code one table entry (the
// same for every column: src from the sort), one 16-byte shared-memory read and per column a
// rotation and an and-or (a 3-bit code at bit 30 or 31 also reads the next word: a funnel shift
// takes it out and a rotation places it).  Eight threads cover a 32-column row
// segment, so each warp's 16-byte writes form 128-byte segments.  The copies are issued before
// griddepcontrol.wait (they read the checkpoint, not the sort's output); the rest runs only when
// the sort accepted g_idx (flag 1).  status (nullable): with flag 0 the first CTA raises
// kStatusGidxGroups there (the stand-alone prepack, which has no other path to take).
template <int BITS>
__global__ void __launch_bounds__(256) k_repack_rows(const uint32_t* __restrict__ qw,
                                                     const uint32_t* src, const int* flag, int K, int N,
                                                     int sw, uint32_t* __restrict__ out, unsigned* status) {
  using P = Pack<BITS>;
  constexpr int PER = P::kPerUnit;
  constexpr int ROWS = P::kRowsPerUnit;
  extern __shared__ uint4 strip_v[];
  uint32_t* strip = reinterpret_cast<uint32_t*>(strip_v);   // [rows + 1][sw]
  const int units = K / PER;
  const int rows = units * ROWS;
  const int n0 = blockIdx.x * sw;
  const int vec = sw / 4;
  const uint32_t sbase = static_cast<uint32_t>(__cvta_generic_to_shared(strip_v));
  for (int i = threadIdx.x; i < rows * vec; i += blockDim.x) {
    const int r = i / vec, q = i - r * vec;
    asm volatile("cp.async.cg.shared.global [%0], [%1], 16;" ::"r"(sbase + 16u * static_cast<uint32_t>(i)),
                 "l"(qw + static_cast<long long>(r) * N + n0 + 4 * q)
                 : "memory");
  }
  for (int i = rows * vec + threadIdx.x; i < (rows + 1) * vec; i += blockDim.x) strip_v[i] = make_uint4(0u, 0u, 0u, 0u);
  // the sort's output (src, flag) is read only after the sort grid has completed; src and flag
  // are plain (not restrict-qualified) pointers so that no load of them moves above the wait
  asm volatile("griddepcontrol.wait;" ::: "memory");
  asm volatile("cp.async.wait_all;" ::: "memory");   // own copies land before any exit
  if (*static_cast<const volatile int*>(flag) != 1) {
    if (status != nullptr && blockIdx.x == 0 && threadIdx.x == 0) atomicOr(status, kStatusGidxGroups);
    return;
  }
  __syncthreads();
  const int c4 = 4 * (threadIdx.x % vec);
  const int lanes = blockDim.x / vec;
  for (int u = threadIdx.x / vec; u < units; u += lanes) {
    uint32_t acc[4][ROWS];
#pragma unroll
    for (int cc = 0; cc < 4; ++cc)
#pragma unroll
      for (int r = 0; r < ROWS; ++r) acc[cc][r] = 0u;
    // the unit's table entries, 16 bytes at a time (written by the sort: coherent loads)
    uint32_t ent[PER];
#pragma unroll
    for (int j = 0; j < PER; j += 4) {
      const uint4 v = *reinterpret_cast<const uint4*>(src + u * PER + j);
      ent[j] = v.x; ent[j + 1] = v.y; ent[j + 2] = v.z; ent[j + 3] = v.w;
    }
#pragma unroll
    for (int j = 0; j < PER; ++j) {
      const uint32_t e = ent[j];
      const uint32_t sh = e & 31u;
      const uint32_t* wp = strip + (e >> 5) * sw + c4;
      const uint4 lo = *reinterpret_cast<const uint4*>(wp);
      const int ob = BITS * j;                             // a constant once unrolled
      if constexpr (BITS == 3) {
        // rot: the code at bit ow of its output word, its bits past bit 31 wrapped to bits 0..
        // Only a code at bit 30 or 31 runs into the next word (2 of a unit's 32): that word is
        // read just then, so the strip is read about once per code instead of twice.
        const uint32_t ow = static_cast<uint32_t>(ob & 31);
        uint32_t rot[4];
        if (sh <= 29u) {
#pragma unroll
          for (int cc = 0; cc < 4; ++cc) rot[cc] = __funnelshift_r((&lo.x)[cc], (&lo.x)[cc], sh - ow);
        } else {
          const uint4 hi = *reinterpret_cast<const uint4*>(wp + sw);
#pragma unroll
          for (int cc = 0; cc < 4; ++cc) {
            const uint32_t code = __funnelshift_r((&lo.x)[cc], (&hi.x)[cc], sh) & 7u;
            rot[cc] = __funnelshift_l(code, code, ow);
          }
        }
#pragma unroll
        for (int cc = 0; cc < 4; ++cc) {
          acc[cc][ob >> 5] |= rot[cc] & (7u << ow);
          if (ow + BITS > 32) acc[cc][(ob >> 5) + 1] |= rot[cc] & (7u >> (32 - ow));
        }
      } else {
        // a rotation by (sh - ob) mod 32 moves the code from bit sh to bit ob (2/4/8-bit codes
        // never straddle a word), and one and-or places it: two instructions per code
#pragma unroll
        for (int cc = 0; cc < 4; ++cc) {
          const uint32_t w = (&lo.x)[cc];
          acc[cc][0] |= __funnelshift_r(w, w, e - static_cast<uint32_t>(ob)) & (P::kMask << ob);
        }
      }
    }
#pragma unroll
    for (int r = 0; r < ROWS; ++r)
      *reinterpret_cast<uint4*>(out + static_cast<long long>(u * ROWS + r) * N + n0 + c4) =
          make_uint4(acc[0][r], acc[1][r], acc[2][r], acc[3][r]);
  }
}

// Consecutive threads on consecutive 8-column pieces of a row: the writes and the perm reads
// coalesce; the reads of A are a gather within the row (the row stays in L1/L2).  The kernel lets
// the dependent GEMM launch at once (its CTAs stream weights meanwhile) and waits for its own
// predecessor before reading A.
__global__ void __launch_bounds__(256) k_gather_cols(const uint16_t* __restrict__ A,
                                                     const int32_t* __restrict__ perm, int M, int K,
                                                     uint16_t* __restrict__ out) {
  asm volatile("griddepcontrol.launch_dependents;" ::: "memory");
  asm volatile("griddepcontrol.wait;" ::: "memory");
  // eight consecutive k' per thread-iteration: two 16-byte reads of perm, eight 2-byte gathers
  // from the row, one 16-byte store (K is a multiple of 32; perm and out are 16-byte aligned)
  const int k8 = K / 8;
  const long long total = static_cast<long long>(M) * k8;
  const long long step = static_cast<long long>(gridDim.x) * blockDim.x;
  for (long long i = static_cast<long long>(blockIdx.x) * blockDim.x + threadIdx.x; i < total; i += step) {
    const int m = static_cast<int>(i / k8), k0 = static_cast<int>(i - static_cast<long long>(m) * k8) * 8;
    const int4 p0 = __ldg(reinterpret_cast<const int4*>(perm + k0));
    const int4 p1 = __ldg(reinterpret_cast<const int4*>(perm + k0 + 4));
    const int src[8] = {p0.x, p0.y, p0.z, p0.w, p1.x, p1.y, p1.z, p1.w};
    const uint16_t* row = A + static_cast<long long>(m) * K;
    uint32_t h[8];
#pragma unroll
    for (int j = 0; j < 8; ++j) {
      const int sk = src[j] < 0 ? 0 : (src[j] >= K ? K - 1 : src[j]);   // a bad entry never reads outside the row
      h[j] = __ldg(row + sk);
    }
    reinterpret_cast<uint4*>(out)[i] = make_uint4(h[0] | (h[1] << 16), h[2] | (h[3] << 16), h[4] | (h[5] << 16),
                                                  h[6] | (h[7] << 16));
  }
}

// Opt in to up to kMaxActOrderSmem bytes of dynamic shared memory for `kern`, once per device
// (the 48 KB default counts the kernel's static shared memory too, so it is raised whatever the
// size asked for).
template <typename F>
cudaError_t allow_smem(F kern, std::atomic<unsigned long long>& done) {
  const int dev = device_info().device;
  if (dev < 64 && (done.load(std::memory_order_relaxed) & (1ull << dev))) return cudaSuccess;
  const cudaError_t e = cudaFuncSetAttribute(kern, cudaFuncAttributeMaxDynamicSharedMemorySize,
                                             static_cast<int>(kMaxActOrderSmem));
  if (e == cudaSuccess && dev < 64) done.fetch_or(1ull << dev, std::memory_order_relaxed);
  return e;
}

size_t sort_groups_smem(int K, int G) { return static_cast<size_t>(G) * 32 * 4 + static_cast<size_t>(K) * 2; }

// With room for the whole row order and code table as well, the sort places rows in shared memory.
bool sort_groups_staged(int K, int G) { return sort_groups_smem(K, G) + static_cast<size_t>(K) * 8 <= kMaxActOrderSmem; }

size_t repack_smem(int K, int bits, int sw) { return (static_cast<size_t>(K) * bits / 32 + 1) * sw * 4; }

template <int BITS>
cudaError_t launch_sort_bits(const int32_t* g_idx, int K, int G, int group, int32_t* perm, uint32_t* src,
                             int* flag, cudaStream_t stream) {
  static std::atomic<unsigned long long> smem_set{0};
  const int staged = sort_groups_staged(K, G) ? 1 : 0;
  const size_t smem = sort_groups_smem(K, G) + (staged ? static_cast<size_t>(K) * 8 : 0);
  cudaError_t e = allow_smem(k_sort_groups<BITS>, smem_set);
  if (e != cudaSuccess) return e;
  k_sort_groups<BITS><<<1, kSortThreads, smem, stream>>>(g_idx, K, G, group, perm, src, flag, staged);
  return cudaGetLastError();
}

template <int BITS>
cudaError_t launch_repack_bits(const int32_t* qweight, const uint32_t* src, const int* flag, int K, int N,
                               int32_t* out, unsigned* status, cudaStream_t stream) {
  static std::atomic<unsigned long long> smem_set{0};
  const int sw = repack_strip_width(K, BITS);
  if (sw == 0) return cudaErrorInvalidValue;
  const size_t smem = repack_smem(K, BITS, sw);
  cudaError_t e = allow_smem(k_repack_rows<BITS>, smem_set);
  if (e != cudaSuccess) return e;
  cudaLaunchConfig_t cfg = {};
  cfg.gridDim = dim3(static_cast<unsigned>(N / sw), 1, 1);
  cfg.blockDim = dim3(256, 1, 1);
  cfg.dynamicSmemBytes = smem;
  cfg.stream = stream;
  cudaLaunchAttribute attr[1];
  attr[0].id = cudaLaunchAttributeProgrammaticStreamSerialization;
  attr[0].val.programmaticStreamSerializationAllowed = 1;
  cfg.attrs = attr;
  cfg.numAttrs = 1;
  return cudaLaunchKernelEx(&cfg, k_repack_rows<BITS>, reinterpret_cast<const uint32_t*>(qweight), src, flag, K,
                            N, sw, reinterpret_cast<uint32_t*>(out), status);
}

}  // namespace

int repack_strip_width(int K, int bits) {
  for (int sw = 32; sw >= 4; sw /= 2)
    if (repack_smem(K, bits, sw) <= kMaxActOrderSmem) return sw;
  return 0;
}

bool sort_groups_fits(int K, int G, int group) {
  return K > 0 && K % 32 == 0 && K / 32 <= 65535 && G > 0 && G < 65535 && group > 0 && group <= 65535 &&
         sort_groups_smem(K, G) <= kMaxActOrderSmem;
}

cudaError_t launch_sort_groups(const int32_t* g_idx, int K, int G, int group, int bits, int32_t* perm,
                               uint32_t* src, int* flag, cudaStream_t stream) {
  if (!sort_groups_fits(K, G, group)) return cudaErrorInvalidValue;
  switch (bits) {
    case 2: return launch_sort_bits<2>(g_idx, K, G, group, perm, src, flag, stream);
    case 3: return launch_sort_bits<3>(g_idx, K, G, group, perm, src, flag, stream);
    case 4: return launch_sort_bits<4>(g_idx, K, G, group, perm, src, flag, stream);
    case 8: return launch_sort_bits<8>(g_idx, K, G, group, perm, src, flag, stream);
    default: return cudaErrorInvalidValue;
  }
}

cudaError_t launch_repack_rows(const int32_t* qweight, const uint32_t* src, const int* flag, int K, int N,
                               int bits, int32_t* out, unsigned* status, cudaStream_t stream) {
  switch (bits) {
    case 2: return launch_repack_bits<2>(qweight, src, flag, K, N, out, status, stream);
    case 3: return launch_repack_bits<3>(qweight, src, flag, K, N, out, status, stream);
    case 4: return launch_repack_bits<4>(qweight, src, flag, K, N, out, status, stream);
    case 8: return launch_repack_bits<8>(qweight, src, flag, K, N, out, status, stream);
    default: return cudaErrorInvalidValue;
  }
}

cudaError_t launch_gather_cols(const void* A, const int32_t* perm, int M, int K, void* out,
                               cudaStream_t stream) {
  const long long total = static_cast<long long>(M) * (K / 8);   // 8-column pieces
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
