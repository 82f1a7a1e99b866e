// prefill.cu -- compute-bound GPTQ GEMM for many tokens (M > 16) on the 5th-generation tensor
// cores: C = A @ dequant(W) with tcgen05.mma (kind::f16, fp32 accumulators in TMEM).
//
// The page "增强 vLLM 对 GPTQv2 格式的支持：分析与实现" (section "调整细节：根据格式选择处理方
// 式") describes gptq_gemm's large-M path as a reconstruct kernel (dequantize with
// zeros[i] + zero_offset) followed by a GEMM.  Here the reconstruction never leaves the SM: each
// packed weight tile is dequantized straight into the shared-memory layout the tensor core reads,
// and a 256 x 256 output tile accumulates over K in tensor memory.
//
// Per CTA (persistent, one per SM, 704 threads, warp-specialised):
//   warp 4      TMA producer: A tile [256 x 64] (128-byte swizzle) and the packed qweight tile
//               [64 k x 256 n] for each k-step into a 3-stage ring;
//   warps 6-21  dequantizers, two threads per tile column (4 chunks of 8 k each): exact
//               q - zero as fp16 (DiffPairs), then one rounding of (q - zero) * scale to fp16
//               (HMUL2: an exact product rounded once), stored K-major with the 128-byte swizzle
//               into a 3-stage B ring (2 for 8-bit), then fence.proxy.async + mbarrier arrive.
//               The next group's scale and zero words are loaded one group ahead;
//   warp 5      TMEM owner and MMA issuer: per k-step 4 x 2 tcgen05.mma (M=128, N=256, K=16),
//               one per 128-row half of A, both reading the same B tile; tcgen05.commit frees
//               the ring slots and signals the accumulators;
//   warps 0-3   epilogue: tcgen05.ld of the two 128 x 256 fp32 accumulators (512 TMEM
//               columns), times the row's power-of-two scale (bf16 input), rounding to A's dtype,
//               direct 64-byte row-segment stores.
// The multiply is fp16 x fp16 for both activation types.  bf16 activations are first rewritten
// into the caller's workspace as fp16 times a power of two per row (k_rows_to_f16, exact), and
// that power of two is multiplied back into the fp32 accumulators: a bf16 weight operand would
// carry up to 2^-8 relative error per product, beyond the GEMM's 2e-3 bound, while the fp16
// weight carries 2^-11.
// Every mbarrier wait is bounded (2 s of %globaltimer): on expiry the kernel sets
// GPTQ_DEV_TIMEOUT in the status word, every role stops, in-flight copies and MMAs are waited
// for (bounded), TMEM is freed and the CTA exits.
#include <cuda.h>
#include <cudaTypedefs.h>

#include <mutex>

#include "gptq_device.cuh"
#include "gptq_internal.h"
#include "sm100_ptx.cuh"

namespace gptq {
namespace prefill {

constexpr int kBM = 256;            // rows of A per tile (two UMMA M=128 halves)
constexpr int kBN = 256;            // columns per tile (UMMA N=256)
constexpr int kBK = 64;             // k per stage: one 128-byte swizzle row of 16-bit values
constexpr int kEpiWarps = 4;
constexpr int kProducerWarp = 4;
constexpr int kMmaWarp = 5;
constexpr int kDqWarp0 = 6;
constexpr int kDqWarps = 16;        // two threads per tile column (4 chunks each)
constexpr int kThreads = (kDqWarp0 + kDqWarps) * 32;
constexpr uint32_t kTmemCols = 512; // two 128 x 256 fp32 accumulators
constexpr uint32_t kATileBytes = kBM * kBK * 2;
constexpr uint32_t kBTileBytes = kBN * kBK * 2;
constexpr uint64_t kWaitLimitNs = 2000000000ull;

template <int BITS>
struct Geo {
  static constexpr int kRows = kBK * BITS / 32;                // qweight rows per k-step
  static constexpr uint32_t kWBytes = kBN * kRows * 4;         // packed tile bytes
  static constexpr int kStages = 3;                            // A + packed-W ring depth
  static constexpr int kBStages = BITS == 8 ? 2 : 3;           // dequantized-B ring depth
  static constexpr uint32_t kOffW = kStages * kATileBytes;
  static constexpr uint32_t kOffB = kOffW + kStages * kWBytes;
  static constexpr uint32_t kOffBar = kOffB + Geo::kBStages * kBTileBytes;
  // barriers: full[S], empty[S], bfull[BS], bempty[BS], acc_full, acc_empty, drain
  static constexpr uint32_t kNumBars = 2 * kStages + 2 * Geo::kBStages + 3;
  static constexpr uint32_t kOffMisc = kOffBar + kNumBars * 8;  // tmem base, abort flag
  // epilogue staging: per epilogue warp 32 rows x 64 bytes (one 32-column chunk of its rows)
  static constexpr uint32_t kOffEpi = (kOffMisc + 16 + 127) & ~127u;
  static constexpr uint32_t kBytes = kOffEpi + kEpiWarps * 32 * 64;
  static constexpr size_t kDynSmem = kBytes + 1024;             // slack to align the base
};

struct Args {
  int M, N, K, group, G, zero_offset, zwords;
  const int32_t* qzeros;
  const __half* scales;
  const int32_t* g_idx;
  const float* row_scale;   // bf16 input: 2^e per row of A (the fp16 copy was divided by it)
  void* C;
  unsigned* status;
  const int* run_flag;      // nullable: run only if *run_flag == run_when
  int run_when;
};

struct Sync {
  uint32_t base;        // shared address of the aligned dynamic shared memory
  volatile int* abort;
  unsigned* status;
};

// Bounded wait on an mbarrier phase; false if the wait ran out or another role aborted.
__device__ __forceinline__ bool wait_bar(const Sync& s, uint32_t bar, uint32_t parity,
                                         uint64_t limit_ns = kWaitLimitNs) {
  if (ptx::mbar_try_wait(bar, parity)) return true;
  const uint64_t t0 = ptx::globaltimer();
  while (true) {
    if (ptx::mbar_try_wait_hint(bar, parity, 200000u)) return true;
    if (*s.abort) return false;
    if (ptx::globaltimer() - t0 > limit_ns) {
      *s.abort = 1;
      atomicOr(s.status, kStatusTimeout);
      return false;
    }
  }
}

// Byte offset of (row, 16-byte chunk) in a K-major tile stored with the 128-byte swizzle.
__device__ __forceinline__ uint32_t swz(int row, int chunk) {
  return static_cast<uint32_t>((row >> 3) * 1024 + (row & 7) * 128 + ((chunk ^ (row & 7)) << 4));
}

// Runtime zero of column n in qzeros row g.
template <int BITS>
__device__ __forceinline__ int zero_of(const Args& a, int g, int n) {
  const int32_t* row = a.qzeros + static_cast<long long>(g) * a.zwords;
  const int bit = BITS * n;
  uint32_t v = static_cast<uint32_t>(__ldg(row + (bit >> 5))) >> (bit & 31);
  if ((bit & 31) + BITS > 32) v |= static_cast<uint32_t>(__ldg(row + (bit >> 5) + 1)) << (32 - (bit & 31));
  return static_cast<int>(v & Pack<BITS>::kMask) + a.zero_offset;
}

template <int BITS>
__device__ __forceinline__ int clamp_group(const Args& a, int k) {
  if (a.g_idx == nullptr) return k / a.group;
  int g = __ldg(a.g_idx + k);
  if (g < 0 || g >= a.G) {
    atomicOr(a.status, kStatusGidxRange);
    g = g < 0 ? 0 : a.G - 1;
  }
  return g;
}

// Code j (0..7) of local chunk c (0..3) of one thread's half k-step (32 consecutive k), whose
// packed words are w[0 .. R/2 - 1].
template <int BITS>
__device__ __forceinline__ uint32_t local_code(const uint32_t (&w)[Geo<BITS>::kRows / 2], int c,
                                               int j) {
  if constexpr (BITS == 4) {
    return (w[c] >> (4 * j)) & 15u;
  } else if constexpr (BITS == 2) {
    return (w[c >> 1] >> (2 * (8 * (c & 1) + j))) & 3u;
  } else if constexpr (BITS == 8) {
    return (w[2 * c + (j >> 2)] >> (8 * (j & 3))) & 255u;
  } else {
    return code3(w[0], w[1], w[2], 8 * c + j);
  }
}

// ------------------------------------------------------------------------------ dequant
// Per-group constants of one column: the exact-unpack constants of DiffPairs, the fp16 scale in
// both halves of a word, the scale as fp32 and the runtime zero.
template <int BITS>
struct ColConsts {
  uint32_t kz[DiffPairs<__half, BITS>::kConsts];
  uint32_t s2;
  float s;
  int z;
  __device__ __forceinline__ void set(float sc, uint16_t sbits, int zero) {
    s = sc;
    z = zero;
    s2 = static_cast<uint32_t>(sbits) | (static_cast<uint32_t>(sbits) << 16);
    DiffPairs<__half, BITS>::consts(zero, kz);
  }
};

// 3-bit: the pair (of DiffPairs<__half, 3>) holding code k of a unit, and which half of it.
__host__ __device__ constexpr int pair_of_k3(int k) {
  for (int p = 0; p < 16; ++p)
    if (code3_pair(p, 0) == k || code3_pair(p, 1) == k) return p;
  return 0;
}
__host__ __device__ constexpr int half_of_k3(int k) {
  for (int p = 0; p < 16; ++p)
    if (code3_pair(p, 1) == k) return 1;
  return 0;
}

// One 3-bit unit (32 consecutive k of one column, words w0..w2) as four 16-byte chunks of
// RN((q - z) s): the exact (q - z) pairs of DiffPairs (its own pairing of the 32 codes), one HMUL2
// per pair, then each output word (k = 2i, 2i + 1) gathered from its two pairs' halves by one
// byte permute.
template <bool PERMA>
__device__ __forceinline__ void dq_unit3(uint32_t w0, uint32_t w1, uint32_t w2, const ColConsts<3>& cc,
                                         uint4 (&out)[4]) {
  uint32_t d[16];
  DiffPairs<__half, 3>::run3(w0, w1, w2, cc.kz, d);
#pragma unroll
  for (int p = 0; p < 16; ++p) d[p] = hmul2(d[p], cc.s2);
  if constexpr (PERMA) {
#pragma unroll
    for (int c = 0; c < 4; ++c) out[c] = make_uint4(d[4 * c], d[4 * c + 1], d[4 * c + 2], d[4 * c + 3]);
    return;
  }
#pragma unroll
  for (int i = 0; i < 16; ++i) {
    const int ka = 2 * i, kb = 2 * i + 1;
    const uint32_t sel = static_cast<uint32_t>(2 * half_of_k3(ka)) | static_cast<uint32_t>(2 * half_of_k3(ka) + 1) << 4 |
                         static_cast<uint32_t>(4 + 2 * half_of_k3(kb)) << 8 |
                         static_cast<uint32_t>(5 + 2 * half_of_k3(kb)) << 12;
    (&out[i >> 2].x)[i & 3] = __byte_perm(d[pair_of_k3(ka)], d[pair_of_k3(kb)], sel);
  }
}

// The k order of the dequantized pairs.  Each width's exact-pair unpack yields (q - z) pairs whose
// two k are not adjacent; writing them to the B tile in natural k order costs one byte permute per
// word.  With bf16 activations the fp16 copy of A is written anyway (k_rows_to_f16), so it can take
// the pairs' order instead: inside each block of `span` k, position j of the tile (and of the copy
// of A) holds k = a_src<BITS>(j).  The contraction does not depend on the order of k, only on A
// and B agreeing.  BITS 0: natural order.
template <int BITS>
__host__ __device__ constexpr int a_span() { return BITS == 3 ? 32 : BITS == 2 ? 16 : 8; }
template <int BITS>
__host__ __device__ constexpr int a_src(int j) {
  if constexpr (BITS == 4) {
    return (j & ~7) + ((j & 7) >> 1) + 4 * (j & 1);      // pairs (p, p + 4)
  } else if constexpr (BITS == 2) {
    return (j & ~15) + ((j & 15) >> 1) + 8 * (j & 1);    // pairs (p, p + 8)
  } else if constexpr (BITS == 8) {
    return (j & ~3) + ((j & 3) == 1 ? 2 : (j & 3) == 2 ? 1 : (j & 3));   // pairs (0, 2), (1, 3)
  } else if constexpr (BITS == 3) {
    return (j & 1) ? code3_pair(j >> 1, 1) : code3_pair(j >> 1, 0);
  } else {
    return j;
  }
}

// One 16-byte chunk (8 consecutive k of one column) for 4-bit: word w.
template <bool PERMA>
__device__ __forceinline__ uint4 dq_chunk4(uint32_t w, const ColConsts<4>& cc) {
  uint32_t d[4], e[4];
  DiffPairs<__half, 4>::run(w, cc.kz, d);                // d[p] = (k p, k p+4) - z, exact
#pragma unroll
  for (int p = 0; p < 4; ++p) e[p] = hmul2(d[p], cc.s2); // one rounding: RN((q - z) s)
  if constexpr (PERMA) return make_uint4(e[0], e[1], e[2], e[3]);
  return make_uint4(__byte_perm(e[0], e[1], 0x5410), __byte_perm(e[2], e[3], 0x5410),
                    __byte_perm(e[0], e[1], 0x7632), __byte_perm(e[2], e[3], 0x7632));
}

// Two chunks (16 consecutive k of one column) for 2-bit: word w.
template <bool PERMA>
__device__ __forceinline__ void dq_chunks2(uint32_t w, const ColConsts<2>& cc, uint4& lo, uint4& hi) {
  uint32_t d[8], e[8];
  DiffPairs<__half, 2>::run(w, cc.kz, d);                // d[p] = (k p, k p+8) - z
#pragma unroll
  for (int p = 0; p < 8; ++p) e[p] = hmul2(d[p], cc.s2);
  if constexpr (PERMA) {
    lo = make_uint4(e[0], e[1], e[2], e[3]);
    hi = make_uint4(e[4], e[5], e[6], e[7]);
    return;
  }
  lo = make_uint4(__byte_perm(e[0], e[1], 0x5410), __byte_perm(e[2], e[3], 0x5410),
                  __byte_perm(e[4], e[5], 0x5410), __byte_perm(e[6], e[7], 0x5410));
  hi = make_uint4(__byte_perm(e[0], e[1], 0x7632), __byte_perm(e[2], e[3], 0x7632),
                  __byte_perm(e[4], e[5], 0x7632), __byte_perm(e[6], e[7], 0x7632));
}

// One chunk for 8-bit: words w0 (k 0..3) and w1 (k 4..7).
template <bool PERMA>
__device__ __forceinline__ uint4 dq_chunk8(uint32_t w0, uint32_t w1, const ColConsts<8>& cc) {
  uint32_t d0[2], d1[2];
  DiffPairs<__half, 8>::run(w0, cc.kz, d0);              // (k0, k2), (k1, k3) - z
  DiffPairs<__half, 8>::run(w1, cc.kz, d1);
  const uint32_t a0 = hmul2(d0[0], cc.s2), a1 = hmul2(d0[1], cc.s2);
  const uint32_t b0 = hmul2(d1[0], cc.s2), b1 = hmul2(d1[1], cc.s2);
  if constexpr (PERMA) return make_uint4(a0, a1, b0, b1);
  return make_uint4(__byte_perm(a0, a1, 0x5410), __byte_perm(a0, a1, 0x7632),
                    __byte_perm(b0, b1, 0x5410), __byte_perm(b0, b1, 0x7632));
}

// bf16 activations for the fp16 multiply: out[m][k] = fp16(A[m][k] * 2^-e_m), row_scale[m] = 2^e_m,
// with max_k |A[m][k]| * 2^-e_m in [2^15, 2^16) -- below fp16's largest finite value for any bf16
// significand.  Multiplying by a power of two is exact, and so is the conversion for every value in
// fp16's normal range; values more than 2^29 below the row's largest round (their products are far
// below the GEMM's absolute tolerance).  One CTA per row at a time, 16-byte loads and stores.  With
// perm (act-order rows sorted by group) the output column k takes A[m][perm[k]] (the row maximum
// does not depend on the order); with PB (a width) the columns of each block of a_span<PB>() are
// written in the order a_src<PB> of that width's dequantized pairs.  run_flag as in Args.
template <int PB>
__global__ void __launch_bounds__(256) k_rows_to_f16(const uint16_t* __restrict__ A, int M, int K,
                                                     const int32_t* __restrict__ perm,
                                                     const int* run_flag, int run_when,
                                                     uint16_t* __restrict__ out, float* __restrict__ row_scale) {
  if (run_flag != nullptr && *run_flag != run_when) return;
  __shared__ uint32_t warp_max[8];
  for (int m = blockIdx.x; m < M; m += gridDim.x) {
    const uint4* row = reinterpret_cast<const uint4*>(A + static_cast<long long>(m) * K);
    uint4* orow = reinterpret_cast<uint4*>(out + static_cast<long long>(m) * K);
    const int nv = K / 8;
    uint32_t mx = 0u;
    for (int i = threadIdx.x; i < nv; i += blockDim.x) {
      const uint4 v = __ldg(row + i);
#pragma unroll
      for (int j = 0; j < 4; ++j) {
        const uint32_t x = (&v.x)[j];
        mx = max(mx, max(x & 0x7FFFu, (x >> 16) & 0x7FFFu));
      }
    }
    mx = __reduce_max_sync(0xFFFFFFFFu, mx);
    if ((threadIdx.x & 31) == 0) warp_max[threadIdx.x >> 5] = mx;
    __syncthreads();
    mx = 0u;
#pragma unroll
    for (int w = 0; w < 8; ++w) mx = max(mx, warp_max[w]);
    int e = mx ? static_cast<int>(mx >> 7) - 127 - 15 : 0;   // exponent field of max|a|, minus 15
    e = e < -126 ? -126 : (e > 126 ? 126 : e);               // 2^e and 2^-e stay normal floats
    const float inv = __uint_as_float(static_cast<uint32_t>(127 - e) << 23);
    constexpr int kSpan = PB == 0 ? 8 : a_span<PB>();      // columns per block
    constexpr int kV = kSpan / 8;                           // 16-byte pieces per block
    for (int b = threadIdx.x; b < K / kSpan; b += blockDim.x) {
      uint32_t h[kSpan];                                    // the block's bf16 values, in k order
      if (perm == nullptr) {
#pragma unroll
        for (int v = 0; v < kV; ++v) {
          const uint4 x = __ldg(row + b * kV + v);
#pragma unroll
          for (int j = 0; j < 4; ++j) {
            h[8 * v + 2 * j] = (&x.x)[j] & 0xFFFFu;
            h[8 * v + 2 * j + 1] = (&x.x)[j] >> 16;
          }
        }
      } else {
        const uint16_t* r16 = A + static_cast<long long>(m) * K;
#pragma unroll
        for (int j = 0; j < kSpan; ++j) {
          int src = __ldg(perm + b * kSpan + j);
          src = src < 0 ? 0 : (src >= K ? K - 1 : src);   // a bad entry never reads outside the row
          h[j] = __ldg(r16 + src);
        }
      }
#pragma unroll
      for (int v = 0; v < kV; ++v) {
        uint4 o;
#pragma unroll
        for (int j = 0; j < 4; ++j) {
          const int j0 = 8 * v + 2 * j;
          const uint32_t lo = h[PB == 0 ? j0 : a_src<PB>(j0)], hi = h[PB == 0 ? j0 + 1 : a_src<PB>(j0 + 1)];
          (&o.x)[j] = pack2(__uint_as_float(lo << 16) * inv, __uint_as_float(hi << 16) * inv, __half());
        }
        orow[b * kV + v] = o;
      }
    }
    if (threadIdx.x == 0) row_scale[m] = __uint_as_float(static_cast<uint32_t>(e + 127) << 23);
    __syncthreads();                                       // warp_max is reused by the next row
  }
}

// TOUT: the output (and activation) type; the multiply is fp16 x fp16 for both.  PERMA: the fp16
// copy of A is in the pairs' k order (a_src), and so are the B tiles.
template <int BITS, typename TOUT, bool PERK, bool PERMA>
__global__ void __launch_bounds__(kThreads, 1)
    k_prefill(const __grid_constant__ CUtensorMap tmA, const __grid_constant__ CUtensorMap tmW,
              const Args a) {
  using Gm = Geo<BITS>;
  constexpr int kStages = Gm::kStages;
  constexpr int kBStages = Gm::kBStages;
  extern __shared__ unsigned char smem_raw[];
  if (a.run_flag != nullptr && *a.run_flag != a.run_when) return;   // flag-gated launch: not this one
  unsigned char* smem = reinterpret_cast<unsigned char*>(
      (reinterpret_cast<uintptr_t>(smem_raw) + 1023) & ~static_cast<uintptr_t>(1023));
  const uint32_t sbase = ptx::smem_addr(smem);
  const int warp = threadIdx.x >> 5, lane = threadIdx.x & 31;

  const uint32_t bar0 = sbase + Gm::kOffBar;
  auto full = [&](int s) { return bar0 + 8u * s; };
  auto empty = [&](int s) { return bar0 + 8u * (kStages + s); };
  auto bfull = [&](int s) { return bar0 + 8u * (2 * kStages + s); };
  auto bempty = [&](int s) { return bar0 + 8u * (2 * kStages + kBStages + s); };
  const uint32_t acc_full = bar0 + 8u * (2 * kStages + 2 * kBStages);
  const uint32_t acc_empty = acc_full + 8u;
  const uint32_t drain = acc_full + 16u;
  uint32_t* tmem_slot = reinterpret_cast<uint32_t*>(smem + Gm::kOffMisc);
  volatile int* abort_flag = reinterpret_cast<volatile int*>(smem + Gm::kOffMisc + 4);

  if (threadIdx.x == 0) {
    for (int s = 0; s < kStages; ++s) {
      ptx::mbar_init(full(s), 1);
      ptx::mbar_init(empty(s), 1 + kDqWarps);
    }
    for (int s = 0; s < kBStages; ++s) {
      ptx::mbar_init(bfull(s), kDqWarps * 32);
      ptx::mbar_init(bempty(s), 1);
    }
    ptx::mbar_init(acc_full, 1);
    ptx::mbar_init(acc_empty, kEpiWarps);
    ptx::mbar_init(drain, 1);
    *abort_flag = 0;
    ptx::fence_mbar_init();
  }
  if (warp == kProducerWarp && lane == 0) {
    ptx::prefetch_tmap(&tmA);
    ptx::prefetch_tmap(&tmW);
  }
  if (warp == kMmaWarp) {
    ptx::tmem_alloc(ptx::smem_addr(tmem_slot), kTmemCols);
    ptx::tmem_relinquish();
  }
  ptx::tc_fence_before();
  __syncthreads();
  ptx::tc_fence_after();
  const uint32_t tmem = *tmem_slot;
  const Sync sy{sbase, abort_flag, a.status};

  const int num_m = (a.M + kBM - 1) / kBM;
  const int num_n = (a.N + kBN - 1) / kBN;
  const int num_tiles = num_m * num_n;
  const int ksteps = (a.K + kBK - 1) / kBK;

  if (warp == kProducerWarp) {
    // ---------------------------------------------------------------- TMA producer
    if (lane == 0) {
      int s = 0;
      uint32_t ph = 0;
      uint32_t issued = 0, last_par[kStages] = {};
      bool ok = true;
      for (int t = blockIdx.x; ok && t < num_tiles; t += gridDim.x) {
        const int mt = t % num_m, nt = t / num_m;
        for (int ks = 0; ks < ksteps; ++ks) {
          if (!wait_bar(sy, empty(s), ph ^ 1u)) { ok = false; break; }
          ptx::mbar_arrive_expect_tx(full(s), kATileBytes + Gm::kWBytes);
          ptx::tma_load_2d(sbase + s * kATileBytes, &tmA, ks * kBK, mt * kBM, full(s));
          ptx::tma_load_2d(sbase + Gm::kOffW + s * Gm::kWBytes, &tmW, nt * kBN, ks * Gm::kRows,
                           full(s));
          issued |= 1u << s;
          last_par[s] = ph;
          if (++s == kStages) { s = 0; ph ^= 1u; }
        }
      }
      if (!ok) {
        // let the copies already issued land before the CTA's shared memory goes away
        const uint64_t t0 = ptx::globaltimer();
        for (int i = 0; i < kStages; ++i)
          if (issued & (1u << i))
            while (!ptx::mbar_try_wait(full(i), last_par[i]) && ptx::globaltimer() - t0 < kWaitLimitNs) {}
      }
    }
  } else if (warp == kMmaWarp) {
    // ---------------------------------------------------------------- MMA issuer
    if (lane == 0) {
      constexpr uint32_t idesc =
          ptx::umma_idesc_f16(0u, 128u, static_cast<uint32_t>(kBN));   // fp16 x fp16
      int s = 0, sb = 0;
      uint32_t ph = 0, phb = 0, aph = 0;
      bool ok = true;
      for (int t = blockIdx.x; ok && t < num_tiles; t += gridDim.x) {
        if (!wait_bar(sy, acc_empty, aph ^ 1u)) { ok = false; break; }
        ptx::tc_fence_after();
        for (int ks = 0; ks < ksteps; ++ks) {
          if (!wait_bar(sy, full(s), ph) || !wait_bar(sy, bfull(sb), phb)) { ok = false; break; }
          ptx::tc_fence_after();
          const uint32_t a_addr = sbase + s * kATileBytes;
          const uint32_t b_addr = sbase + Gm::kOffB + sb * kBTileBytes;
#pragma unroll
          for (int kk = 0; kk < kBK / 16; ++kk) {
            const uint64_t bd = ptx::umma_desc_sw128_kmajor(b_addr + kk * 32);
            const uint32_t acc = (ks | kk) != 0;
            ptx::umma_f16(tmem, ptx::umma_desc_sw128_kmajor(a_addr + kk * 32), bd, idesc, acc);
            ptx::umma_f16(tmem + 256, ptx::umma_desc_sw128_kmajor(a_addr + 128 * 128 + kk * 32), bd,
                          idesc, acc);
          }
          ptx::umma_commit(empty(s));
          ptx::umma_commit(bempty(sb));
          if (++s == kStages) { s = 0; ph ^= 1u; }
          if (++sb == kBStages) { sb = 0; phb ^= 1u; }
        }
        if (!ok) break;
        ptx::umma_commit(acc_full);
        aph ^= 1u;
      }
      if (!ok) {
        // wait (bounded) for the MMAs already issued before TMEM is released
        ptx::umma_commit(drain);
        const uint64_t t0 = ptx::globaltimer();
        while (!ptx::mbar_try_wait(drain, 0) && ptx::globaltimer() - t0 < kWaitLimitNs) {}
      }
    }
  } else if (warp >= kDqWarp0) {
    // ---------------------------------------------------------------- dequantizers
    // Two threads per tile column: thread (col, hf) dequantizes chunks 4 hf .. 4 hf + 3 of
    // column col (k = 32 hf .. 32 hf + 31 of the k-step), i.e. words hf R/2 .. hf R/2 + R/2 - 1.
    constexpr int kHalfRows = Gm::kRows / 2;
    const int dq = threadIdx.x - kDqWarp0 * 32;
    const int col = dq % kBN;
    const int hf = dq / kBN;
    const bool group32 = a.group % 32 == 0;   // one group over each thread's 32 k of a k-step
    int s = 0, sb = 0;
    uint32_t ph = 0, phb = 0;
    bool ok = true;
    for (int t = blockIdx.x; ok && t < num_tiles; t += gridDim.x) {
      const int nt = t / num_m;
      const int n = nt * kBN + col;
      const bool n_ok = n < a.N;
      const int nc = n_ok ? n : a.N - 1;      // clamped column for scale/zero reads
      int gnext = 0;                          // first k of the next group (fast path)
      int pf_g = -1;                          // group whose scale/zero are prefetched (starts at gnext)
      uint16_t pf_s = 0;
      uint2 pf_z = make_uint2(0u, 0u);
      ColConsts<BITS> cc;
      // the column's scale and zero field in group 0; group g is g rows further
      const __half* s_col = a.scales + nc;
      const int zbit = BITS * nc;
      const int32_t* z_col = a.qzeros + (zbit >> 5);
      const int zsh = zbit & 31;
      for (int ks = 0; ks < ksteps; ++ks) {
        if (!wait_bar(sy, full(s), ph)) { ok = false; break; }
        uint32_t wl[kHalfRows];
        const uint32_t* wt = reinterpret_cast<const uint32_t*>(smem + Gm::kOffW + s * Gm::kWBytes);
#pragma unroll
        for (int r = 0; r < kHalfRows; ++r) wl[r] = wt[(hf * kHalfRows + r) * kBN + col];
        __syncwarp();
        if (lane == 0) ptx::mbar_arrive(empty(s));
        if (!wait_bar(sy, bempty(sb), phb ^ 1u)) { ok = false; break; }
        unsigned char* bt = smem + Gm::kOffB + sb * kBTileBytes;
        const int kst = ks * kBK + 32 * hf;     // first k of this thread's half of the k-step
        if constexpr (!PERK) {
          // One group per 16 k at least (fast-path condition), tracked without division.  The
          // next group's scale and zero word are prefetched into registers one group ahead so
          // that no global load sits on the dequant critical path.
          auto load_group = [&](int g) {
            pf_s = __half_as_ushort(__ldg(s_col + static_cast<long long>(g) * a.N));
            const int32_t* zp = z_col + static_cast<long long>(g) * a.zwords;
            pf_z.x = static_cast<uint32_t>(__ldg(zp));
            if constexpr (BITS == 3) pf_z.y = zsh + 3 > 32 ? static_cast<uint32_t>(__ldg(zp + 1)) : 0u;
          };
          auto group_at = [&](int k) {
            if (k >= gnext) {
              int g = pf_g;                              // the prefetched group starts at gnext
              if (g < 0 || k >= gnext + a.group) {       // first group of the tile: load now
                g = k / a.group;
                load_group(g);
              }
              gnext = (g + 1) * a.group;
              uint32_t zf = pf_z.x >> zsh;
              if constexpr (BITS == 3) zf |= zsh + 3 > 32 ? pf_z.y << (32 - zsh) : 0u;
              cc.set(__half2float(__ushort_as_half(pf_s)), pf_s,
                     static_cast<int>(zf & Pack<BITS>::kMask) + a.zero_offset);
              pf_g = gnext < a.K ? g + 1 : -1;           // prefetch group g + 1
              if (pf_g >= 0) load_group(pf_g);
            }
          };
          if constexpr (BITS == 4) {
#pragma unroll
            for (int c = 0; c < 4; ++c) {
              const int k0 = kst + 8 * c;
              uint4 out = make_uint4(0u, 0u, 0u, 0u);
              if (k0 < a.K) {
                group_at(k0);
                if (n_ok) out = dq_chunk4<PERMA>(wl[c], cc);
              }
              *reinterpret_cast<uint4*>(bt + swz(col, 4 * hf + c)) = out;
            }
          } else if constexpr (BITS == 2) {
#pragma unroll
            for (int i = 0; i < 2; ++i) {
              const int k0 = kst + 16 * i;
              uint4 lo = make_uint4(0u, 0u, 0u, 0u), hi = lo;
              if (k0 < a.K) {
                group_at(k0);
                if (n_ok) dq_chunks2<PERMA>(wl[i], cc, lo, hi);
              }
              *reinterpret_cast<uint4*>(bt + swz(col, 4 * hf + 2 * i)) = lo;
              *reinterpret_cast<uint4*>(bt + swz(col, 4 * hf + 2 * i + 1)) = hi;
            }
          } else if constexpr (BITS == 8) {
#pragma unroll
            for (int c = 0; c < 4; ++c) {
              const int k0 = kst + 8 * c;
              uint4 out = make_uint4(0u, 0u, 0u, 0u);
              if (k0 < a.K) {
                group_at(k0);
                if (n_ok) out = dq_chunk8<PERMA>(wl[2 * c], wl[2 * c + 1], cc);
              }
              *reinterpret_cast<uint4*>(bt + swz(col, 4 * hf + c)) = out;
            }
          } else if (group32 && kst + 32 <= a.K) {
            // 3-bit, the thread's unit inside one group: exact pairs, one rounding each
            uint4 out[4] = {make_uint4(0u, 0u, 0u, 0u), make_uint4(0u, 0u, 0u, 0u), make_uint4(0u, 0u, 0u, 0u),
                            make_uint4(0u, 0u, 0u, 0u)};
            group_at(kst);
            if (n_ok) dq_unit3<PERMA>(wl[0], wl[1], wl[2], cc, out);
#pragma unroll
            for (int c = 0; c < 4; ++c) *reinterpret_cast<uint4*>(bt + swz(col, 4 * hf + c)) = out[c];
          } else {
#pragma unroll
            for (int c = 0; c < 4; ++c) {
              const int k0 = kst + 8 * c;
              uint4 out = make_uint4(0u, 0u, 0u, 0u);
              if (k0 < a.K) {
                group_at(k0);
                if (n_ok) {
                  // (with PERMA the launcher takes this path only for halves past K: a 3-bit
                  // PERMA launch has groups of whole 32-k units)
                  float v[8];
#pragma unroll
                  for (int j = 0; j < 8; ++j) {
                    const int sk = PERMA ? a_src<BITS>(8 * c + j) : 8 * c + j;
                    v[j] = diff_f32(local_code<BITS>(wl, sk >> 3, sk & 7), cc.z) * cc.s;
                  }
                  out = make_uint4(pack2(v[0], v[1], __half()), pack2(v[2], v[3], __half()),
                                   pack2(v[4], v[5], __half()), pack2(v[6], v[7], __half()));
                }
              }
              *reinterpret_cast<uint4*>(bt + swz(col, 4 * hf + c)) = out;
            }
          }
        } else {
#pragma unroll
          for (int c = 0; c < 4; ++c) {
            const int k0 = kst + c * 8;
            uint4 out = make_uint4(0u, 0u, 0u, 0u);
            if (n_ok && k0 < a.K) {
              float v[8];
#pragma unroll
              for (int j = 0; j < 8; ++j) {
                const int sk = PERMA ? a_src<BITS>(8 * c + j) : 8 * c + j;   // k - kst
                const int g = clamp_group<BITS>(a, kst + sk);
                const float sj = __half2float(a.scales[static_cast<long long>(g) * a.N + n]);
                v[j] = diff_f32(local_code<BITS>(wl, sk >> 3, sk & 7), zero_of<BITS>(a, g, n)) * sj;
              }
              out = make_uint4(pack2(v[0], v[1], __half()), pack2(v[2], v[3], __half()),
                               pack2(v[4], v[5], __half()), pack2(v[6], v[7], __half()));
            }
            *reinterpret_cast<uint4*>(bt + swz(col, 4 * hf + c)) = out;
          }
        }
        ptx::fence_proxy_async_smem();
        ptx::mbar_arrive(bfull(sb));
        if (++s == kStages) { s = 0; ph ^= 1u; }
        if (++sb == kBStages) { sb = 0; phb ^= 1u; }
      }
    }
  } else {
    // ---------------------------------------------------------------- epilogue (warps 0-3)
    // Each chunk (32 rows x 32 columns) goes TMEM -> registers (lane = row) -> shared memory ->
    // global: the staging turns 32 rows' 16-byte pieces per store instruction into 8 rows' 64-byte
    // segments.  Chunk v of row r sits at slot v ^ ((r >> 1) & 3), so that both the row-wise
    // writes and the segment-wise reads are free of bank conflicts.
    const int q = warp;   // TMEM lanes 32q .. 32q + 31
    uint32_t aph = 0;
    TOUT* C = static_cast<TOUT*>(a.C);
    uint4* stage = reinterpret_cast<uint4*>(smem + Gm::kOffEpi) + q * 128;
    for (int t = blockIdx.x; t < num_tiles; t += gridDim.x) {
      const int mt = t % num_m, nt = t / num_m;
      if (!wait_bar(sy, acc_full, aph)) break;
      ptx::tc_fence_after();
#pragma unroll 1
      for (int half = 0; half < 2; ++half) {
        const int m = mt * kBM + half * 128 + q * 32 + lane;
        const float rs = (a.row_scale != nullptr && m < a.M) ? a.row_scale[m] : 1.0f;
#pragma unroll 1
        for (int cc = 0; cc < kBN / 32; ++cc) {
          uint32_t r[32];
          ptx::tmem_ld_32x32b_x32(tmem + (static_cast<uint32_t>(q * 32) << 16) + half * 256 + cc * 32, r);
          ptx::tmem_ld_wait();
          const int n0 = nt * kBN + cc * 32;
#pragma unroll
          for (int v = 0; v < 4; ++v) {
            uint4 o;
            o.x = pack2(__uint_as_float(r[8 * v + 0]) * rs, __uint_as_float(r[8 * v + 1]) * rs, TOUT());
            o.y = pack2(__uint_as_float(r[8 * v + 2]) * rs, __uint_as_float(r[8 * v + 3]) * rs, TOUT());
            o.z = pack2(__uint_as_float(r[8 * v + 4]) * rs, __uint_as_float(r[8 * v + 5]) * rs, TOUT());
            o.w = pack2(__uint_as_float(r[8 * v + 6]) * rs, __uint_as_float(r[8 * v + 7]) * rs, TOUT());
            stage[lane * 4 + (v ^ ((lane >> 1) & 3))] = o;
          }
          __syncwarp();
          if (n0 < a.N) {
#pragma unroll
            for (int j = 0; j < 4; ++j) {
              const int row = 8 * j + (lane >> 2), sg = lane & 3;
              const int mr = mt * kBM + half * 128 + q * 32 + row;
              const uint4 val = stage[row * 4 + (sg ^ ((row >> 1) & 3))];
              if (mr < a.M) *reinterpret_cast<uint4*>(C + static_cast<long long>(mr) * a.N + n0 + 8 * sg) = val;
            }
          }
          __syncwarp();
        }
      }
      ptx::tc_fence_before();
      __syncwarp();
      if (lane == 0) ptx::mbar_arrive(acc_empty);
      aph ^= 1u;
    }
  }

  ptx::tc_fence_before();
  __syncthreads();
  if (warp == kMmaWarp) {
    ptx::tc_fence_after();
    ptx::tmem_dealloc(tmem, kTmemCols);
  }
}

// Self-test of the bounded wait: one CTA waits, with the kernels' own wait routine, on an
// mbarrier phase that nothing completes.  The wait must give up after `limit_ns`, raise the abort
// flag and set the timeout bit of the status word; the kernel then returns normally.
__global__ void k_wait_selftest(unsigned* status, uint64_t limit_ns, int* waited_out) {
  __shared__ __align__(8) uint64_t bar;
  __shared__ int abort_flag;
  const uint32_t b = ptx::smem_addr(&bar);
  if (threadIdx.x == 0) {
    ptx::mbar_init(b, 1);
    abort_flag = 0;
    ptx::fence_mbar_init();
  }
  __syncthreads();
  const Sync sy{0u, &abort_flag, status};
  const bool ok = wait_bar(sy, b, 0u, limit_ns);   // no arrival will ever come
  if (threadIdx.x == 0) *waited_out = ok ? 0 : 1;
}

// ------------------------------------------------------------------------------ host side
PFN_cuTensorMapEncodeTiled_v12000 encode_fn() {
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
  return fn;
}

template <int BITS, typename TOUT, bool PERK, bool PERMA>
cudaError_t launch_typed(const Problem& p, const void* A16, const float* row_scale, cudaStream_t stream) {
  using Gm = Geo<BITS>;
  static_assert(Gm::kDynSmem <= 232448, "the layout must fit one CTA's shared memory (227 KB)");
  PFN_cuTensorMapEncodeTiled_v12000 enc = encode_fn();
  if (!enc) return cudaErrorNotSupported;
  CUtensorMap tmA, tmW;
  {
    const cuuint64_t dims[2] = {static_cast<cuuint64_t>(p.K), static_cast<cuuint64_t>(p.M)};
    const cuuint64_t strides[1] = {static_cast<cuuint64_t>(p.K) * 2};
    const cuuint32_t box[2] = {static_cast<cuuint32_t>(kBK), static_cast<cuuint32_t>(kBM)};
    const cuuint32_t estr[2] = {1, 1};
    CUresult r = enc(&tmA, CU_TENSOR_MAP_DATA_TYPE_FLOAT16, 2, const_cast<void*>(A16), dims, strides, box, estr,
                     CU_TENSOR_MAP_INTERLEAVE_NONE, CU_TENSOR_MAP_SWIZZLE_128B,
                     CU_TENSOR_MAP_L2_PROMOTION_L2_256B, CU_TENSOR_MAP_FLOAT_OOB_FILL_NONE);
    if (r != CUDA_SUCCESS) return cudaErrorInvalidValue;
  }
  {
    const cuuint64_t rows = static_cast<cuuint64_t>(p.K) * BITS / 32;
    const cuuint64_t dims[2] = {static_cast<cuuint64_t>(p.N), rows};
    const cuuint64_t strides[1] = {static_cast<cuuint64_t>(p.N) * 4};
    const cuuint32_t box[2] = {static_cast<cuuint32_t>(kBN), static_cast<cuuint32_t>(Gm::kRows)};
    const cuuint32_t estr[2] = {1, 1};
    CUresult r = enc(&tmW, CU_TENSOR_MAP_DATA_TYPE_INT32, 2, const_cast<int32_t*>(p.qweight), dims,
                     strides, box, estr, CU_TENSOR_MAP_INTERLEAVE_NONE, CU_TENSOR_MAP_SWIZZLE_NONE,
                     CU_TENSOR_MAP_L2_PROMOTION_L2_256B, CU_TENSOR_MAP_FLOAT_OOB_FILL_NONE);
    if (r != CUDA_SUCCESS) return cudaErrorInvalidValue;
  }
  Args a;
  a.M = p.M; a.N = p.N; a.K = p.K; a.group = p.group; a.G = p.G; a.zero_offset = p.zero_offset;
  a.zwords = p.N * BITS / 32;
  a.qzeros = p.qzeros;
  a.scales = static_cast<const __half*>(p.scales);
  a.g_idx = p.g_idx;
  a.row_scale = row_scale;
  a.C = p.out;
  a.status = p.status;
  a.run_flag = p.run_flag;
  a.run_when = p.run_when;
  auto kern = k_prefill<BITS, TOUT, PERK, PERMA>;
  static bool attr_set = false;   // per instantiation; the attribute is per function
  if (!attr_set) {
    cudaError_t e = cudaFuncSetAttribute(kern, cudaFuncAttributeMaxDynamicSharedMemorySize,
                                         static_cast<int>(Gm::kDynSmem));
    if (e != cudaSuccess) return e;
    attr_set = true;
  }
  const int tiles = ((p.M + kBM - 1) / kBM) * ((p.N + kBN - 1) / kBN);
  const int grid = tiles < device_info().sm_count ? tiles : device_info().sm_count;
  kern<<<grid, kThreads, Gm::kDynSmem, stream>>>(tmA, tmW, a);
  return cudaGetLastError();
}

// fast path: one group per unpacked word (2-bit words hold 16 k) and per 8-k chunk
template <int BITS>
bool per_k_groups(const Problem& p) {
  return p.g_idx != nullptr || (p.group % (BITS == 2 ? 16 : 8)) != 0;
}

// A in the pairs' k order: possible when the copy of A is written here (bf16), and for 3-bit (whose
// order spans a 32-k unit) when each unit lies in one group or the groups are looked up per k.
template <int BITS>
bool pairs_order(const Problem& p) {
  return p.dtype == 1 && (BITS != 3 || per_k_groups<BITS>(p) || p.group % 32 == 0);
}

template <int BITS, typename TOUT, bool PERMA>
cudaError_t launch_t(const Problem& p, const void* A16, const float* row_scale, cudaStream_t stream) {
  return per_k_groups<BITS>(p) ? launch_typed<BITS, TOUT, true, PERMA>(p, A16, row_scale, stream)
                               : launch_typed<BITS, TOUT, false, PERMA>(p, A16, row_scale, stream);
}

template <int BITS>
cudaError_t launch_bits(const Problem& p, cudaStream_t stream) {
  if (p.dtype == 0 && p.perm == nullptr) return launch_t<BITS, __half, false>(p, p.A, nullptr, stream);
  // bf16, or columns gathered through perm: the fp16 copy of A (and for bf16 the row scales) in
  // the caller's workspace
  const size_t a_bytes = (static_cast<size_t>(p.M) * p.K * 2 + 255) & ~static_cast<size_t>(255);
  if (p.workspace == nullptr || p.workspace_bytes < prefill_workspace_bytes(p.M, p.K)) return cudaErrorInvalidValue;
  uint16_t* A16 = static_cast<uint16_t*>(p.workspace);
  cudaError_t e;
  if (p.dtype == 0) {
    e = launch_gather_cols(p.A, p.perm, p.M, p.K, A16, stream);
    if (e != cudaSuccess) return e;
    return launch_t<BITS, __half, false>(p, A16, nullptr, stream);
  }
  float* row_scale = reinterpret_cast<float*>(static_cast<unsigned char*>(p.workspace) + a_bytes);
  const int blocks = p.M < device_info().sm_count * 8 ? p.M : device_info().sm_count * 8;
  const bool perma = pairs_order<BITS>(p);
  if (perma)
    k_rows_to_f16<BITS><<<blocks, 256, 0, stream>>>(static_cast<const uint16_t*>(p.A), p.M, p.K, p.perm,
                                                     p.run_flag, p.run_when, A16, row_scale);
  else
    k_rows_to_f16<0><<<blocks, 256, 0, stream>>>(static_cast<const uint16_t*>(p.A), p.M, p.K, p.perm,
                                                  p.run_flag, p.run_when, A16, row_scale);
  e = cudaGetLastError();
  if (e != cudaSuccess) return e;
  return perma ? launch_t<BITS, __nv_bfloat16, true>(p, A16, row_scale, stream)
               : launch_t<BITS, __nv_bfloat16, false>(p, A16, row_scale, stream);
}

}  // namespace prefill

cudaError_t launch_wait_selftest(unsigned* status, uint64_t limit_ns, int* flag, cudaStream_t stream) {
  prefill::k_wait_selftest<<<1, 32, 0, stream>>>(status, limit_ns, flag);
  return cudaGetLastError();
}

size_t prefill_workspace_bytes(int M, int K) {
  if (M <= 0 || K <= 0) return 0;
  return ((static_cast<size_t>(M) * K * 2 + 255) & ~static_cast<size_t>(255)) +
         ((static_cast<size_t>(M) * 4 + 255) & ~static_cast<size_t>(255));
}

cudaError_t launch_prefill(const Problem& p, cudaStream_t stream) {
  switch (p.bits) {
    case 2: return prefill::launch_bits<2>(p, stream);
    case 3: return prefill::launch_bits<3>(p, stream);
    case 4: return prefill::launch_bits<4>(p, stream);
    case 8: return prefill::launch_bits<8>(p, stream);
    default: return cudaErrorInvalidValue;
  }
}

}  // namespace gptq
