// dequant.cu -- standalone dequantization W[k][n] = RN((q - zero) * scale).
//
// The capability of the reconstruct kernel on the page "增强 vLLM 对 GPTQv2 格式的支持：分析
// 与实现" (section "调整细节：根据格式选择处理方式": reconstruct_exllama_2bit_kernel calls
// dequant_2bit_16 on each 32-bit lane of a 128-bit load with zeros[i] + zero_offset), for every
// width, both checkpoint formats and act-order.  The result is bit-exact: q - zero is exact and
// the product is rounded once to the output dtype.
//
// Memory-bound in principle (it writes four times the packed bytes at 4 bits), so the unpack must
// cost few instructions per weight.  The output is written with streaming (evict-first) stores: it
// is written once and not read here (measured 2-9 % faster than default stores).  Each thread owns one packed unit of 8 adjacent columns (two
// 16-byte loads per qweight row) and writes 16 bytes per k, so a warp writes 512 contiguous bytes
// of each output row.  With one group per unit (no act-order, groups of at least a unit) the codes
// become exact fp16 (q - zero) pairs (DiffPairs: a mask into a magic mantissa and one fp16 op per
// pair), then fp16 output: one HMUL2 per pair (an exact product rounded once); bf16 output: the
// pair widened to fp32, one fp32x2 product (exact) and one conversion that rounds once.  Otherwise
// (act-order, or groups smaller than a unit) each weight is formed in fp32: magic-number q - zero,
// one product, one rounding.
#include "gptq_device.cuh"
#include "gptq_internal.h"
#include "sm100_ptx.cuh"

namespace gptq {
namespace {

constexpr int kThreads = 256;
constexpr int kCols = 8;             // columns per thread

struct DqArgs {
  const int32_t* qweight;
  const int32_t* qzeros;
  const __half* scales;
  const int32_t* g_idx;
  int K, N, group, G, zero_offset, zwords, units;
  void* W;
  unsigned* status;
};

// Scales and runtime zeros of columns n0 .. n0 + 7 for group g.
template <int BITS>
__device__ __forceinline__ void load_group8(const DqArgs& a, int g, int n0, uint32_t (&sbits)[kCols / 2],
                                            int (&z)[kCols]) {
  const uint4 sv = __ldg(reinterpret_cast<const uint4*>(a.scales + static_cast<long long>(g) * a.N + n0));
  sbits[0] = sv.x; sbits[1] = sv.y; sbits[2] = sv.z; sbits[3] = sv.w;
  const int32_t* zrow = a.qzeros + static_cast<long long>(g) * a.zwords;
  const uint32_t zlo = zeros4<BITS>(zrow, n0), zhi = zeros4<BITS>(zrow, n0 + 4);
#pragma unroll
  for (int c = 0; c < 4; ++c) {
    z[c] = static_cast<int>((zlo >> (BITS * c)) & Pack<BITS>::kMask) + a.zero_offset;
    z[c + 4] = static_cast<int>((zhi >> (BITS * c)) & Pack<BITS>::kMask) + a.zero_offset;
  }
}

__device__ __forceinline__ float h_lo(uint32_t x) { return __half2float(__ushort_as_half(lo16(x))); }
__device__ __forceinline__ float h_hi(uint32_t x) { return __half2float(__ushort_as_half(hi16(x))); }

// (q - z) * s for the two halves of an exact fp16 pair, as a T pair, rounded once.
template <typename T>
__device__ __forceinline__ uint32_t scale_pair(uint32_t d, uint32_t s2, float s) {
  if constexpr (std::is_same<T, __half>::value) {
    return hmul2(d, s2);
  } else {
    const float2 p = ptx::mul_f32x2(make_float2(h_lo(d), h_hi(d)), make_float2(s, s));
    return pack2(p.x, p.y, __nv_bfloat16());
  }
}

// One unit, one group: exact pairs, then 16-byte row stores.
template <int BITS, typename T>
__device__ __forceinline__ void unit_pairs(const DqArgs& a, const uint32_t (&wv)[Pack<BITS>::kRowsPerUnit][kCols],
                                           int u, int n0, T* W) {
  using DP = DiffPairs<__half, BITS>;
  constexpr int PER = Pack<BITS>::kPerUnit;
  constexpr int NP = DP::kPairs;
  const int g = (u * PER) / a.group;
  uint32_t sbits[kCols / 2];
  int z[kCols];
  load_group8<BITS>(a, g, n0, sbits, z);
  // e[c][p]: column c's pair p, (q - z) * s rounded to T
  uint32_t e[kCols][NP];
#pragma unroll
  for (int c = 0; c < kCols; ++c) {
    uint32_t kz[DP::kConsts];
    DP::consts(z[c], kz);
    if constexpr (BITS == 3)
      DP::run3(wv[0][c], wv[1][c], wv[2][c], kz, e[c]);
    else
      DP::run(wv[0][c], kz, e[c]);
    const uint32_t sb = c & 1 ? (sbits[c >> 1] >> 16) : (sbits[c >> 1] & 0xFFFFu);
    const float s = __half2float(__ushort_as_half(static_cast<uint16_t>(sb)));
#pragma unroll
    for (int p = 0; p < NP; ++p) e[c][p] = scale_pair<T>(e[c][p], sb * 0x00010001u, s);
  }
  // row k = lo_k(p) gathers the low halves of pair p over the 8 columns, row hi_k(p) the high
#pragma unroll
  for (int p = 0; p < NP; ++p) {
    uint4 lo, hi;
#pragma unroll
    for (int i = 0; i < 4; ++i) {
      (&lo.x)[i] = __byte_perm(e[2 * i][p], e[2 * i + 1][p], 0x5410);
      (&hi.x)[i] = __byte_perm(e[2 * i][p], e[2 * i + 1][p], 0x7632);
    }
    const long long k_lo = static_cast<long long>(u) * PER + DP::lo_k(p);
    const long long k_hi = static_cast<long long>(u) * PER + DP::hi_k(p);
    __stcs(reinterpret_cast<uint4*>(W + k_lo * a.N + n0), lo);   // written once: evict first
    __stcs(reinterpret_cast<uint4*>(W + k_hi * a.N + n0), hi);
  }
}

template <int BITS, typename T, bool ACT, bool PAIRS>
__global__ void __launch_bounds__(kThreads) k_dequant(const DqArgs a) {
  using P = Pack<BITS>;
  constexpr int PER = P::kPerUnit;
  constexpr int ROWS = P::kRowsPerUnit;
  const int n8_count = a.N / kCols;
  const long long total = static_cast<long long>(a.units) * n8_count;
  T* W = static_cast<T*>(a.W);
  for (long long idx = static_cast<long long>(blockIdx.x) * kThreads + threadIdx.x; idx < total;
       idx += static_cast<long long>(gridDim.x) * kThreads) {
    const int u = static_cast<int>(idx / n8_count);
    const int n0 = static_cast<int>(idx - static_cast<long long>(u) * n8_count) * kCols;
    uint32_t wv[ROWS][kCols];
#pragma unroll
    for (int r = 0; r < ROWS; ++r) {
      const int32_t* src = a.qweight + (static_cast<long long>(u) * ROWS + r) * a.N + n0;
      const uint4 lo = ld_stream_v4(src), hi = ld_stream_v4(src + 4);
      wv[r][0] = lo.x; wv[r][1] = lo.y; wv[r][2] = lo.z; wv[r][3] = lo.w;
      wv[r][4] = hi.x; wv[r][5] = hi.y; wv[r][6] = hi.z; wv[r][7] = hi.w;
    }
    if constexpr (PAIRS) {
      unit_pairs<BITS, T>(a, wv, u, n0, W);
      continue;
    }
    int cur_g = -1;
    float s[kCols];
    int z[kCols];
#pragma unroll 4
    for (int j = 0; j < PER; ++j) {
      const int k = u * PER + j;
      int g;
      if constexpr (ACT) {
        g = __ldg(a.g_idx + k);
        if (g < 0 || g >= a.G) {
          atomicOr(a.status, kStatusGidxRange);
          g = g < 0 ? 0 : a.G - 1;
        }
      } else {
        g = k / a.group;
      }
      if (g != cur_g) {
        uint32_t sbits[kCols / 2];
        load_group8<BITS>(a, g, n0, sbits, z);
#pragma unroll
        for (int c = 0; c < kCols; ++c)
          s[c] = __half2float(__ushort_as_half(static_cast<uint16_t>(c & 1 ? sbits[c >> 1] >> 16 : sbits[c >> 1] & 0xFFFFu)));
        cur_g = g;
      }
      float w[kCols];
#pragma unroll
      for (int c = 0; c < kCols; ++c) {
        uint32_t code;
        if constexpr (BITS == 3) {
          code = code3(wv[0][c], wv[1][c], wv[2][c], j);
        } else {
          code = (wv[0][c] >> (BITS * j)) & P::kMask;
        }
        w[c] = diff_f32(code, z[c]) * s[c];   // exact
      }
      uint4 out;
      out.x = pack2(w[0], w[1], T());
      out.y = pack2(w[2], w[3], T());
      out.z = pack2(w[4], w[5], T());
      out.w = pack2(w[6], w[7], T());
      __stcs(reinterpret_cast<uint4*>(W + static_cast<long long>(k) * a.N + n0), out);   // written once: evict first
    }
  }
}

template <int BITS, typename T>
cudaError_t launch_typed(const Problem& p, cudaStream_t stream) {
  DqArgs a;
  a.qweight = p.qweight; a.qzeros = p.qzeros;
  a.scales = static_cast<const __half*>(p.scales);
  a.g_idx = p.g_idx; a.K = p.K; a.N = p.N; a.group = p.group; a.G = p.G;
  a.zero_offset = p.zero_offset; a.zwords = p.N * BITS / 32;
  a.units = p.K / Pack<BITS>::kPerUnit;
  a.W = p.out; a.status = p.status;
  const long long total = static_cast<long long>(a.units) * (p.N / kCols);
  const long long need = (total + kThreads - 1) / kThreads;
  const long long cap = static_cast<long long>(device_info().sm_count) * 8;
  const int grid = static_cast<int>(need < cap ? need : cap);
  // one group per unit: the pair path
  const bool pairs = p.g_idx == nullptr && p.group % Pack<BITS>::kPerUnit == 0;
  if (p.g_idx)
    k_dequant<BITS, T, true, false><<<grid, kThreads, 0, stream>>>(a);
  else if (pairs)
    k_dequant<BITS, T, false, true><<<grid, kThreads, 0, stream>>>(a);
  else
    k_dequant<BITS, T, false, false><<<grid, kThreads, 0, stream>>>(a);
  return cudaGetLastError();
}

template <int BITS>
cudaError_t launch_bits(const Problem& p, cudaStream_t stream) {
  return p.dtype == 0 ? launch_typed<BITS, __half>(p, stream)
                      : launch_typed<BITS, __nv_bfloat16>(p, stream);
}

}  // namespace

cudaError_t launch_dequant(const Problem& p, cudaStream_t stream) {
  switch (p.bits) {
    case 2: return launch_bits<2>(p, stream);
    case 3: return launch_bits<3>(p, stream);
    case 4: return launch_bits<4>(p, stream);
    case 8: return launch_bits<8>(p, stream);
    default: return cudaErrorInvalidValue;
  }
}

}  // namespace gptq
