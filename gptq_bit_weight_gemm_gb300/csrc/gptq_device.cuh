// gptq_device.cuh -- device-side building blocks shared by the GPTQ kernels (sm_103a).
//
// Packed layout (page "增强 vLLM 对 GPTQv2 格式的支持：分析与实现", section
// "调整细节：根据格式选择处理方式", which unpacks 16 two-bit codes from one int32 word): each
// qweight column is an LSB-first bit stream of its K codes, code k at stream bits
// [b*k, b*k + b).  For b in {2, 4, 8} a "unit" is one word holding 32/b consecutive k; for
// b = 3 a unit is three consecutive words holding 32 consecutive k (codes 10 and 21 of the
// unit straddle words).  qzeros rows use the same stream rule along N.
//
// Dequantization is w = (q - zero) * scale with zero = stored + zero_offset (0 for GPTQv2, 1
// for GPTQv1).  q - zero is an integer in [-256, 255] and is produced here exactly, either as a
// 16-bit float (the "magic number" construction: OR the code into the mantissa of a float
// whose unit in the last place is 1, then subtract the magic plus the zero) or as an fp32.
#pragma once

#include <cuda_bf16.h>
#include <cuda_fp16.h>
#include <stdint.h>

#include <type_traits>

namespace gptq {

constexpr unsigned kStatusTimeout = 0x1u;
constexpr unsigned kStatusGidxRange = 0x2u;
constexpr unsigned kStatusExpertRows = 0x8u;   // grouped GEMM: an expert's row range was invalid

template <int BITS>
struct Pack {
  static constexpr int kPerUnit = BITS == 3 ? 32 : 32 / BITS;   // k values per unit
  static constexpr int kRowsPerUnit = BITS == 3 ? 3 : 1;        // qweight rows per unit
  static constexpr uint32_t kMask = (1u << BITS) - 1u;
};

// ------------------------------------------------------------------------------------------
// Loads
// ------------------------------------------------------------------------------------------
// Streaming 16-byte load through the non-coherent path, not kept in L1.
__device__ __forceinline__ uint4 ld_stream_v4(const void* p) {
  uint4 v;
  asm volatile("ld.global.nc.L1::no_allocate.v4.u32 {%0,%1,%2,%3}, [%4];"
               : "=r"(v.x), "=r"(v.y), "=r"(v.z), "=r"(v.w)
               : "l"(p));
  return v;
}

__device__ __forceinline__ uint32_t lop3_and_or(uint32_t a, uint32_t mask, uint32_t magic) {
  uint32_t r;
  // (a & mask) | magic
  asm("lop3.b32 %0, %1, %2, %3, 0xEA;" : "=r"(r) : "r"(a), "r"(mask), "r"(magic));
  return r;
}

// Code j (0..31) of a 3-bit unit whose words are w0, w1, w2 (LSB-first 96-bit stream).
__device__ __forceinline__ uint32_t code3(uint32_t w0, uint32_t w1, uint32_t w2, int j) {
  const int bit = 3 * j;
  if (bit + 3 <= 32) return (w0 >> bit) & 7u;
  if (bit < 32) return __funnelshift_r(w0, w1, bit) & 7u;
  if (bit + 3 <= 64) return (w1 >> (bit - 32)) & 7u;
  if (bit < 64) return __funnelshift_r(w1, w2, bit - 32) & 7u;
  return (w2 >> (bit - 64)) & 7u;
}

// Stored zeros of 4 adjacent columns n0..n0+3 (n0 % 4 == 0) of qzeros row `row` (words),
// returned as a 4 x BITS-bit field: column n0 + c at bits [BITS*c, BITS*c + BITS).
template <int BITS>
__device__ __forceinline__ uint32_t zeros4(const int32_t* __restrict__ row, int n0) {
  if constexpr (BITS == 3) {
    const int bit = 3 * n0;
    const int w = bit >> 5, s = bit & 31;
    uint32_t lo = static_cast<uint32_t>(__ldg(row + w));
    uint32_t hi = (s + 12 > 32) ? static_cast<uint32_t>(__ldg(row + w + 1)) : 0u;
    return __funnelshift_r(lo, hi, s) & 0xFFFu;
  } else {
    const int bit = BITS * n0;
    uint32_t word = static_cast<uint32_t>(__ldg(row + (bit >> 5)));
    return BITS == 8 ? word : (word >> (bit & 31)) & ((1u << (4 * BITS)) - 1u);
  }
}

// ------------------------------------------------------------------------------------------
// 16-bit float traits
// ------------------------------------------------------------------------------------------
template <typename T>
struct F16Traits;

template <>
struct F16Traits<__half> {
  using T2 = __half2;
  __device__ static __forceinline__ float to_f32(__half x) { return __half2float(x); }
  __device__ static __forceinline__ __half from_f32(float x) { return __float2half_rn(x); }
  __device__ static __forceinline__ uint16_t bits(__half x) { return __half_as_ushort(x); }
  __device__ static __forceinline__ __half from_bits(uint16_t b) { return __ushort_as_half(b); }
};

template <>
struct F16Traits<__nv_bfloat16> {
  using T2 = __nv_bfloat162;
  __device__ static __forceinline__ float to_f32(__nv_bfloat16 x) { return __bfloat162float(x); }
  __device__ static __forceinline__ __nv_bfloat16 from_f32(float x) {
    return __float2bfloat16_rn(x);
  }
  __device__ static __forceinline__ uint16_t bits(__nv_bfloat16 x) {
    return __bfloat16_as_ushort(x);
  }
  __device__ static __forceinline__ __nv_bfloat16 from_bits(uint16_t b) { return __ushort_as_bfloat16(b); }
};

__device__ __forceinline__ uint16_t lo16(uint32_t x) { return static_cast<uint16_t>(x & 0xFFFFu); }
__device__ __forceinline__ uint16_t hi16(uint32_t x) { return static_cast<uint16_t>(x >> 16); }

__device__ __forceinline__ uint32_t sub2(uint32_t a, uint32_t b, __half) {
  __half2 r = __hsub2(*reinterpret_cast<__half2*>(&a), *reinterpret_cast<__half2*>(&b));
  return *reinterpret_cast<uint32_t*>(&r);
}
__device__ __forceinline__ uint32_t fma2(uint32_t a, uint32_t b, uint32_t c, __half) {
  __half2 r = __hfma2(*reinterpret_cast<__half2*>(&a), *reinterpret_cast<__half2*>(&b),
                      *reinterpret_cast<__half2*>(&c));
  return *reinterpret_cast<uint32_t*>(&r);
}
__device__ __forceinline__ uint32_t sub2(uint32_t a, uint32_t b, __nv_bfloat16) {
  __nv_bfloat162 r =
      __hsub2(*reinterpret_cast<__nv_bfloat162*>(&a), *reinterpret_cast<__nv_bfloat162*>(&b));
  return *reinterpret_cast<uint32_t*>(&r);
}
__device__ __forceinline__ uint32_t fma2(uint32_t a, uint32_t b, uint32_t c, __nv_bfloat16) {
  __nv_bfloat162 r = __hfma2(*reinterpret_cast<__nv_bfloat162*>(&a),
                             *reinterpret_cast<__nv_bfloat162*>(&b),
                             *reinterpret_cast<__nv_bfloat162*>(&c));
  return *reinterpret_cast<uint32_t*>(&r);
}

__device__ __forceinline__ uint32_t hmul2(uint32_t a, uint32_t b) {
  __half2 r = __hmul2(*reinterpret_cast<__half2*>(&a), *reinterpret_cast<__half2*>(&b));
  return *reinterpret_cast<uint32_t*>(&r);
}

// Pack two fp32 into a 16-bit pair (lo, hi), rounding to nearest-even.
__device__ __forceinline__ uint32_t pack2(float lo, float hi, __half) {
  __half2 r = __floats2half2_rn(lo, hi);
  return *reinterpret_cast<uint32_t*>(&r);
}
__device__ __forceinline__ uint32_t pack2(float lo, float hi, __nv_bfloat16) {
  __nv_bfloat162 r = __floats2bfloat162_rn(lo, hi);
  return *reinterpret_cast<uint32_t*>(&r);
}

// Both halves set to the 16-bit float with bit pattern base + mult * z.  Above a power of two
// 2^e the 16-bit formats step by 2^(e - 10) (fp16) or 2^(e - 7) (bf16), so 2^e + z (or its
// negative) has the pattern bits(2^e) + z * 2^(10 - e) (fp16) while that stays below the next
// power of two; DiffPairs uses this for its per-zero constants, all exact for 0 <= z <= 2^BITS.
__device__ __forceinline__ uint32_t splat_bits(uint32_t base, uint32_t mult, int z) {
  return (base + mult * static_cast<uint32_t>(z)) * 0x00010001u;
}

// ------------------------------------------------------------------------------------------
// Exact (q - zero) pairs from one packed word, as 16-bit floats.
//
// DiffPairs<T, BITS> turns one packed word (three for 3-bit) into kPairs registers of two
// 16-bit values each; pair p holds the codes of k = lo_k(p) (low half) and k = hi_k(p) (high half).
// The code is OR-ed into the mantissa of a magic number M with unit last place (1024 for fp16,
// 128 for bf16); a code sitting `sh` bits up reads as M + 2^sh q, and one sub or fma with a
// per-zero constant (consts(), computed once per group) gives q - zero exactly.  Valid for
// __half with 2, 3, 4 and 8 bits and for __nv_bfloat16 with 2 and 4 bits.
// ------------------------------------------------------------------------------------------
template <typename T, int BITS>
struct DiffPairs;

template <>
struct DiffPairs<__half, 4> {
  static constexpr int kPairs = 4, kConsts = 2;
  __device__ static __forceinline__ int lo_k(int p) { return p; }
  __device__ static __forceinline__ int hi_k(int p) { return p + 4; }
  __device__ static __forceinline__ void consts(int z, uint32_t (&k)[kConsts]) {
    k[0] = splat_bits(0x6400u, 1u, z);     // 1024 + z
    k[1] = splat_bits(0xD400u, 16u, z);    // -(64 + z)
  }
  __device__ static __forceinline__ void run(uint32_t w, const uint32_t (&k)[kConsts],
                                             uint32_t (&d)[kPairs]) {
    const uint32_t M2 = 0x64006400u, inv16 = 0x2C002C00u;
    const uint32_t w8 = w >> 8;
    d[0] = sub2(lop3_and_or(w, 0x000F000Fu, M2), k[0], __half());
    d[1] = fma2(lop3_and_or(w, 0x00F000F0u, M2), inv16, k[1], __half());
    d[2] = sub2(lop3_and_or(w8, 0x000F000Fu, M2), k[0], __half());
    d[3] = fma2(lop3_and_or(w8, 0x00F000F0u, M2), inv16, k[1], __half());
  }
};

template <>
struct DiffPairs<__half, 2> {
  static constexpr int kPairs = 8, kConsts = 4;
  __device__ static __forceinline__ int lo_k(int p) { return p; }
  __device__ static __forceinline__ int hi_k(int p) { return p + 8; }
  __device__ static __forceinline__ void consts(int z, uint32_t (&k)[kConsts]) {
    k[0] = splat_bits(0x6400u, 1u, z);     // 1024 + z
    k[1] = splat_bits(0xDC00u, 4u, z);     // -(256 + z)
    k[2] = splat_bits(0xD400u, 16u, z);    // -(64 + z)
    k[3] = splat_bits(0xCC00u, 64u, z);    // -(16 + z)
  }
  __device__ static __forceinline__ void run(uint32_t w, const uint32_t (&k)[kConsts],
                                             uint32_t (&d)[kPairs]) {
    const uint32_t M2 = 0x64006400u;
    const uint32_t inv4 = 0x34003400u, inv16 = 0x2C002C00u, inv64 = 0x24002400u;
#pragma unroll
    for (int h = 0; h < 2; ++h) {
      const uint32_t x = h ? (w >> 8) : w;
      d[4 * h + 0] = sub2(lop3_and_or(x, 0x00030003u, M2), k[0], __half());
      d[4 * h + 1] = fma2(lop3_and_or(x, 0x000C000Cu, M2), inv4, k[1], __half());
      d[4 * h + 2] = fma2(lop3_and_or(x, 0x00300030u, M2), inv16, k[2], __half());
      d[4 * h + 3] = fma2(lop3_and_or(x, 0x00C000C0u, M2), inv64, k[3], __half());
    }
  }
};

template <>
struct DiffPairs<__half, 8> {
  static constexpr int kPairs = 2, kConsts = 1;
  __device__ static __forceinline__ int lo_k(int p) { return p; }
  __device__ static __forceinline__ int hi_k(int p) { return p + 2; }
  __device__ static __forceinline__ void consts(int z, uint32_t (&k)[kConsts]) {
    k[0] = splat_bits(0x6400u, 1u, z);     // 1024 + z
  }
  __device__ static __forceinline__ void run(uint32_t w, const uint32_t (&k)[kConsts],
                                             uint32_t (&d)[kPairs]) {
    // bytes (0, 2) and (1, 3) under the 0x64 exponent byte
    d[0] = sub2(__byte_perm(w, 0x64646464u, 0x4240u), k[0], __half());
    d[1] = sub2(__byte_perm(w, 0x64646464u, 0x4341u), k[0], __half());
  }
};

template <>
struct DiffPairs<__nv_bfloat16, 4> {
  static constexpr int kPairs = 4, kConsts = 1;
  __device__ static __forceinline__ int lo_k(int p) { return p; }
  __device__ static __forceinline__ int hi_k(int p) { return p + 4; }
  __device__ static __forceinline__ void consts(int z, uint32_t (&k)[kConsts]) {
    k[0] = splat_bits(0x4300u, 1u, z);     // 128 + z
  }
  __device__ static __forceinline__ void run(uint32_t w, const uint32_t (&k)[kConsts],
                                             uint32_t (&d)[kPairs]) {
    const uint32_t M2 = 0x43004300u;
    d[0] = sub2(lop3_and_or(w, 0x000F000Fu, M2), k[0], __nv_bfloat16());
    d[1] = sub2(lop3_and_or(w >> 4, 0x000F000Fu, M2), k[0], __nv_bfloat16());
    d[2] = sub2(lop3_and_or(w >> 8, 0x000F000Fu, M2), k[0], __nv_bfloat16());
    d[3] = sub2(lop3_and_or(w >> 12, 0x000F000Fu, M2), k[0], __nv_bfloat16());
  }
};

template <>
struct DiffPairs<__nv_bfloat16, 2> {
  static constexpr int kPairs = 8, kConsts = 3;
  __device__ static __forceinline__ int lo_k(int p) { return p; }
  __device__ static __forceinline__ int hi_k(int p) { return p + 8; }
  __device__ static __forceinline__ void consts(int z, uint32_t (&k)[kConsts]) {
    k[0] = splat_bits(0x4300u, 1u, z);     // 128 + z
    k[1] = splat_bits(0xC200u, 4u, z);     // -(32 + z)
    k[2] = splat_bits(0xC100u, 16u, z);    // -(8 + z)
  }
  __device__ static __forceinline__ void run(uint32_t w, const uint32_t (&k)[kConsts],
                                             uint32_t (&d)[kPairs]) {
    const uint32_t M2 = 0x43004300u;
    const uint32_t inv4 = 0x3E803E80u, inv16 = 0x3D803D80u;   // 0.25, 0.0625 in bf16
#pragma unroll
    for (int h = 0; h < 2; ++h) {
      const uint32_t x = h ? (w >> 8) : w;
      d[4 * h + 0] = sub2(lop3_and_or(x, 0x00030003u, M2), k[0], __nv_bfloat16());
      d[4 * h + 1] = fma2(lop3_and_or(x, 0x000C000Cu, M2), inv4, k[1], __nv_bfloat16());
      d[4 * h + 2] = fma2(lop3_and_or(x, 0x00300030u, M2), inv16, k[2], __nv_bfloat16());
      d[4 * h + 3] = sub2(lop3_and_or(x >> 6, 0x00030003u, M2), k[0], __nv_bfloat16());
    }
  }
};

// ------------------------------------------------------------------------------------------
// Raw codes as 16-bit floats, zero not subtracted: the 3-bit pairing.
//
// CodePairs<__half, 3>::run3 turns the 3 words of a 3-bit unit into 16 registers of two fp16
// values each, 1024 + 2^shift_lo(p) * q (low half) and 1024 + 2^shift_hi(p) * q (high half) for
// the codes lo_k(p), hi_k(p), with masks only; DiffPairs<__half, 3> then takes the zero out
// exactly.
// ------------------------------------------------------------------------------------------
template <typename T, int BITS>
struct CodePairs;

// 3-bit, fp16: a unit is 32 codes in a 96-bit LSB-first stream of 3 words (code j at bit 3j).
// A pair can be read by one mask when its two codes sit at bits [p, p+3) and [16+p', 16+p'+3)
// (p, p' <= 7: inside the fp16 mantissa) of one 32-bit window of the stream, i.e. a window
// starting at bit s with p = 3 lo - s and p' = 3 hi - s - 16.  This pairing of the 32 codes
// uses 9 windows: the 3 words themselves and 6 shifts (s = 4, 10, 35, 38, 58, 70).
__host__ __device__ constexpr int code3_pair(int p, int which) {   // which: 0 lo, 1 hi, 2 window
  constexpr int t[16][3] = {{0, 6, 0},    {1, 7, 0},    {2, 9, 4},    {3, 8, 4},
                            {4, 11, 10},  {5, 10, 10},  {12, 16, 32}, {13, 17, 32},
                            {14, 18, 35}, {15, 19, 38}, {20, 27, 58}, {21, 26, 58},
                            {22, 28, 64}, {23, 29, 64}, {24, 31, 70}, {25, 30, 70}};
  return t[p][which];
}

template <>
struct CodePairs<__half, 3> {
  static constexpr int kPairs = 16;
  static constexpr float kMagic = 1024.0f;
  __host__ __device__ static constexpr int lo_k(int p) { return code3_pair(p, 0); }
  __host__ __device__ static constexpr int hi_k(int p) { return code3_pair(p, 1); }
  __host__ __device__ static constexpr int shift_lo(int p) { return 3 * lo_k(p) - code3_pair(p, 2); }
  __host__ __device__ static constexpr int shift_hi(int p) { return 3 * hi_k(p) - code3_pair(p, 2) - 16; }
  __device__ static __forceinline__ void run3(uint32_t w0, uint32_t w1, uint32_t w2, uint32_t (&d)[kPairs]) {
    const uint32_t x[9] = {w0,
                           w0 >> 4,
                           __funnelshift_r(w0, w1, 10),
                           w1,
                           w1 >> 3,
                           w1 >> 6,
                           __funnelshift_r(w1, w2, 26),
                           w2,
                           w2 >> 6};
#pragma unroll
    for (int p = 0; p < kPairs; ++p) {
      const int s = code3_pair(p, 2);
      const int xi = s == 0 ? 0 : s == 4 ? 1 : s == 10 ? 2 : s == 32 ? 3 : s == 35 ? 4
                   : s == 38 ? 5 : s == 58 ? 6 : s == 64 ? 7 : 8;
      const uint32_t mask = (7u << shift_lo(p)) | (7u << (16 + shift_hi(p)));
      d[p] = lop3_and_or(x[xi], mask, 0x64006400u);
    }
  }
};

// 3-bit, fp16, exact q - z in the pairing of CodePairs<__half, 3>: one fma per pair turns the
// raw pair (1024 + 2^slo q_lo, 1024 + 2^shi q_hi) into (q_lo, q_hi) -- the product by
// (2^-slo, 2^-shi) and the sum with -(1024 2^-slo, 1024 2^-shi) are exact, so one rounding of an
// exact small integer -- and one sub takes the zero (consts(): z in both halves).
template <>
struct DiffPairs<__half, 3> {
  static constexpr int kPairs = 16, kConsts = 1;
  __host__ __device__ static constexpr int lo_k(int p) { return CodePairs<__half, 3>::lo_k(p); }
  __host__ __device__ static constexpr int hi_k(int p) { return CodePairs<__half, 3>::hi_k(p); }
  __device__ static __forceinline__ void consts(int z, uint32_t (&k)[kConsts]) {
    const uint32_t h = __half_as_ushort(__int2half_rn(z));   // an integer in [0, 8]: exact
    k[0] = h * 0x00010001u;
  }
  __device__ static __forceinline__ void run3(uint32_t w0, uint32_t w1, uint32_t w2,
                                              const uint32_t (&k)[kConsts], uint32_t (&d)[kPairs]) {
    CodePairs<__half, 3>::run3(w0, w1, w2, d);
#pragma unroll
    for (int p = 0; p < kPairs; ++p) {
      constexpr int kExpBias = 15;
      const int slo = CodePairs<__half, 3>::shift_lo(p), shi = CodePairs<__half, 3>::shift_hi(p);
      // fp16 bit patterns of 2^-s and of -1024 * 2^-s (exponent fields 15 - s and 25 - s)
      const uint32_t mult = static_cast<uint32_t>((kExpBias - slo) << 10) |
                            (static_cast<uint32_t>((kExpBias - shi) << 10) << 16);
      const uint32_t neg = (0x8000u | static_cast<uint32_t>((kExpBias + 10 - slo) << 10)) |
                           ((0x8000u | static_cast<uint32_t>((kExpBias + 10 - shi) << 10)) << 16);
      d[p] = sub2(fma2(d[p], mult, neg, __half()), k[0], __half());
    }
  }
};

// Exact q - z as an fp32 (any width): magic 2^23 has ulp 1.
__device__ __forceinline__ float diff_f32(uint32_t code, int z) {
  return __uint_as_float(0x4B000000u | code) - (8388608.0f + static_cast<float>(z));
}

}  // namespace gptq
