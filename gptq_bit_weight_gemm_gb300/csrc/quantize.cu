// quantize.cu -- round-to-nearest GPTQ checkpoint writer on the device.
//
// Page "增强 vLLM 对 GPTQv2 格式的支持：分析与实现", section "LLM 的权重量化":
//   scale = (wmax - wmin) / (2^b - 1),  zero = -round(wmin / scale),
//   q = clamp(round(w / scale) + zero);  symmetric: zero = round((2^b - 1) / 2) with
//   scale = 2 max|w| / (2^b - 1);
// section "从 GPTQv1 到 GPTQv2": v1 stores clamp(zero - 1), v2 stores zero.
// Arithmetic is fp32 with correctly rounded division and round-half-to-even; the scale is
// stored as fp16 and zero and q are computed with the stored value.  Three passes:
//   1. per (group, run of columns sharing a qzeros unit): min/max over the group's rows,
//      scale, zero; writes scales and the v2 qzeros words;
//   2. per (qweight unit, 4 columns): codes against the stored scale/zero, packed along K;
//   3. v1 only: every stored zero z becomes clamp(z - 1).
#include "gptq_device.cuh"
#include "gptq_internal.h"

namespace gptq {
namespace {

constexpr int kThreads = 256;
constexpr unsigned kStatusScaleOverflow = 0x4u;

struct QArgs {
  const float* W;
  const int32_t* g_idx;
  int K, N, group, G, sym, zwords;
  int32_t* qweight;
  int32_t* qzeros;
  __half* scales;
  unsigned* status;
};

template <int BITS>
struct ZUnit {   // qzeros packing unit along N
  static constexpr int kCols = BITS == 3 ? 32 : 32 / BITS;
  static constexpr int kWords = BITS == 3 ? 3 : 1;
};

template <int BITS>
__global__ void __launch_bounds__(kThreads) k_quant_params(const QArgs a) {
  constexpr int COLS = ZUnit<BITS>::kCols;
  constexpr int WORDS = ZUnit<BITS>::kWords;
  const int units_n = a.N / COLS;
  const long long total = static_cast<long long>(a.G) * units_n;
  const float maxq = static_cast<float>((1 << BITS) - 1);
  for (long long idx = static_cast<long long>(blockIdx.x) * kThreads + threadIdx.x; idx < total;
       idx += static_cast<long long>(gridDim.x) * kThreads) {
    const int g = static_cast<int>(idx / units_n);
    const int un = static_cast<int>(idx - static_cast<long long>(g) * units_n);
    const int n0 = un * COLS;
    float lo[COLS], hi[COLS];
#pragma unroll
    for (int c = 0; c < COLS; ++c) { lo[c] = __int_as_float(0x7f800000); hi[c] = -lo[c]; }
    const int kb = a.g_idx ? 0 : g * a.group;
    const int ke = a.g_idx ? a.K : kb + a.group;
    for (int k = kb; k < ke; ++k) {
      if (a.g_idx && __ldg(a.g_idx + k) != g) continue;
      const float4* row = reinterpret_cast<const float4*>(a.W + static_cast<long long>(k) * a.N + n0);
#pragma unroll
      for (int v = 0; v < COLS / 4; ++v) {
        const float4 x = __ldg(row + v);
        lo[4 * v] = fminf(lo[4 * v], x.x); hi[4 * v] = fmaxf(hi[4 * v], x.x);
        lo[4 * v + 1] = fminf(lo[4 * v + 1], x.y); hi[4 * v + 1] = fmaxf(hi[4 * v + 1], x.y);
        lo[4 * v + 2] = fminf(lo[4 * v + 2], x.z); hi[4 * v + 2] = fmaxf(hi[4 * v + 2], x.z);
        lo[4 * v + 3] = fminf(lo[4 * v + 3], x.w); hi[4 * v + 3] = fmaxf(hi[4 * v + 3], x.w);
      }
    }
    uint32_t words[WORDS];
#pragma unroll
    for (int w = 0; w < WORDS; ++w) words[w] = 0u;
#pragma unroll
    for (int c = 0; c < COLS; ++c) {
      float s32;
      if (a.sym) {
        const float amax = fmaxf(fabsf(lo[c]), fabsf(hi[c]));
        s32 = __fdiv_rn(2.0f * amax, maxq);
      } else {
        s32 = __fdiv_rn(__fsub_rn(hi[c], lo[c]), maxq);
      }
      uint16_t h = __half_as_ushort(__float2half_rn(s32));
      if ((h & 0x7fffu) == 0) h = 0x3c00u;             // degenerate group: scale 1
      if ((h & 0x7c00u) == 0x7c00u) atomicOr(a.status, kStatusScaleOverflow);
      a.scales[static_cast<long long>(g) * a.N + n0 + c] = __ushort_as_half(h);
      const float s = __half2float(__ushort_as_half(h));
      float z;
      if (a.sym) {
        z = rintf(maxq / 2.0f);
      } else {
        z = -rintf(__fdiv_rn(lo[c], s));
        z = fminf(fmaxf(z, 0.0f), maxq);
      }
      const uint32_t zc = static_cast<uint32_t>(z);
      const int bit = BITS * c;                          // position in this unit's stream
      words[bit >> 5] |= zc << (bit & 31);
      if ((bit & 31) + BITS > 32) words[(bit >> 5) + 1] |= zc >> (32 - (bit & 31));
    }
    int32_t* out = a.qzeros + static_cast<long long>(g) * a.zwords + un * WORDS;
#pragma unroll
    for (int w = 0; w < WORDS; ++w) out[w] = static_cast<int32_t>(words[w]);
  }
}

template <int BITS>
__global__ void __launch_bounds__(kThreads) k_quant_codes(const QArgs a) {
  using P = Pack<BITS>;
  constexpr int PER = P::kPerUnit;
  constexpr int ROWS = P::kRowsPerUnit;
  const float maxq = static_cast<float>((1 << BITS) - 1);
  const int n4_count = a.N / 4;
  const int units = a.K / PER;
  const long long total = static_cast<long long>(units) * n4_count;
  for (long long idx = static_cast<long long>(blockIdx.x) * kThreads + threadIdx.x; idx < total;
       idx += static_cast<long long>(gridDim.x) * kThreads) {
    const int u = static_cast<int>(idx / n4_count);
    const int n0 = static_cast<int>(idx - static_cast<long long>(u) * n4_count) * 4;
    uint32_t words[ROWS][4];
#pragma unroll
    for (int r = 0; r < ROWS; ++r)
#pragma unroll
      for (int c = 0; c < 4; ++c) words[r][c] = 0u;
    int cur_g = -1;
    float s[4], z[4];
    for (int j = 0; j < PER; ++j) {
      const int k = u * PER + j;
      int g = a.g_idx ? __ldg(a.g_idx + k) : k / a.group;
      if (g < 0 || g >= a.G) {
        atomicOr(a.status, kStatusGidxRange);
        g = g < 0 ? 0 : a.G - 1;
      }
      if (g != cur_g) {
        const __half* srow = a.scales + static_cast<long long>(g) * a.N + n0;
        const uint32_t zf = zeros4<BITS>(a.qzeros + static_cast<long long>(g) * a.zwords, n0);
#pragma unroll
        for (int c = 0; c < 4; ++c) {
          s[c] = __half2float(srow[c]);
          z[c] = static_cast<float>((zf >> (BITS * c)) & P::kMask);
        }
        cur_g = g;
      }
      const float4 x = __ldg(reinterpret_cast<const float4*>(a.W + static_cast<long long>(k) * a.N + n0));
      const float xv[4] = {x.x, x.y, x.z, x.w};
      const int bit = BITS * j;                          // position in this unit's stream
#pragma unroll
      for (int c = 0; c < 4; ++c) {
        float v = rintf(__fdiv_rn(xv[c], s[c])) + z[c];
        v = fminf(fmaxf(v, 0.0f), maxq);
        const uint32_t q = static_cast<uint32_t>(v);
        words[(bit >> 5)][c] |= q << (bit & 31);
        if ((bit & 31) + BITS > 32) words[(bit >> 5) + 1][c] |= q >> (32 - (bit & 31));
      }
    }
#pragma unroll
    for (int r = 0; r < ROWS; ++r)
      *reinterpret_cast<uint4*>(a.qweight + (static_cast<long long>(u) * ROWS + r) * a.N + n0) =
          make_uint4(words[r][0], words[r][1], words[r][2], words[r][3]);
  }
}

// v1 storage: every zero field z of qzeros becomes clamp(z - 1, 0, 2^b - 1).
template <int BITS>
__global__ void __launch_bounds__(kThreads) k_zeros_to_v1(int32_t* qzeros, long long units) {
  constexpr int COLS = ZUnit<BITS>::kCols;
  constexpr int WORDS = ZUnit<BITS>::kWords;
  constexpr uint32_t MASK = (1u << BITS) - 1u;
  for (long long i = static_cast<long long>(blockIdx.x) * kThreads + threadIdx.x; i < units;
       i += static_cast<long long>(gridDim.x) * kThreads) {
    uint32_t in[WORDS], out[WORDS];
#pragma unroll
    for (int w = 0; w < WORDS; ++w) { in[w] = static_cast<uint32_t>(qzeros[i * WORDS + w]); out[w] = 0u; }
#pragma unroll
    for (int c = 0; c < COLS; ++c) {
      const int bit = BITS * c;
      uint32_t f = in[bit >> 5] >> (bit & 31);
      if ((bit & 31) + BITS > 32) f |= in[(bit >> 5) + 1] << (32 - (bit & 31));
      f &= MASK;
      const uint32_t v = f > 0 ? f - 1 : 0u;
      out[bit >> 5] |= v << (bit & 31);
      if ((bit & 31) + BITS > 32) out[(bit >> 5) + 1] |= v >> (32 - (bit & 31));
    }
#pragma unroll
    for (int w = 0; w < WORDS; ++w) qzeros[i * WORDS + w] = static_cast<int32_t>(out[w]);
  }
}

// Launched after the writer kernels, without programmatic dependent launch, so it starts only
// when they have completed and their stores are visible.  The GEMM kernels read the checkpoint
// before their own dependency wait (they may start while the kernel before them runs); with
// this kernel in between, a GEMM issued right after gptq_quantize_rtn (or after the device
// prepack, which ends with it too) overlaps only this empty kernel, never the writers.
__global__ void k_writer_fence() {}

int grid_for(long long work) {
  const long long need = (work + kThreads - 1) / kThreads;
  const long long cap = static_cast<long long>(device_info().sm_count) * 8;
  return static_cast<int>(need < 1 ? 1 : (need < cap ? need : cap));
}

template <int BITS>
cudaError_t launch_bits(const QuantProblem& q, cudaStream_t stream) {
  QArgs a;
  a.W = q.W; a.g_idx = q.g_idx; a.K = q.K; a.N = q.N; a.group = q.group; a.G = q.G;
  a.sym = q.sym; a.zwords = q.N * BITS / 32;
  a.qweight = q.qweight; a.qzeros = q.qzeros;
  a.scales = static_cast<__half*>(q.scales);
  a.status = q.status;
  const long long zunits = static_cast<long long>(q.G) * (q.N / ZUnit<BITS>::kCols);
  k_quant_params<BITS><<<grid_for(zunits), kThreads, 0, stream>>>(a);
  cudaError_t e = cudaGetLastError();
  if (e != cudaSuccess) return e;
  const long long cunits = static_cast<long long>(q.K / Pack<BITS>::kPerUnit) * (q.N / 4);
  k_quant_codes<BITS><<<grid_for(cunits), kThreads, 0, stream>>>(a);
  e = cudaGetLastError();
  if (e != cudaSuccess) return e;
  if (q.fmt == 1) {
    k_zeros_to_v1<BITS><<<grid_for(zunits), kThreads, 0, stream>>>(q.qzeros, zunits);
    e = cudaGetLastError();
    if (e != cudaSuccess) return e;
  }
  k_writer_fence<<<1, 32, 0, stream>>>();
  return cudaGetLastError();
}

}  // namespace

cudaError_t launch_quantize(const QuantProblem& q, cudaStream_t stream) {
  switch (q.bits) {
    case 2: return launch_bits<2>(q, stream);
    case 3: return launch_bits<3>(q, stream);
    case 4: return launch_bits<4>(q, stream);
    case 8: return launch_bits<8>(q, stream);
    default: return cudaErrorInvalidValue;
  }
}

cudaError_t launch_writer_fence(cudaStream_t stream) {
  k_writer_fence<<<1, 32, 0, stream>>>();
  return cudaGetLastError();
}

}  // namespace gptq
