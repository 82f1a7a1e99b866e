// dequant.cu -- standalone dequantization W[k][n] = RN((q - zero) * scale).
//
// The capability of the reconstruct kernel on the page "增强 vLLM 对 GPTQv2 格式的支持：分析
// 与实现" (section "调整细节：根据格式选择处理方式": reconstruct_exllama_2bit_kernel calls
// dequant_2bit_16 on each 32-bit lane of a 128-bit load with zeros[i] + zero_offset), for every
// width, both checkpoint formats and act-order.  q - zero is formed exactly in fp32 (magic
// number 2^23), multiplied by the fp16 scale in fp32 (exact: at most 9 + 11 significant bits)
// and rounded once to the output dtype, so the result is bit-exact.
//
// Memory-bound: each thread owns one packed unit of 4 adjacent columns (one 16-byte load per
// qweight row) and writes 8 bytes per k, so a warp writes 256 contiguous bytes per output row.
#include "gptq_device.cuh"
#include "gptq_internal.h"

namespace gptq {
namespace {

constexpr int kThreads = 256;

struct DqArgs {
  const int32_t* qweight;
  const int32_t* qzeros;
  const __half* scales;
  const int32_t* g_idx;
  int K, N, group, G, zero_offset, zwords, units;
  void* W;
  unsigned* status;
};

template <int BITS, typename T, bool ACT>
__global__ void __launch_bounds__(kThreads) k_dequant(const DqArgs a) {
  using P = Pack<BITS>;
  constexpr int PER = P::kPerUnit;
  constexpr int ROWS = P::kRowsPerUnit;
  const int n4_count = a.N / 4;
  const long long total = static_cast<long long>(a.units) * n4_count;
  T* W = static_cast<T*>(a.W);
  for (long long idx = static_cast<long long>(blockIdx.x) * kThreads + threadIdx.x; idx < total;
       idx += static_cast<long long>(gridDim.x) * kThreads) {
    const int u = static_cast<int>(idx / n4_count);
    const int n0 = static_cast<int>(idx - static_cast<long long>(u) * n4_count) * 4;
    uint4 wv[ROWS];
#pragma unroll
    for (int r = 0; r < ROWS; ++r)
      wv[r] = ld_stream_v4(a.qweight + (static_cast<long long>(u) * ROWS + r) * a.N + n0);
    int cur_g = -1;
    float s[4];
    int z[4];
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
        const uint2 sv =
            __ldg(reinterpret_cast<const uint2*>(a.scales + static_cast<long long>(g) * a.N + n0));
        s[0] = __half2float(__ushort_as_half(static_cast<uint16_t>(sv.x & 0xFFFFu)));
        s[1] = __half2float(__ushort_as_half(static_cast<uint16_t>(sv.x >> 16)));
        s[2] = __half2float(__ushort_as_half(static_cast<uint16_t>(sv.y & 0xFFFFu)));
        s[3] = __half2float(__ushort_as_half(static_cast<uint16_t>(sv.y >> 16)));
        const uint32_t zf = zeros4<BITS>(a.qzeros + static_cast<long long>(g) * a.zwords, n0);
#pragma unroll
        for (int c = 0; c < 4; ++c)
          z[c] = static_cast<int>((zf >> (BITS * c)) & P::kMask) + a.zero_offset;
        cur_g = g;
      }
      float w[4];
#pragma unroll
      for (int c = 0; c < 4; ++c) {
        uint32_t code;
        if constexpr (BITS == 3) {
          code = code3((&wv[0].x)[c], (&wv[1].x)[c], (&wv[2].x)[c], j);
        } else {
          code = ((&wv[0].x)[c] >> (BITS * j)) & P::kMask;
        }
        w[c] = diff_f32(code, z[c]) * s[c];   // exact
      }
      uint2 out;
      out.x = pack2(w[0], w[1], T());
      out.y = pack2(w[2], w[3], T());
      *reinterpret_cast<uint2*>(W + static_cast<long long>(k) * a.N + n0) = out;
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
  const long long total = static_cast<long long>(a.units) * (p.N / 4);
  const long long need = (total + kThreads - 1) / kThreads;
  const long long cap = static_cast<long long>(device_info().sm_count) * 8;
  const int grid = static_cast<int>(need < cap ? need : cap);
  if (p.g_idx)
    k_dequant<BITS, T, true><<<grid, kThreads, 0, stream>>>(a);
  else
    k_dequant<BITS, T, false><<<grid, kThreads, 0, stream>>>(a);
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
