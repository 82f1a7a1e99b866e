// dequant.cu -- standalone dequantization W[k][n] = RN((q - zero) * scale).
//
// The capability of the reconstruct kernel on the page "增强 vLLM 对 GPTQv2 格式的支持：分析
// 与实现" (section "调整细节：根据格式选择处理方式": reconstruct_exllama_2bit_kernel calls
// dequant_2bit_16 on each 32-bit lane of a 128-bit load with zeros[i] + zero_offset), for every
// width, both checkpoint formats and act-order.  q - zero is formed exactly in fp32 (magic
// number 2^23), multiplied by the fp16 scale in fp32 (exact: at most 9 + 11 significant bits)
// and rounded once to the output dtype, so the result is bit-exact.
//
// Memory-bound (it writes four times the packed bytes at 4 bits): each thread owns one packed
// unit of 8 adjacent columns (two 16-byte loads per qweight row) and writes 16 bytes per k, so a
// warp writes 512 contiguous bytes of each output row.
#include "gptq_device.cuh"
#include "gptq_internal.h"

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

template <int BITS, typename T, bool ACT>
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
        const uint4 sv = __ldg(reinterpret_cast<const uint4*>(a.scales + static_cast<long long>(g) * a.N + n0));
#pragma unroll
        for (int c = 0; c < kCols; ++c) {
          const uint32_t word = (&sv.x)[c >> 1];
          s[c] = __half2float(__ushort_as_half(static_cast<uint16_t>(c & 1 ? word >> 16 : word & 0xFFFFu)));
        }
        const int32_t* zrow = a.qzeros + static_cast<long long>(g) * a.zwords;
        const uint32_t zlo = zeros4<BITS>(zrow, n0), zhi = zeros4<BITS>(zrow, n0 + 4);
#pragma unroll
        for (int c = 0; c < 4; ++c) {
          z[c] = static_cast<int>((zlo >> (BITS * c)) & P::kMask) + a.zero_offset;
          z[c + 4] = static_cast<int>((zhi >> (BITS * c)) & P::kMask) + a.zero_offset;
        }
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
      *reinterpret_cast<uint4*>(W + static_cast<long long>(k) * a.N + n0) = out;
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
