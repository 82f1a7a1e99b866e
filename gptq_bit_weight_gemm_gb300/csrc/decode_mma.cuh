// decode_mma.cuh -- GPTQ GEMM for M <= 32 tokens: TMA-streamed packed weights, unpacked in
// registers and multiplied on the tensor cores (mma.sync m16n8k16, fp16/bf16 in, fp32 accumulate).
//
// The problem is a weight stream (page "增强 vLLM 对 GPTQv2 格式的支持：分析与实现", section
// "调整细节：根据格式选择处理方式", notes gptq_gemm's decode speed as the open item).  Grid:
// clusters of cs CTAs split K over 128-column slabs.  Each CTA issues its whole packed slice
// (or as much as its shared-memory share holds) as TMA boxes at launch, stages its group scales
// and zeros and the activations, then unpacks and multiplies while the boxes land; partial sums
// meet through distributed shared memory in a fixed order.  The multiply is "swap-AB": the
// weights are the 16-row A operand (rows = output columns), the tokens the 8-column B operand,
// so unpacked weights never leave registers.
//
// Fragment mapping (PTX m16n8k16, thread = (g, t) = (lane / 4, lane % 4)): a warp owns 32
// columns; thread (g, t) loads the 4 columns of quad col_quad(g).  Tile 0 maps MMA row g to the
// quad's first column and row g+8 to its second; tile 1 maps them to the third and fourth.  A
// k-tile is 4 packed units: thread t holds unit t.  The K order inside an MMA may be any
// permutation shared by A and B, so MMA j of a unit takes the unpacked pairs 2j and 2j+1 of
// thread t's word as the k-slots (2t, 2t+1) and (2t+8, 2t+9) -- and the activations are staged
// in the same pairing, which makes them exactly the B fragment.
//
//  * FOLD (groups aligned to k-tiles, no act-order, 2/4/8-bit): A = q - zero exactly (magic-
//    number unpack), products exact, a fresh accumulator per group folded with the scale:
//    acc += scale * sum_k a_k (q_k - zero).
//  * FULL (act-order, 3-bit, unaligned groups): A = RN((q - zero) * scale) per weight (exact
//    fp32 product, one rounding), accumulated across groups.
#pragma once

#include <cuda.h>

#include "decode.cuh"
#include "sm100_ptx.cuh"

namespace gptq {
namespace decode {

// Pairing of a unit's codes into the two halves of one register: pair p = (lo_k(p), hi_k(p)).
template <int BITS>
struct MmaPairs {
  static constexpr int kPairs = BITS == 3 ? 16 : 16 / BITS;
  static constexpr int kHalf = Pack<BITS>::kPerUnit / 2;
  __device__ static __forceinline__ int lo_k(int p) { return p; }
  __device__ static __forceinline__ int hi_k(int p) { return p + kHalf; }
};

__device__ __forceinline__ void mma16816(float (&c)[4], uint32_t a0, uint32_t a1, uint32_t a2,
                                         uint32_t a3, uint32_t b0, uint32_t b1, __half) {
  asm volatile(
      "mma.sync.aligned.m16n8k16.row.col.f32.f16.f16.f32 {%0,%1,%2,%3}, {%4,%5,%6,%7}, {%8,%9}, "
      "{%0,%1,%2,%3};"
      : "+f"(c[0]), "+f"(c[1]), "+f"(c[2]), "+f"(c[3])
      : "r"(a0), "r"(a1), "r"(a2), "r"(a3), "r"(b0), "r"(b1));
}
__device__ __forceinline__ void mma16816(float (&c)[4], uint32_t a0, uint32_t a1, uint32_t a2,
                                         uint32_t a3, uint32_t b0, uint32_t b1, __nv_bfloat16) {
  asm volatile(
      "mma.sync.aligned.m16n8k16.row.col.f32.bf16.bf16.f32 {%0,%1,%2,%3}, {%4,%5,%6,%7}, {%8,%9}, "
      "{%0,%1,%2,%3};"
      : "+f"(c[0]), "+f"(c[1]), "+f"(c[2]), "+f"(c[3])
      : "r"(a0), "r"(a1), "r"(a2), "r"(a3), "r"(b0), "r"(b1));
}

// Words of the staged activations for one unit (the M real tokens x NP pairs), padded so that
// the 16-byte loads of a warp's 4 units fall in distinct bank groups.
__host__ __device__ constexpr int unit_words(int M, int NP) {
  return M * NP + ((8 - (M * NP) % 32) + 32) % 32;
}

// Staged weight chunks: the 128 columns of a slab are 4 TMA boxes of 32 columns (128 bytes per
// row), each landing in its own 1024-byte aligned slot with the 128-byte swizzle -- the 16-byte
// piece j of row r sits at piece j ^ (r % 8).  A warp reads its 32 columns from one slot.
constexpr int kBoxCols = 32;
constexpr int kBoxRowBytes = kBoxCols * 4;

// Column quad (of the warp's 8) that MMA row group g covers.  With the swizzle, the 8 lanes of
// a 16-byte load phase (g = 2p, 2p+1; t = 0..3, rows t of a k-tile) then hit 8 distinct pieces.
__host__ __device__ constexpr int col_quad(int g) { return ((g & 1) << 2) | (g >> 1); }

// Launch geometry shared by host and device.
struct TmaGeo {
  int cs;              // CTAs per cluster (K split)
  int tiles_per_cta;   // k-tiles (4 units each) of the largest CTA range
  int chunk_tiles;     // k-tiles per TMA chunk
  int chunk_rows;      // packed rows per chunk
  int slot_bytes;      // one 32-column box of a chunk, rounded up to 1024 bytes
  int chunk_bytes;     // 4 slots
  int nbuf;            // chunk buffers (all chunks in flight when nbuf == chunks)
  int max_groups;      // quantization groups a CTA range can touch (FOLD staging)
};

// Shared memory of one CTA: [alignment pad][weight chunk buffers][activation pairs | partial
// sums (aliased in time)][receive slots][group scales][group zero words][mbarriers, flags].
// Activations, partial sums and receive slots are sized by the real token count M, not by the
// MMA token block.
template <int BITS>
struct TmaSmem {
  static constexpr int kZW = kSlab * BITS / 32;        // zero words of a slab per group
  __host__ __device__ static size_t stage_bytes(const TmaGeo& g, int M) {
    const size_t stage = static_cast<size_t>(g.tiles_per_cta) * 4 * unit_words(M, MmaPairs<BITS>::kPairs) * 4;
    const size_t part = static_cast<size_t>(M) * kSlab * 4;
    return ((stage > part ? stage : part) + 127) & ~static_cast<size_t>(127);
  }
  __host__ __device__ static size_t off_stage(const TmaGeo& g) {
    return static_cast<size_t>(g.nbuf) * g.chunk_bytes;
  }
  __host__ __device__ static size_t off_recv(const TmaGeo& g, int M) { return off_stage(g) + stage_bytes(g, M); }
  __host__ __device__ static size_t off_scales(const TmaGeo& g, int M) {
    return off_recv(g, M) + static_cast<size_t>(M) * kSlab * 4;
  }
  __host__ __device__ static size_t off_zeros(const TmaGeo& g, int M) {
    return off_scales(g, M) + static_cast<size_t>(g.max_groups) * kSlab * 2;
  }
  __host__ __device__ static size_t off_misc(const TmaGeo& g, int M) {
    return off_zeros(g, M) + static_cast<size_t>(g.max_groups) * kZW * 4;
  }
  // bytes past the 1024-aligned base, plus the worst-case alignment pad
  __host__ __device__ static size_t bytes(const TmaGeo& g, int M) {
    return off_misc(g, M) + 8 * 16 + 4 * 17 + 1024;
  }
};

__device__ __forceinline__ bool tma_wait(uint32_t bar, uint32_t parity, volatile int* abort_flag,
                                         unsigned* status) {
  if (ptx::mbar_try_wait(bar, parity)) return true;
  const uint64_t t0 = ptx::globaltimer();
  while (true) {
    if (ptx::mbar_try_wait_hint(bar, parity, 100000u)) return true;
    if (*abort_flag) return false;
    if (ptx::globaltimer() - t0 > 2000000000ull) {
      *abort_flag = 1;
      atomicOr(status, kStatusTimeout);
      return false;
    }
  }
}

template <int BITS, int MT, typename T, bool FOLD>
__global__ void __launch_bounds__(kThreads, (MT <= 8 && BITS != 3 ? 5 : 1))
    k_decode_mma(const __grid_constant__ CUtensorMap tmW, const Args a, const TmaGeo geo) {
  using P = Pack<BITS>;
  using MP = MmaPairs<BITS>;
  using SM = TmaSmem<BITS>;
  constexpr int PER = P::kPerUnit;
  constexpr int ROWS = P::kRowsPerUnit;
  constexpr int NP = MP::kPairs;
  constexpr int NB = MT / 8;                          // token blocks of 8
  constexpr int ZW = SM::kZW;
  const int UW = unit_words(a.M, NP);
  extern __shared__ __align__(128) unsigned char smem_raw[];

  pdl_launch_dependents();
  cluster_arrive_relaxed();
  cg::cluster_group cluster = cg::this_cluster();
  const int cs = static_cast<int>(gridDim.x);
  const int rank = static_cast<int>(blockIdx.x);
  const int n_base = static_cast<int>(blockIdx.y) * kSlab;
  const int warp = threadIdx.x >> 5, lane = threadIdx.x & 31;
  const int gq = lane >> 2, tq = lane & 3;
  const int quad = col_quad(gq);
  const int col0 = warp * 32 + quad * 4;               // first of this thread's 4 columns
  const int n0 = n_base + col0;
  const int n0c = n0 < a.N ? n0 : a.N - 4;

  // CTA range in k-tiles of 4 units (every warp of the CTA covers all of it, 32 columns each)
  const int tiles_total = (a.units + 3) / 4;
  int ct0, ct1;
  split(tiles_total, cs, rank, ct0, ct1);
  const int cu0 = ct0 * 4;
  const int ntile = ct1 - ct0;
  const int nchunk = (ntile + geo.chunk_tiles - 1) / geo.chunk_tiles;

  // 1024-byte aligned base (the swizzled boxes need it); the host adds the pad to the size
  uint8_t* smem = smem_raw + ((1024u - (ptx::smem_addr(smem_raw) & 1023u)) & 1023u);
  uint8_t* sbuf = smem;                                               // weight chunks
  uint32_t* sB = reinterpret_cast<uint32_t*>(smem + SM::off_stage(geo));
  float* recv = reinterpret_cast<float*>(smem + SM::off_recv(geo, a.M));
  uint16_t* sS = reinterpret_cast<uint16_t*>(smem + SM::off_scales(geo, a.M));
  uint32_t* sZ = reinterpret_cast<uint32_t*>(smem + SM::off_zeros(geo, a.M));
  uint8_t* misc = smem + SM::off_misc(geo, a.M);
  const uint32_t bar0 = ptx::smem_addr(misc);
  volatile int* abort_flag = reinterpret_cast<volatile int*>(misc + 8 * 16);

  // Issue the packed slice into shared memory: chunk c of this CTA lands in buffer c % nbuf.
  // The copies read weights only; they are issued before griddepcontrol.wait because global
  // memory (through L2) is coherent for them and the weights are not produced by the kernel
  // this one may overlap with.
  if (threadIdx.x == 0) {
    for (int b = 0; b < geo.nbuf; ++b) ptx::mbar_init(bar0 + 8 * b, 1);
    *abort_flag = 0;
    ptx::fence_mbar_init();
  }
  __syncthreads();
  volatile int* last_issued = abort_flag + 1;          // [nbuf] last chunk issued per buffer
  auto issue = [&](int c) {
    const int b = c % geo.nbuf;
    last_issued[b] = c;
    const uint32_t dst = ptx::smem_addr(sbuf + static_cast<size_t>(b) * geo.chunk_bytes);
    const int row0 = (cu0 + c * geo.chunk_tiles * 4) * ROWS;
    ptx::mbar_arrive_expect_tx(bar0 + 8 * b, static_cast<uint32_t>(4 * geo.chunk_rows * kBoxRowBytes));
#pragma unroll
    for (int w = 0; w < 4; ++w)
      ptx::tma_load_2d(dst + w * geo.slot_bytes, &tmW, n_base + w * kBoxCols, row0, bar0 + 8 * b);
  };
  if (threadIdx.x == 0)
    for (int c = 0; c < nchunk && c < geo.nbuf; ++c) issue(c);

  // Scales and zero words of the groups this range touches (FOLD): staged once, so the loop
  // below reads them from shared memory.  Like the weights they come before griddepcontrol.wait.
  const int g_lo = (cu0 * PER) / a.group;
  if constexpr (FOLD) {
    const int g_end = (ct1 * 4 * PER - 1) / a.group;
    const int ngrp = ntile > 0 ? (g_end < a.G - 1 ? g_end : a.G - 1) - g_lo + 1 : 0;
    for (int i = threadIdx.x; i < ngrp * (kSlab / 4); i += kThreads) {
      const int gi = i >> 5, q = i & 31;
      const int n = n_base + 4 * q;
      uint2 v = make_uint2(0u, 0u);
      if (n < a.N)
        v = __ldg(reinterpret_cast<const uint2*>(a.scales + static_cast<long long>(g_lo + gi) * a.N + n));
      *reinterpret_cast<uint2*>(sS + gi * kSlab + 4 * q) = v;
    }
    for (int i = threadIdx.x; i < ngrp * ZW; i += kThreads) {
      const int gi = i / ZW, w = i - gi * ZW;
      const int wg = n_base * BITS / 32 + w;
      sZ[gi * ZW + w] = wg < a.zwords
                            ? static_cast<uint32_t>(__ldg(a.qzeros + static_cast<long long>(g_lo + gi) * a.zwords + wg))
                            : 0u;
    }
  }
  pdl_wait();

  // Stage activations: sB[u][m][p] = (a[m][k0 + lo_k(p)], a[m][k0 + hi_k(p)]), zero past K or M.
  const uint16_t* A16 = static_cast<const uint16_t*>(a.A);
  const int nunits = ntile * 4;
  stage_pairs<PER, NP>(A16, a.M, a.K, cu0, nunits, a.units,
                       [](int p) { return MP::lo_k(p); }, [](int p) { return MP::hi_k(p); },
                       [&](int uu, int m, int p, uint32_t v) { sB[uu * UW + m * NP + p] = v; });
  __syncthreads();

  float acc[2][NB][4];
#pragma unroll
  for (int t = 0; t < 2; ++t)
#pragma unroll
    for (int nb = 0; nb < NB; ++nb)
#pragma unroll
      for (int i = 0; i < 4; ++i) acc[t][nb][i] = 0.f;

  // B fragments of k-tile kt for this thread: unit tq, tokens 8 nb + gq, pairs 0..NP-1.
  auto load_b = [&](int kt, uint32_t (&bf)[NB][NP]) {
#pragma unroll
    for (int nb = 0; nb < NB; ++nb) {
      if (8 * nb + gq >= a.M) {                         // absent token: zero B column
#pragma unroll
        for (int i = 0; i < NP; ++i) bf[nb][i] = 0u;
        continue;
      }
      const uint32_t* src = sB + (kt * 4 + tq) * UW + (8 * nb + gq) * NP;
      if constexpr (NP % 4 == 0) {
#pragma unroll
        for (int i = 0; i < NP / 4; ++i) {
          const uint4 v = reinterpret_cast<const uint4*>(src)[i];
          bf[nb][4 * i] = v.x; bf[nb][4 * i + 1] = v.y; bf[nb][4 * i + 2] = v.z; bf[nb][4 * i + 3] = v.w;
        }
      } else {
        const uint2 v = reinterpret_cast<const uint2*>(src)[0];
        bf[nb][0] = v.x; bf[nb][1] = v.y;
      }
    }
  };
  // this thread's 16 bytes of packed row r of a chunk buffer
  const uint8_t* wslot = sbuf + warp * geo.slot_bytes;
  auto wrow = [&](const uint8_t* cb, int r) {
    return *reinterpret_cast<const uint4*>(cb + r * kBoxRowBytes + ((quad ^ (r & 7)) << 4));
  };

  if constexpr (FOLD) {
    using DP = DiffPairs<T, BITS>;
    static_assert(DP::kPairs == NP, "pairing must match the activation staging");
    float cg[2][NB][4];
    float s[4];
    uint32_t kz[4][DP::kConsts];
    const int tpg = a.group / (4 * PER);               // k-tiles per group (>= 1 here)
    int gi = 0;                                        // group of the current tile, from g_lo
    int left = tpg - (ct0 % tpg);
    const int zwi = (col0 * BITS) >> 5, zsh = (col0 * BITS) & 31;
    auto set_group = [&]() {
      const uint2 sv = *reinterpret_cast<const uint2*>(sS + gi * kSlab + col0);
      s[0] = __half2float(__ushort_as_half(lo16(sv.x)));
      s[1] = __half2float(__ushort_as_half(hi16(sv.x)));
      s[2] = __half2float(__ushort_as_half(lo16(sv.y)));
      s[3] = __half2float(__ushort_as_half(hi16(sv.y)));
      const uint32_t zf = sZ[gi * ZW + zwi] >> zsh;
#pragma unroll
      for (int c = 0; c < 4; ++c)
        DP::consts(static_cast<int>((zf >> (BITS * c)) & P::kMask) + a.zero_offset, kz[c]);
#pragma unroll
      for (int t = 0; t < 2; ++t)
#pragma unroll
        for (int nb = 0; nb < NB; ++nb)
#pragma unroll
          for (int i = 0; i < 4; ++i) cg[t][nb][i] = 0.f;
    };
    auto fold = [&]() {
#pragma unroll
      for (int t = 0; t < 2; ++t)
#pragma unroll
        for (int nb = 0; nb < NB; ++nb) {
          acc[t][nb][0] = fmaf(s[2 * t], cg[t][nb][0], acc[t][nb][0]);
          acc[t][nb][1] = fmaf(s[2 * t], cg[t][nb][1], acc[t][nb][1]);
          acc[t][nb][2] = fmaf(s[2 * t + 1], cg[t][nb][2], acc[t][nb][2]);
          acc[t][nb][3] = fmaf(s[2 * t + 1], cg[t][nb][3], acc[t][nb][3]);
        }
    };
    if (ntile > 0) set_group();
    for (int c = 0; c < nchunk; ++c) {
      const bool ok = tma_wait(bar0 + 8 * (c % geo.nbuf), (c / geo.nbuf) & 1, abort_flag, a.status);
      const uint8_t* cb = wslot + static_cast<size_t>(c % geo.nbuf) * geo.chunk_bytes;
      const int kt0 = c * geo.chunk_tiles;
      const int kt_end = kt0 + geo.chunk_tiles < ntile ? kt0 + geo.chunk_tiles : ntile;
      for (int kt = kt0; ok && kt < kt_end; ++kt) {
        const uint4 wv = wrow(cb, (kt - kt0) * 4 + tq);
        uint32_t bf[NB][NP];
        load_b(kt, bf);
        uint32_t d[4][NP];
#pragma unroll
        for (int cc = 0; cc < 4; ++cc) DP::run((&wv.x)[cc], kz[cc], d[cc]);
#pragma unroll
        for (int j = 0; j < NP / 2; ++j)
#pragma unroll
          for (int t = 0; t < 2; ++t)
#pragma unroll
            for (int nb = 0; nb < NB; ++nb)
              mma16816(cg[t][nb], d[2 * t][2 * j], d[2 * t + 1][2 * j], d[2 * t][2 * j + 1],
                       d[2 * t + 1][2 * j + 1], bf[nb][2 * j], bf[nb][2 * j + 1], T());
        if (--left == 0) {                              // group boundary (warp-uniform)
          fold();
          left = tpg;
          if (kt + 1 < ntile) {
            ++gi;
            set_group();
          }
        }
      }
      if (c + geo.nbuf < nchunk) {                      // refill this buffer with chunk c + nbuf
        __syncthreads();
        if (threadIdx.x == 0 && !*abort_flag) { ptx::fence_proxy_async_smem(); issue(c + geo.nbuf); }
      }
    }
    if (ntile > 0 && left != tpg) fold();
  } else {
    for (int c = 0; c < nchunk; ++c) {
      const bool ok = tma_wait(bar0 + 8 * (c % geo.nbuf), (c / geo.nbuf) & 1, abort_flag, a.status);
      const uint8_t* cb = wslot + static_cast<size_t>(c % geo.nbuf) * geo.chunk_bytes;
      const int kt0 = c * geo.chunk_tiles;
      const int kt_end = kt0 + geo.chunk_tiles < ntile ? kt0 + geo.chunk_tiles : ntile;
      for (int kt = kt0; ok && kt < kt_end; ++kt) {
        const int rl = ((kt - kt0) * 4 + tq) * ROWS;   // first row of the unit
        uint4 wv[ROWS];
#pragma unroll
        for (int r = 0; r < ROWS; ++r) wv[r] = wrow(cb, rl + r);
        uint32_t bf[NB][NP];
        load_b(kt, bf);
        const int u = cu0 + kt * 4 + tq;
        const int uk = (u < a.units ? u : a.units - 1) * PER;
        // dequantize this unit for 4 columns: w[c][p] = RN((q - z) * s) pairs
        uint32_t w[4][NP];
        float s[4];
        int z[4];
        int cur_g = -1;
#pragma unroll
        for (int p = 0; p < NP; ++p) {
          float v[4][2];
#pragma unroll
          for (int h = 0; h < 2; ++h) {
            const int j = h ? MP::hi_k(p) : MP::lo_k(p);
            const int k = uk + j;
            const int gg = a.g_idx ? checked_group(a, k) : k / a.group;
            if (gg != cur_g) {
              load_sz<BITS>(a, gg, n0c, s, z);
              cur_g = gg;
            }
#pragma unroll
            for (int cc = 0; cc < 4; ++cc) v[cc][h] = diff_f32(unit_code<BITS>(wv, cc, j), z[cc]) * s[cc];
          }
#pragma unroll
          for (int cc = 0; cc < 4; ++cc) w[cc][p] = pack2(v[cc][0], v[cc][1], T());
        }
#pragma unroll
        for (int j = 0; j < NP / 2; ++j)
#pragma unroll
          for (int t = 0; t < 2; ++t)
#pragma unroll
            for (int nb = 0; nb < NB; ++nb)
              mma16816(acc[t][nb], w[2 * t][2 * j], w[2 * t + 1][2 * j], w[2 * t][2 * j + 1],
                       w[2 * t + 1][2 * j + 1], bf[nb][2 * j], bf[nb][2 * j + 1], T());
      }
      if (c + geo.nbuf < nchunk) {
        __syncthreads();
        if (threadIdx.x == 0 && !*abort_flag) { ptx::fence_proxy_async_smem(); issue(c + geo.nbuf); }
      }
    }
  }

  // ---- this CTA's partial sums -> shared memory, then the cluster reduce-scatter
  __syncthreads();                                      // done with the staged activations
  float* part = reinterpret_cast<float*>(sB);           // [M][kSlab], aliases the staging
  // recv ([cs][M][kSlab / cs]) has a region of its own: peers may push into it while this CTA
  // is still reading its staged activations.
  const int Mr = a.M;
#pragma unroll
  for (int t = 0; t < 2; ++t)
#pragma unroll
    for (int nb = 0; nb < NB; ++nb) {
      const int col = col0 + 2 * t;
      const int m = nb * 8 + 2 * tq;
      if (m < Mr) {
        part[m * kSlab + col] = acc[t][nb][0];
        part[m * kSlab + col + 1] = acc[t][nb][2];
      }
      if (m + 1 < Mr) {
        part[(m + 1) * kSlab + col] = acc[t][nb][1];
        part[(m + 1) * kSlab + col + 1] = acc[t][nb][3];
      }
    }
  __syncthreads();
  const int per_rank = kSlab / cs;                      // cs is a power of two
  const int pr_shift = __ffs(per_rank) - 1;
  cluster_wait();
  for (int i = threadIdx.x; i < Mr * kSlab; i += kThreads) {
    const int m = i / kSlab, col = i - m * kSlab;
    const int owner = col >> pr_shift;
    float* dst = cluster.map_shared_rank(recv, owner);
    dst[(rank * Mr + m) * per_rank + (col - owner * per_rank)] = part[i];
  }
  cluster.sync();
  T* C = static_cast<T*>(a.C);
  for (int i = threadIdx.x; i < Mr * per_rank; i += kThreads) {
    const int m = i >> pr_shift, c = i - (m << pr_shift);
    const int n = n_base + rank * per_rank + c;
    if (n < a.N) {
      float v = 0.f;
      for (int q = 0; q < cs; ++q) v += recv[(q * Mr + m) * per_rank + c];
      C[static_cast<long long>(m) * a.N + n] = F16Traits<T>::from_f32(v);
    }
  }
  if (*abort_flag && threadIdx.x == 0) {
    // after a timeout, let every copy already issued land before shared memory is released
    const uint64_t t0 = ptx::globaltimer();
    for (int b = 0; b < nchunk && b < geo.nbuf; ++b) {
      const int last = last_issued[b];
      while (!ptx::mbar_try_wait(bar0 + 8 * b, (last / geo.nbuf) & 1) &&
             ptx::globaltimer() - t0 < 2000000000ull) {}
    }
  }
}

// Chunking of a CTA range: chunks of at most 16 KB whose k-tile count divides the range when it
// can; as many buffers as the shared-memory share of one CTA allows when every CTA of the grid
// is resident at once (one wave), at least 2 -- all of them for the common one-token shapes, so
// the whole slice is in flight from the first cycle.
template <int BITS>
TmaGeo make_geo(int units, int cs, int M, int group, int ctas, int sm_count, int max_per_sm) {
  constexpr int ROWS = Pack<BITS>::kRowsPerUnit;
  constexpr int PER = Pack<BITS>::kPerUnit;
  TmaGeo g;
  g.cs = cs;
  const int tiles_total = (units + 3) / 4;
  g.tiles_per_cta = (tiles_total + cs - 1) / cs;
  const int tile_bytes = 4 * ROWS * kSlab * 4;
  const int tpg = group / (4 * PER);
  g.max_groups = (tpg >= 1 ? (g.tiles_per_cta + tpg - 1) / tpg : g.tiles_per_cta) + 1;
  int per_sm = (ctas + sm_count - 1) / sm_count;
  if (per_sm > max_per_sm) per_sm = max_per_sm;
  if (per_sm < 1) per_sm = 1;
  auto layout = [&](int ct) {
    g.chunk_tiles = ct;
    g.chunk_rows = ct * 4 * ROWS;
    g.slot_bytes = (g.chunk_rows * kBoxRowBytes + 1023) & ~1023;
    g.chunk_bytes = 4 * g.slot_bytes;
    const int chunks = (g.tiles_per_cta + ct - 1) / ct;
    g.nbuf = 0;
    const size_t fixed = TmaSmem<BITS>::bytes(g, M);          // everything but the buffers
    const long long budget = static_cast<long long>(233472 / per_sm) - 1024 - static_cast<long long>(fixed);
    int fit = budget > 0 ? static_cast<int>(budget / g.chunk_bytes) : 0;
    if (fit > 16) fit = 16;
    g.nbuf = chunks < fit ? chunks : fit;
    return chunks;
  };
  int ct = 1;
  for (int d = 1; d * tile_bytes <= 16 * 1024 && d <= g.tiles_per_cta; ++d)
    if (g.tiles_per_cta % d == 0) ct = d;
  int chunks = layout(ct);
  while (g.nbuf < 2 && g.nbuf < chunks && ct > 1) chunks = layout(ct = (ct + 1) / 2);
  if (g.nbuf < 1) g.nbuf = 1;
  if (g.nbuf < 2 && chunks >= 2) g.nbuf = 2;                  // past one wave rather than serial
  return g;
}

template <int BITS, int MT, typename T, bool FOLD>
cudaError_t launch_mma(const Problem& p, int cs, cudaStream_t stream) {
  Args a;
  a.A = p.A; a.M = p.M; a.K = p.K; a.N = p.N;
  a.qweight = p.qweight; a.qzeros = p.qzeros;
  a.scales = static_cast<const __half*>(p.scales);
  a.g_idx = p.g_idx; a.group = p.group; a.G = p.G; a.zero_offset = p.zero_offset;
  a.zwords = p.N * BITS / 32;
  a.units = p.K / Pack<BITS>::kPerUnit;
  a.C = p.out; a.status = p.status;
  const int slabs = (p.N + kSlab - 1) / kSlab;
  constexpr int kMaxPerSm = (MT <= 16 && BITS != 3) ? 5 : 4;   // register-limited residency
  const TmaGeo geo = make_geo<BITS>(a.units, cs, p.M, p.group, slabs * cs, device_info().sm_count, kMaxPerSm);
  CUtensorMap tmW;
  {
    constexpr int ROWS = Pack<BITS>::kRowsPerUnit;
    const cuuint64_t dims[2] = {static_cast<cuuint64_t>(p.N), static_cast<cuuint64_t>(a.units) * ROWS};
    const cuuint64_t strides[1] = {static_cast<cuuint64_t>(p.N) * 4};
    const cuuint32_t box[2] = {static_cast<cuuint32_t>(kBoxCols), static_cast<cuuint32_t>(geo.chunk_rows)};
    const cuuint32_t estr[2] = {1, 1};
    if (!encode_tensor_map(&tmW, CU_TENSOR_MAP_DATA_TYPE_INT32, const_cast<int32_t*>(p.qweight), dims,
                           strides, box, estr, CU_TENSOR_MAP_SWIZZLE_128B))
      return cudaErrorInvalidValue;
  }
  const size_t smem = TmaSmem<BITS>::bytes(geo, p.M);
  auto kern = k_decode_mma<BITS, MT, T, FOLD>;
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
  return cudaLaunchKernelEx(&cfg, kern, tmW, a, geo);
}

}  // namespace decode
}  // namespace gptq
