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
//  * FOLD (groups aligned to k-tiles, no act-order, 2/4/8-bit and fp16 3-bit): A = the exact
//    difference q - zero as a 16-bit float (masks into the mantissa of a magic number, then one
//    sub or fma with a per-group constant, DiffPairs), B = the activations, a fresh fp32
//    accumulator R per group; at the group end acc += scale * R.  A group whose codes all equal
//    its zero contributes exactly 0, whatever the scale and the activations.  Tiles go in blocks
//    of 4 inside one chunk and one group.
//  * FULL (act-order, 3-bit, unaligned groups): A = RN((q - zero) * scale) per weight (exact
//    fp32 product, one rounding), accumulated across groups.
//
// Cost model that shaped it (measured on GB300): a k-tile of 4 packed words per warp costs the
// dispatch of its integer-pipe ops (16 lanes, 2 cycles each), its mma.sync (about 8 cycles per
// m16n8k16 per SM sub-partition) and its fp16 ops, added rather than overlapped; the raw-code
// unpack (4 masks + 1 shift + 4 fp16 sub/fma per 4-bit word) and the per-group constants staged
// in shared memory keep the count per word low.
#pragma once

#include <cuda.h>

#include <atomic>

#include "decode.cuh"
#include "sm100_ptx.cuh"

namespace gptq {
namespace decode {

// Pairing of a unit's codes into the two halves of one register: pair p = (lo_k(p), hi_k(p)).
template <int BITS>
struct MmaPairs {
  static constexpr int kPairs = 16 / BITS;
  static constexpr int kHalf = Pack<BITS>::kPerUnit / 2;
  __device__ static __forceinline__ int lo_k(int p) { return p; }
  __device__ static __forceinline__ int hi_k(int p) { return p + kHalf; }
};
// 3-bit: the pairing under which every pair is one mask of one stream window (CodePairs<half, 3>)
template <>
struct MmaPairs<3> {
  static constexpr int kPairs = 16;
  __device__ static __forceinline__ int lo_k(int p) { return code3_pair(p, 0); }
  __device__ static __forceinline__ int hi_k(int p) { return code3_pair(p, 1); }
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
constexpr size_t kMaxCtaSmem = 227 * 1024;   // dynamic shared memory one CTA may opt into
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
  int full_groups;     // FULL: groups staged in shared memory (all G with g_idx), 0 = read via L1
  int full_k;          // FULL: k values of the largest CTA range (their group indices are staged)
};

// Shared memory of one CTA: [alignment pad][weight chunk buffers][activation pairs | partial
// sums, several tokens (aliased in time)][receive slots][FOLD: per group and column, the scale
// bits and the runtime zero][FULL: per group and column scale and zero, per k its group]
// [mbarriers, flags].
// Activations, partial sums and receive slots are sized by the real token count M, not by the
// MMA token block.
template <int BITS>
struct TmaSmem {
  __host__ __device__ static size_t stage_bytes(const TmaGeo& g, int M) {
    const size_t stage = static_cast<size_t>(g.tiles_per_cta) * 4 * unit_words(M, MmaPairs<BITS>::kPairs) * 4;
    // partial sums of several tokens (one token pushes them from registers)
    const size_t part = M > 1 ? static_cast<size_t>(M) * kSlab * 4 : 0;
    return ((stage > part ? stage : part) + 127) & ~static_cast<size_t>(127);
  }
  __host__ __device__ static size_t off_stage(const TmaGeo& g) {
    return static_cast<size_t>(g.nbuf) * g.chunk_bytes;
  }
  __host__ __device__ static size_t off_recv(const TmaGeo& g, int M) { return off_stage(g) + stage_bytes(g, M); }
  __host__ __device__ static size_t off_gconst(const TmaGeo& g, int M) {
    return off_recv(g, M) + static_cast<size_t>(M) * kSlab * 4;
  }
  __host__ __device__ static size_t off_full(const TmaGeo& g, int M) {
    return off_gconst(g, M) + static_cast<size_t>(g.max_groups) * kSlab * 4;
  }
  // FULL staging: (scale bits | zero << 16) per group and column, then a group index per k
  __host__ __device__ static size_t full_bytes(const TmaGeo& g) {
    return g.full_groups > 0
               ? ((static_cast<size_t>(g.full_groups) * kSlab * 4 + static_cast<size_t>(g.full_k) * 2 + 15) & ~static_cast<size_t>(15))
               : 0;
  }
  __host__ __device__ static size_t off_misc(const TmaGeo& g, int M) {
    return off_full(g, M) + full_bytes(g);
  }
  // bytes past the 1024-aligned base (mbarriers, the abort flag, the issued-chunk record, per
  // token the largest staged magnitude and its power-of-two scale), plus the worst-case
  // alignment pad
  __host__ __device__ static size_t bytes(const TmaGeo& g, int M) {
    return off_misc(g, M) + 8 * kWarps * g.nbuf + 4 * (kWarps * g.nbuf + 1) + 8 * static_cast<size_t>(M) + 1024;
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

// Grouped launches: the expert of grid slot `slot` -- the slot-th expert (in order) whose rows
// [offsets[e], offsets[e + 1]) are non-empty and valid (within [0, rows], at most max_m) -- found
// by each warp on its own, 32 experts per step (a ballot, then the rank-th set bit).  Returns
// {e or -1, offsets[e], offsets[e + 1], 1 if any expert's range is malformed}.  Kept out of line
// so that it does not shape the register allocation of the kernel's main loop.
static __device__ __noinline__ int4 find_expert(const int32_t* offsets, int experts, int rows, int max_m, int slot) {
  const int lane = threadIdx.x & 31;
  int e = -1, o0 = 0, o1 = 0, seen = 0;
  bool bad_any = false;
  for (int base = 0; base < experts; base += 32) {
    const int x = base + lane;
    int b0 = 0, b1 = 0;
    if (x < experts) {
      b0 = offsets[x];
      b1 = offsets[x + 1];
    }
    const bool bad = x < experts && (b0 < 0 || b1 < b0 || b1 > rows || b1 - b0 > max_m);
    const unsigned held = __ballot_sync(0xFFFFFFFFu, x < experts && !bad && b1 > b0);
    bad_any |= __ballot_sync(0xFFFFFFFFu, bad) != 0u;
    const int cnt = __popc(held);
    if (e < 0 && slot < seen + cnt) {
      const int src = static_cast<int>(__fns(held, 0u, slot - seen + 1));
      e = base + src;
      o0 = __shfl_sync(0xFFFFFFFFu, b0, src);
      o1 = __shfl_sync(0xFFFFFFFFu, b1, src);
    }
    seen += cnt;
  }
  return make_int4(e, o0, o1, bad_any ? 1 : 0);
}

template <int BITS, int MT, int MX, typename T, bool FOLD, bool GROUPED = false>
__global__ void __launch_bounds__(kThreads, (MT <= 16 && BITS != 3 ? 5 : 1))
    k_decode_mma(const __grid_constant__ CUtensorMap tmW, const Args args, const TmaGeo geo) {
  using P = Pack<BITS>;
  using MP = MmaPairs<BITS>;
  using SM = TmaSmem<BITS>;
  // The multiply type TC.  The FOLD path with 2- and 4-bit codes multiplies exact (q - zero)
  // integers and unrounded activations in T itself.  Everywhere else the multiply runs in fp16:
  // the FULL path rounds each weight (a bf16 weight would carry up to 2^-8 relative error, more
  // than the GEMM's 2e-3 bound; fp16 carries 2^-11), and bf16 cannot hold the 8-bit and 3-bit
  // codes' magic-number forms exactly.  bf16 activations are then staged as fp16 times a power of
  // two per token (exact), and the partial sums are scaled back in fp32 before the one rounding.
  constexpr bool kBf16 = std::is_same<T, __nv_bfloat16>::value;
  constexpr bool kNative = !kBf16 || (FOLD && (BITS == 2 || BITS == 4));
  constexpr bool kConvert = !kNative;
  using TC = typename std::conditional<kNative, T, __half>::type;
  // the exact-difference unpack of the FOLD path
  using DP = DiffPairs<TC, BITS>;
  constexpr int PER = P::kPerUnit;
  constexpr int ROWS = P::kRowsPerUnit;
  constexpr int NP = MP::kPairs;
  constexpr int NB = (MT + 7) / 8;                    // token blocks of 8
  extern __shared__ __align__(128) unsigned char smem_raw[];

  // a flag-gated launch whose flag says no: every CTA leaves before any barrier or copy
  if (args.run_flag != nullptr && *args.run_flag != args.run_when) return;
  pdl_launch_dependents();
  // Grouped: the expert e of slot blockIdx.z multiplies rows [offsets[e], offsets[e + 1]) of A
  // into the same rows of C, with its own scales, zeros and packed rows (e * K * bits / 32 onward
  // in the stacked weight).  The offsets come from the kernel before this one, so they are read
  // after griddepcontrol.wait; a slot without an expert, the same for every CTA of its cluster,
  // leaves before any cluster barrier or copy.
  Args ga = args;                                     // the expert's view (grouped only)
  int w_row0 = 0;
  if constexpr (GROUPED) {
    pdl_wait();
    // With a slot per expert, slot z is expert z (two offsets read; a malformed range is flagged
    // by its own slot).  With fewer slots than experts (fewer rows than experts), slot z takes the
    // z-th expert that holds rows: every expert's range is read, and a malformed one (ga.M: the
    // caller's max_m, <= MT) holds none and is flagged by the grid's first CTA.
    int e, o0, o1;
    if (static_cast<int>(gridDim.z) == ga.experts) {
      e = static_cast<int>(blockIdx.z);
      o0 = ga.offsets[e];
      o1 = ga.offsets[e + 1];
      if (o0 == o1) return;
      if (o0 < 0 || o1 < o0 || o1 > ga.rows || o1 - o0 > ga.M) {
        if (threadIdx.x == 0 && blockIdx.x == 0 && blockIdx.y == 0) atomicOr(ga.status, kStatusExpertRows);
        return;
      }
    } else {
      const int4 f = find_expert(ga.offsets, ga.experts, ga.rows, ga.M, static_cast<int>(blockIdx.z));
      if (f.w && threadIdx.x == 0 && blockIdx.x == 0 && blockIdx.y == 0 && blockIdx.z == 0)
        atomicOr(ga.status, kStatusExpertRows);
      e = f.x;
      o0 = f.y;
      o1 = f.z;
      if (e < 0) return;                               // fewer experts hold rows than slots
    }
    ga.M = o1 - o0;
    ga.A = static_cast<const uint16_t*>(ga.A) + static_cast<long long>(o0) * ga.K;
    ga.C = static_cast<uint16_t*>(ga.C) + static_cast<long long>(o0) * ga.N;
    ga.qzeros += static_cast<long long>(e) * ga.G * ga.zwords;
    ga.scales += static_cast<long long>(e) * ga.G * ga.N;
    w_row0 = e * ga.units * ROWS;
  }
  const Args& a = GROUPED ? ga : args;
  // token split (one weight, grid z = token blocks of MT): this CTA's block of rows of A and C
  const int tz = GROUPED ? 0 : static_cast<int>(blockIdx.z);
  const int Mtok = MX > 0 ? MX : (GROUPED ? a.M : min(MT, a.M - tz * MT));   // tokens (compile-time when MX > 0)
  const int UW = unit_words(Mtok, NP);
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
  float* recv = reinterpret_cast<float*>(smem + SM::off_recv(geo, Mtok));
  uint32_t* sK = reinterpret_cast<uint32_t*>(smem + SM::off_gconst(geo, Mtok));   // [group][word][column]
  uint32_t* sSZ = reinterpret_cast<uint32_t*>(smem + SM::off_full(geo, Mtok));  // [group][column]
  uint16_t* sG = reinterpret_cast<uint16_t*>(sSZ + geo.full_groups * kSlab);    // [k of the range]
  uint8_t* misc = smem + SM::off_misc(geo, Mtok);
  const uint32_t bar0 = ptx::smem_addr(misc);
  volatile int* abort_flag = reinterpret_cast<volatile int*>(misc + 8 * kWarps * geo.nbuf);
  // bf16 activations: per token the largest staged |a| (bf16 bits) and the power of two 2^e the
  // fp16 staging was divided by
  uint32_t* tok_max = reinterpret_cast<uint32_t*>(misc + 8 * kWarps * geo.nbuf + 4 * (kWarps * geo.nbuf + 1));
  float* tok_scale = reinterpret_cast<float*>(tok_max + Mtok);
  // With refills (more chunks than buffers) and 2 to 8 tokens, warp w's box slot of buffer b
  // arrives on its own mbarrier, so warps refill and stream independently; otherwise one mbarrier
  // per chunk, refilled by the whole CTA at once (all 512 bytes of each row together, which
  // measured faster for 16 and 32 tokens).
  auto bar = [&](int w, int b) { return bar0 + 8u * static_cast<uint32_t>(w * geo.nbuf + b); };

  // Scales and zeros of the groups this range touches (FOLD): their loads go out first, ahead
  // of the weight stream (behind it they would wait for the whole slice), and land in shared
  // memory per group and column as (scale bits | runtime zero << 16).
  const int g_lo = (cu0 * PER) / a.group;
  const int g_end = (ct1 * 4 * PER - 1) / a.group;
  const int ngrp = ntile > 0 ? (g_end < a.G - 1 ? g_end : a.G - 1) - g_lo + 1 : 0;
  // The loads only fetch raw words: nothing consumes them before the weight copies are issued
  // (a shift of a loaded word right away would hold thread 0 for a full memory latency first).
  constexpr int kGB = 4;                               // group items per thread in flight
  uint2 gsv[kGB];
  uint2 gzw[kGB];                                      // the qzeros word(s) holding the 4 fields
  auto group_loads = [&](int base) {
#pragma unroll
    for (int j = 0; j < kGB; ++j) {
      const int i = base + j * kThreads + static_cast<int>(threadIdx.x);
      gsv[j] = make_uint2(0u, 0u);
      gzw[j] = make_uint2(0u, 0u);
      const int n = n_base + 4 * (i & 31);
      if (i < ngrp * 32 && n < a.N) {
        const int g = g_lo + (i >> 5);
        gsv[j] = __ldg(reinterpret_cast<const uint2*>(a.scales + static_cast<long long>(g) * a.N + n));
        const int32_t* zrow = a.qzeros + static_cast<long long>(g) * a.zwords;
        const int bit = BITS * n;
        gzw[j].x = static_cast<uint32_t>(__ldg(zrow + (bit >> 5)));
        if (BITS == 3 && (bit & 31) + 12 > 32) gzw[j].y = static_cast<uint32_t>(__ldg(zrow + (bit >> 5) + 1));
      }
    }
  };
  auto group_stores = [&](int base) {
#pragma unroll
    for (int j = 0; j < kGB; ++j) {
      const int i = base + j * kThreads + static_cast<int>(threadIdx.x);
      if (i < ngrp * 32) {
        // the 4 zero fields of columns n .. n + 3, LSB-first (4 * BITS bits)
        const uint32_t zf = __funnelshift_r(gzw[j].x, gzw[j].y, (BITS * (n_base + 4 * (i & 31))) & 31);
        uint32_t w[4];
#pragma unroll
        for (int c = 0; c < 4; ++c) {
          const uint32_t h = c & 1 ? hi16(c < 2 ? gsv[j].x : gsv[j].y) : lo16(c < 2 ? gsv[j].x : gsv[j].y);
          w[c] = h | ((((zf >> (BITS * c)) & P::kMask) + a.zero_offset) << 16);
        }
        *reinterpret_cast<uint4*>(sK + (i >> 5) * kSlab + 4 * (i & 31)) = make_uint4(w[0], w[1], w[2], w[3]);
      }
    }
  };
  if constexpr (FOLD) group_loads(0);

  // Issue the packed slice into shared memory: chunk c of this CTA lands in buffer c % nbuf.
  // The copies read weights only; they are issued before griddepcontrol.wait because global
  // memory (through L2) is coherent for them and the weights are not produced by the kernel
  // this one may overlap with.
  const bool per_warp = MT == 8 && geo.nbuf < nchunk;
  const int bw = per_warp ? warp : 0;                  // this warp's mbarrier row
  if (threadIdx.x == 0) {
    for (int w = 0; w < (per_warp ? kWarps : 1); ++w)
      for (int b = 0; b < geo.nbuf; ++b) ptx::mbar_init(bar(w, b), 1);
    *abort_flag = 0;
    ptx::fence_mbar_init();
  }
  if (kConvert && static_cast<int>(threadIdx.x) < Mtok) tok_max[threadIdx.x] = 0u;
  __syncthreads();
  volatile int* last_issued = abort_flag + 1;          // [warp][nbuf] last chunk issued per buffer
  // the packed weights are read once: evict them first, so that activations and other reused
  // data keep their place in L2
  const uint64_t stream_policy = ptx::policy_evict_first();
  // Interleaved weights (gptq_prepack_interleave): warp w's 32-column block is contiguous along
  // K, 512 * ROWS bytes per k-tile in lane order, so one 1D bulk copy moves its part of a chunk;
  // its byte count stops at the CTA's last k-tile (nothing past the block is read) and a block
  // past N copies nothing.
  constexpr uint32_t kIlTile = 512u * ROWS;
  auto il_bytes = [&](int w, int c) -> uint32_t {
    if ((n_base >> 5) + w >= (a.N >> 5)) return 0u;
    const int nt = ntile - c * geo.chunk_tiles;
    return static_cast<uint32_t>(nt < geo.chunk_tiles ? nt : geo.chunk_tiles) * kIlTile;
  };
  auto il_copy = [&](int w, int c, uint32_t dst, uint32_t barw, uint32_t bytes) {
    if (bytes == 0u) return;
    const size_t tile0 = static_cast<size_t>((n_base >> 5) + w) * a.il_tiles + ct0 + c * geo.chunk_tiles;
    ptx::bulk_load_hint(dst, reinterpret_cast<const uint8_t*>(a.qweight) + tile0 * kIlTile, bytes, barw,
                        stream_policy);
  };
  // copy warp w's 32 columns of chunk c into buffer c % nbuf (its own slot and mbarrier)
  auto issue_for = [&](int w, int c) {
    const int b = c % geo.nbuf;
    last_issued[w * geo.nbuf + b] = c;
    const uint32_t dst = ptx::smem_addr(sbuf + static_cast<size_t>(b) * geo.chunk_bytes +
                                        static_cast<size_t>(w) * geo.slot_bytes);
    if (a.il_tiles) {
      const uint32_t bytes = il_bytes(w, c);
      ptx::mbar_arrive_expect_tx(bar(w, b), bytes);
      il_copy(w, c, dst, bar(w, b), bytes);
      return;
    }
    const int row0 = w_row0 + (cu0 + c * geo.chunk_tiles * 4) * ROWS;
    ptx::mbar_arrive_expect_tx(bar(w, b), static_cast<uint32_t>(geo.chunk_rows * kBoxRowBytes));
    ptx::tma_load_2d_hint(dst, &tmW, n_base + w * kBoxCols, row0, bar(w, b), stream_policy);
  };
  // all four slots of chunk c on one mbarrier (single-barrier mode)
  auto issue_chunk = [&](int c) {
    const int b = c % geo.nbuf;
    last_issued[b] = c;
    auto slot_addr = [&](int w) {
      return ptx::smem_addr(sbuf + static_cast<size_t>(b) * geo.chunk_bytes + static_cast<size_t>(w) * geo.slot_bytes);
    };
    if (a.il_tiles) {
      uint32_t total = 0u;
      for (int w = 0; w < kWarps; ++w) total += il_bytes(w, c);
      ptx::mbar_arrive_expect_tx(bar(0, b), total);
      for (int w = 0; w < kWarps; ++w) il_copy(w, c, slot_addr(w), bar(0, b), il_bytes(w, c));
      return;
    }
    const int row0 = w_row0 + (cu0 + c * geo.chunk_tiles * 4) * ROWS;
    ptx::mbar_arrive_expect_tx(bar(0, b), static_cast<uint32_t>(kWarps * geo.chunk_rows * kBoxRowBytes));
    for (int w = 0; w < kWarps; ++w)
      ptx::tma_load_2d_hint(slot_addr(w), &tmW, n_base + w * kBoxCols, row0, bar(0, b), stream_policy);
  };
  // refill after chunk c_next - nbuf was consumed: per warp (its slot) or by the whole CTA
  // (per_warp is uniform over the CTA, and so is the loop's chunk sequence)
  auto refill = [&](int c_next) {
    if (per_warp) {
      __syncwarp();
      if (lane == 0 && !*abort_flag) { ptx::fence_proxy_async_smem(); issue_for(warp, c_next); }
    } else {
      __syncthreads();
      if (threadIdx.x == 0 && !*abort_flag) { ptx::fence_proxy_async_smem(); issue_chunk(c_next); }
    }
  };
  if (threadIdx.x == 0) {                                // the first chunks in one burst
    for (int c = 0; c < nchunk && c < geo.nbuf; ++c) {
      if (per_warp) {
        for (int w = 0; w < kWarps; ++w) issue_for(w, c);
      } else {
        issue_chunk(c);
      }
    }
  }

  if constexpr (FOLD) {
    group_stores(0);
    for (int base = kGB * kThreads; base < ngrp * 32; base += kGB * kThreads) {
      group_loads(base);
      group_stores(base);
    }
  } else if (geo.full_groups > 0) {
    // FULL: scales and runtime zeros (fp16 bits of each, scale in the low half) and the group of
    // every k of the range, read once into shared memory (with g_idx every group may occur, so
    // all G are staged).  Checkpoint data, like the weights, so this too precedes
    // griddepcontrol.wait.
    const int g_base = a.g_idx ? 0 : g_lo;
    const int ng = a.g_idx ? a.G : ngrp;
    for (int i = threadIdx.x; i < ng * 32; i += kThreads) {
      const int gi = i >> 5, n = n_base + 4 * (i & 31);
      uint4 v = make_uint4(0u, 0u, 0u, 0u);
      if (n < a.N) {
        const int g = g_base + gi;
        const uint2 sv = __ldg(reinterpret_cast<const uint2*>(a.scales + static_cast<long long>(g) * a.N + n));
        const uint32_t zf = zeros4<BITS>(a.qzeros + static_cast<long long>(g) * a.zwords, n);
        uint32_t zz[4];
#pragma unroll
        for (int c = 0; c < 4; ++c)   // an integer in [0, 256]: exact in fp16
          zz[c] = __half_as_ushort(__int2half_rn(static_cast<int>(((zf >> (BITS * c)) & P::kMask) + a.zero_offset)));
        v = make_uint4(lo16(sv.x) | (zz[0] << 16), hi16(sv.x) | (zz[1] << 16), lo16(sv.y) | (zz[2] << 16),
                       hi16(sv.y) | (zz[3] << 16));
      }
      *reinterpret_cast<uint4*>(sSZ + gi * kSlab + 4 * (i & 31)) = v;
    }
    const int k0 = cu0 * PER, nk = ntile * 4 * PER;
    for (int i = threadIdx.x; i < nk; i += kThreads) {
      const int k = k0 + i < a.K ? k0 + i : a.K - 1;
      const int g = a.g_idx ? checked_group(a, k) : k / a.group;
      sG[i] = static_cast<uint16_t>(g - g_base);
    }
  }
  pdl_wait();

  // Stage activations: sB[u][m][p] = (a[m][k0 + lo_k(p)], a[m][k0 + hi_k(p)]), zero past K or M.
  const uint16_t* A16 = static_cast<const uint16_t*>(a.A) + static_cast<long long>(tz) * MT * a.K;
  const int nunits = ntile * 4;
  stage_pairs<PER, NP>(A16, a.perm, Mtok, a.K, cu0, nunits, a.units,
                       [](int p) { return MP::lo_k(p); }, [](int p) { return MP::hi_k(p); },
                       [&](int uu, int m, int p, uint32_t v) { sB[uu * UW + m * NP + p] = v; },
                       static_cast<int>(threadIdx.x), kThreads);
  __syncthreads();
  if constexpr (kConvert) {
    // bf16 -> fp16: per token, 2^e with max|a| * 2^-e in [2^15, 2^16) (below fp16's largest
    // finite value for any bf16 significand); every staged value times 2^-e is exact and, in
    // fp16's normal range, exactly representable; the partial sums are multiplied by 2^e before
    // the reduction.
    // per-thread maxima over the staged items (unit, token); where the token count divides the
    // CTA, a thread's items all belong to one token and it flushes once
    {
      int cur_m = -1;
      uint32_t mx = 0u;
      for (int it = threadIdx.x; it < nunits * Mtok; it += kThreads) {
        const int uu = it / Mtok, m = it - uu * Mtok;
        if (m != cur_m) {
          if (mx) atomicMax(tok_max + cur_m, mx);
          cur_m = m;
          mx = 0u;
        }
        const uint32_t* src = sB + uu * UW + m * NP;
#pragma unroll
        for (int p = 0; p < NP; ++p) {
          const uint32_t v = src[p];
          mx = max(mx, max(v & 0x7FFFu, (v >> 16) & 0x7FFFu));
        }
      }
      if (mx) atomicMax(tok_max + cur_m, mx);
    }
    __syncthreads();
    if (static_cast<int>(threadIdx.x) < Mtok) {
      const uint32_t mx = tok_max[threadIdx.x];
      int e = mx ? static_cast<int>(mx >> 7) - 127 - 15 : 0;   // exponent field of max|a|, minus 15
      e = e < -126 ? -126 : (e > 126 ? 126 : e);               // 2^e and 2^-e stay normal floats
      tok_scale[threadIdx.x] = __uint_as_float(static_cast<uint32_t>(e + 127) << 23);
    }
    __syncthreads();
    for (int it = threadIdx.x; it < nunits * Mtok; it += kThreads) {
      const int uu = it / Mtok, m = it - uu * Mtok;
      const float inv = __uint_as_float((254u << 23) - __float_as_uint(tok_scale[m]));   // 2^-e
      uint32_t* w = sB + uu * UW + m * NP;
#pragma unroll
      for (int p = 0; p < NP; ++p) {
        const uint32_t v = w[p];
        w[p] = pack2(__uint_as_float(v << 16) * inv, __uint_as_float(v & 0xFFFF0000u) * inv, __half());
      }
    }
    __syncthreads();
  }

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
      if (8 * nb + gq >= Mtok) {                         // absent token: zero B column
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
  // this thread's 16 bytes of row r (0 .. ROWS - 1) of its unit in local k-tile l of a chunk slot:
  // the tensor-map layout holds 128-byte rows with the 128-byte swizzle, the interleaved one
  // 512-byte k-tile rows in lane order
  const uint8_t* wslot = sbuf + warp * geo.slot_bytes;
  auto wfrag = [&](const uint8_t* slot, int l, int r) {
    if (a.il_tiles) return *reinterpret_cast<const uint4*>(slot + (l * ROWS + r) * 512 + lane * 16);
    const int row = (l * 4 + tq) * ROWS + r;
    return *reinterpret_cast<const uint4*>(slot + row * kBoxRowBytes + ((quad ^ (row & 7)) << 4));
  };

  if constexpr (FOLD) {
    static_assert(DP::kPairs == NP, "pairing must match the activation staging");
    // MMAs of exact (q - zero) pairs into a per-group accumulator cg; at each group end
    //   acc += scale * cg.
    // Tiles go in blocks of 4 where a block stays inside one chunk and one group (shared-memory
    // offsets then are immediates); absent tokens read token M-1's activations (their outputs
    // are never stored).
    float cg[2][NB][4];
    float gs[4];                                       // the current group's scales (4 columns)
    uint32_t gk[4][DP::kConsts];                       // and the unpack constants of its zeros
    auto load_group = [&](int gi) {
      const uint4 v = *reinterpret_cast<const uint4*>(sK + gi * kSlab + col0);
#pragma unroll
      for (int c = 0; c < 4; ++c) {
        const uint32_t e = (&v.x)[c];
        gs[c] = __half2float(__ushort_as_half(lo16(e)));
        DP::consts(static_cast<int>(e >> 16), gk[c]);
      }
    };
    auto clear_cg = [&]() {
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
        for (int nb = 0; nb < NB; ++nb)
#pragma unroll
          for (int i = 0; i < 4; ++i) acc[t][nb][i] = fmaf(gs[2 * t + (i >> 1)], cg[t][nb][i], acc[t][nb][i]);
    };
    int boff[NB];                                      // word offset of this thread's tokens
#pragma unroll
    for (int nb = 0; nb < NB; ++nb) {
      const int m = 8 * nb + gq;
      boff[nb] = (m < Mtok ? m : Mtok - 1) * NP + tq * UW;
    }
    // 3-bit: unit tq of local tile l is rows 3 (4 l + tq) .. +2 of the chunk; pairs per column
    auto tile3 = [&](const uint8_t* cslot, int l, int kt) {
      uint4 wv[3];
#pragma unroll
      for (int r = 0; r < 3; ++r) wv[r] = wfrag(cslot, l, r);
      uint32_t bf[NB][NP];
#pragma unroll
      for (int nb = 0; nb < NB; ++nb) {
        const uint32_t* src = sB + kt * 4 * UW + boff[nb];
#pragma unroll
        for (int i = 0; i < NP / 4; ++i) {
          const uint4 v = reinterpret_cast<const uint4*>(src)[i];
          bf[nb][4 * i] = v.x; bf[nb][4 * i + 1] = v.y; bf[nb][4 * i + 2] = v.z; bf[nb][4 * i + 3] = v.w;
        }
      }
#pragma unroll
      for (int t = 0; t < 2; ++t) {
        uint32_t d0[NP], d1[NP];
        if constexpr (BITS == 3) {
          DP::run3((&wv[0].x)[2 * t], (&wv[1].x)[2 * t], (&wv[2].x)[2 * t], gk[2 * t], d0);
          DP::run3((&wv[0].x)[2 * t + 1], (&wv[1].x)[2 * t + 1], (&wv[2].x)[2 * t + 1], gk[2 * t + 1], d1);
        }
#pragma unroll
        for (int j = 0; j < NP / 2; ++j)
#pragma unroll
          for (int nb = 0; nb < NB; ++nb)
            mma16816(cg[t][nb], d0[2 * j], d1[2 * j], d0[2 * j + 1], d1[2 * j + 1], bf[nb][2 * j],
                     bf[nb][2 * j + 1], TC());
      }
    };
    auto tile = [&](const uint8_t* wp, int kt) {
      const uint4 wv = *reinterpret_cast<const uint4*>(wp);
      uint32_t bf[NB][NP];
#pragma unroll
      for (int nb = 0; nb < NB; ++nb) {
        const uint32_t* src = sB + kt * 4 * UW + boff[nb];
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
      uint32_t d[4][NP];
#pragma unroll
      for (int cc = 0; cc < 4; ++cc) {
        if constexpr (BITS != 3) DP::run((&wv.x)[cc], gk[cc], d[cc]);
      }
#pragma unroll
      for (int j = 0; j < NP / 2; ++j)
#pragma unroll
        for (int t = 0; t < 2; ++t)
#pragma unroll
          for (int nb = 0; nb < NB; ++nb)
            mma16816(cg[t][nb], d[2 * t][2 * j], d[2 * t + 1][2 * j], d[2 * t][2 * j + 1],
                     d[2 * t + 1][2 * j + 1], bf[nb][2 * j], bf[nb][2 * j + 1], TC());
    };
    const int tpg = a.group / (4 * PER);               // k-tiles per group (>= 1 here)
    int gi = 0, g_end_kt = tpg - (ct0 % tpg);          // local group, tile where it ends
    int c = -1, chunk_kt = 0, chunk_end = 0;
    bool ok = true, dirty = false;
    const uint8_t* we = wslot;                         // rows of even / odd k-tiles of the chunk
    const uint8_t* wo = wslot;
    const uint8_t* cslot = wslot;                      // this warp's box slot of the chunk
    clear_cg();
    if (ntile > 0) load_group(0);
    for (int kt = 0; kt < ntile;) {                    // control flow is uniform over the CTA
      if (kt == chunk_end) {
        if (c >= 0 && c + geo.nbuf < nchunk) refill(c + geo.nbuf);   // the buffer just consumed
        ++c;
        ok = __all_sync(0xFFFFFFFFu, tma_wait(bar(bw, c % geo.nbuf), (c / geo.nbuf) & 1, abort_flag, a.status));
        cslot = wslot + static_cast<size_t>(c % geo.nbuf) * geo.chunk_bytes;
        if (a.il_tiles) {
          we = wo = cslot + lane * 16;
        } else {
          const uint8_t* cb = cslot + tq * kBoxRowBytes;
          we = cb + ((quad ^ tq) << 4);
          wo = cb + ((quad ^ tq ^ 4) << 4);
        }
        chunk_kt = c * geo.chunk_tiles;
        chunk_end = chunk_kt + geo.chunk_tiles < ntile ? chunk_kt + geo.chunk_tiles : ntile;
      }
      const int lim = chunk_end < g_end_kt ? chunk_end : g_end_kt;
      const int l0 = kt - chunk_kt;
      if constexpr (BITS == 3) {
        if (ok) tile3(cslot, l0, kt);
        kt += 1;
      } else if (lim - kt >= 4) {
        if (ok) {
          const uint8_t* e = (l0 & 1) ? wo : we;
          const uint8_t* o = (l0 & 1) ? we : wo;
#pragma unroll
          for (int u = 0; u < 4; ++u) tile(((u & 1) ? o : e) + (l0 + u) * 4 * kBoxRowBytes, kt + u);
        }
        kt += 4;
      } else {
        if (ok) tile(((l0 & 1) ? wo : we) + l0 * 4 * kBoxRowBytes, kt);
        kt += 1;
      }
      dirty = true;
      if (kt == g_end_kt) {
        fold();
        clear_cg();
        dirty = false;
        ++gi;
        g_end_kt += tpg;
        if (kt < ntile) load_group(gi);
      }
    }
    if (dirty) fold();
  } else {
    for (int c = 0; c < nchunk; ++c) {
      const bool ok = __all_sync(0xFFFFFFFFu, tma_wait(bar(bw, c % geo.nbuf), (c / geo.nbuf) & 1, abort_flag, a.status));
      const uint8_t* cb = wslot + static_cast<size_t>(c % geo.nbuf) * geo.chunk_bytes;
      const int kt0 = c * geo.chunk_tiles;
      const int kt_end = kt0 + geo.chunk_tiles < ntile ? kt0 + geo.chunk_tiles : ntile;
      for (int kt = kt0; ok && kt < kt_end; ++kt) {
        uint4 wv[ROWS];
#pragma unroll
        for (int r = 0; r < ROWS; ++r) wv[r] = wfrag(cb, kt - kt0, r);
        uint32_t bf[NB][NP];
        load_b(kt, bf);
        const int u = cu0 + kt * 4 + tq;
        const int uk = (u < a.units ? u : a.units - 1) * PER;
        const uint16_t* gk = sG + (kt * 4 + tq) * PER;   // staged groups of this unit's k
        // dequantize this unit for 4 columns: w[c][p] = RN((q - z) * s) pairs
        uint32_t w[4][NP];
        if (geo.full_groups > 0) {
          // exact code pairs (q_lo, q_hi) of the 4 columns (the FOLD unpack with a zero of 0), then
          // per pair the (scale, zero) words of its two k's groups for the 4 columns: (q - z) is
          // exact in fp16 and one fp16 product rounds RN((q - z) s) once
          using QP = DiffPairs<__half, BITS>;
          uint32_t kz0[QP::kConsts];
          QP::consts(0, kz0);
#pragma unroll
          for (int cc = 0; cc < 4; ++cc) {
            if constexpr (BITS == 3)
              QP::run3((&wv[0].x)[cc], (&wv[1].x)[cc], (&wv[2].x)[cc], kz0, w[cc]);
            else
              QP::run((&wv[0].x)[cc], kz0, w[cc]);
          }
#pragma unroll
          for (int p = 0; p < NP; ++p) {
            const uint4 wl = *reinterpret_cast<const uint4*>(sSZ + gk[MP::lo_k(p)] * kSlab + col0);
            const uint4 wh = *reinterpret_cast<const uint4*>(sSZ + gk[MP::hi_k(p)] * kSlab + col0);
#pragma unroll
            for (int cc = 0; cc < 4; ++cc) {
              const uint32_t el = (&wl.x)[cc], eh = (&wh.x)[cc];
              w[cc][p] = hmul2(sub2(w[cc][p], __byte_perm(el, eh, 0x7632), __half()), __byte_perm(el, eh, 0x5410));
            }
          }
        } else {
          // groups, scales and zeros read through L1 (too many groups to stage)
          float s[4], zf[4];
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
                int z[4];
                load_sz<BITS>(a, gg, n0c, s, z);
#pragma unroll
                for (int cc = 0; cc < 4; ++cc) zf[cc] = 8388608.0f + static_cast<float>(z[cc]);
                cur_g = gg;
              }
              // q - z exactly (magic 2^23 has ulp 1), one fp32 product, rounded once below
#pragma unroll
              for (int cc = 0; cc < 4; ++cc)
                v[cc][h] = (__uint_as_float(0x4B000000u | unit_code<BITS>(wv, cc, j)) - zf[cc]) * s[cc];
            }
#pragma unroll
            for (int cc = 0; cc < 4; ++cc) w[cc][p] = pack2(v[cc][0], v[cc][1], TC());
          }
        }
#pragma unroll
        for (int j = 0; j < NP / 2; ++j)
#pragma unroll
          for (int t = 0; t < 2; ++t)
#pragma unroll
            for (int nb = 0; nb < NB; ++nb)
              mma16816(acc[t][nb], w[2 * t][2 * j], w[2 * t + 1][2 * j], w[2 * t][2 * j + 1],
                       w[2 * t + 1][2 * j + 1], bf[nb][2 * j], bf[nb][2 * j + 1], TC());
      }
      if (c + geo.nbuf < nchunk) refill(c + geo.nbuf);   // the buffer just consumed
    }
  }

  // ---- the cluster reduce-scatter into the receive slots ([cs][M][kSlab / cs], a region of its
  // own: peers may push while this CTA still reads its staged activations) of the CTA that owns
  // each column.  Fragment element i of acc[t][nb] is column 2t + (i >> 1) of the thread's quad
  // and token 8 nb + 2 tq + (i & 1).
  const int Mr = Mtok;
  const int per_rank = kSlab / cs;                      // cs is a power of two
  const int pr_shift = __ffs(per_rank) - 1;
  if (MX == 1 || Mtok == 1) {
    // one token: 128 sums per CTA, pushed straight from registers (so the staging needs no room
    // for partial sums; the run-time token count takes this branch too when a grouped expert
    // holds one row)
    cluster_wait();
#pragma unroll
    for (int t = 0; t < 2; ++t)
#pragma unroll
      for (int r = 0; r < 2; ++r)
        if (tq == 0) {
          const int col = col0 + 2 * t + r;
          const int owner = col >> pr_shift;
          float* dst = cluster.map_shared_rank(recv, owner);
          dst[rank * per_rank + (col - owner * per_rank)] = kConvert ? acc[t][0][2 * r] * tok_scale[0] : acc[t][0][2 * r];
        }
  } else {
    // several tokens: through shared memory first, so that consecutive threads push consecutive
    // columns (coalesced remote stores)
    __syncthreads();                                    // done with the staged activations
    float* part = reinterpret_cast<float*>(sB);         // [M][kSlab], aliases the staging
#pragma unroll
    for (int t = 0; t < 2; ++t)
#pragma unroll
      for (int nb = 0; nb < NB; ++nb)
#pragma unroll
        for (int i = 0; i < 4; ++i) {
          const int col = col0 + 2 * t + (i >> 1), m = nb * 8 + 2 * tq + (i & 1);
          if (m < Mr) part[m * kSlab + col] = kConvert ? acc[t][nb][i] * tok_scale[m] : acc[t][nb][i];
        }
    __syncthreads();
    cluster_wait();
    for (int i = threadIdx.x; i < Mr * kSlab; i += kThreads) {
      const int m = i / kSlab, col = i - m * kSlab;
      const int owner = col >> pr_shift;
      float* dst = cluster.map_shared_rank(recv, owner);
      dst[(rank * Mr + m) * per_rank + (col - owner * per_rank)] = part[i];
    }
  }
  cluster.sync();
  T* C = static_cast<T*>(a.C) + static_cast<long long>(tz) * MT * a.N;
  for (int i = threadIdx.x; i < Mr * per_rank; i += kThreads) {
    const int m = i >> pr_shift, c = i - (m << pr_shift);
    const int n = n_base + rank * per_rank + c;
    if (n < a.N) {
      float v = 0.f;
      for (int q = 0; q < cs; ++q) v += recv[(q * Mr + m) * per_rank + c];
      C[static_cast<long long>(m) * a.N + n] = F16Traits<T>::from_f32(v);
    }
  }
  if (*abort_flag && lane == 0 && (per_warp || warp == 0)) {
    // after a timeout, let every copy issued on this warp's mbarriers land before shared memory
    // is released
    const uint64_t t0 = ptx::globaltimer();
    for (int b = 0; b < nchunk && b < geo.nbuf; ++b) {
      const int last = last_issued[bw * geo.nbuf + b];
      while (!ptx::mbar_try_wait(bar(bw, b), (last / geo.nbuf) & 1) &&
             ptx::globaltimer() - t0 < 2000000000ull) {}
    }
  }
}

// Chunking of a CTA range: chunks of at most 32 KB whose k-tile count divides the range when it
// can; as many buffers as the shared-memory share of one CTA allows when every CTA of the grid
// is resident at once (one wave), at least 2 -- all of them for the common one-token shapes, so
// the whole slice is in flight from the first cycle.
template <int BITS>
TmaGeo make_geo(int units, int cs, int M, int group, int ctas, int sm_count, int max_per_sm, bool full,
                bool has_gidx, int G) {
  constexpr int ROWS = Pack<BITS>::kRowsPerUnit;
  constexpr int PER = Pack<BITS>::kPerUnit;
  TmaGeo g;
  g.cs = cs;
  const int tiles_total = (units + 3) / 4;
  g.tiles_per_cta = (tiles_total + cs - 1) / cs;
  const int tile_bytes = 4 * ROWS * kSlab * 4;
  const int tpg = group / (4 * PER);
  g.max_groups = (tpg >= 1 ? (g.tiles_per_cta + tpg - 1) / tpg : g.tiles_per_cta) + 1;
  if (full) g.max_groups = 0;                                  // no FOLD constants or sums
  // FULL path: stage scales/zeros (all G with g_idx) and per-k groups when they take <= 24 KB
  g.full_groups = 0;
  g.full_k = g.tiles_per_cta * 4 * PER;
  if (full) {
    const int range_groups = (g.tiles_per_cta * 4 * PER + group - 1) / group + 1;
    const int ng = has_gidx ? G : (range_groups < G ? range_groups : G);
    if (static_cast<size_t>(ng) * kSlab * 4 + static_cast<size_t>(g.full_k) * 2 <= 24 * 1024) g.full_groups = ng;
  }
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
    // an SM holds 228 KB; each CTA takes its size rounded up to 1 KB plus 1 KB reserved
    const long long cap = (static_cast<long long>(233472 / per_sm) - 1024) & ~1023LL;
    const long long budget = cap - static_cast<long long>(fixed);
    // each buffer also takes an mbarrier and a bookkeeping word per warp
    const long long per_buf = g.chunk_bytes + kWarps * (8 + 4);
    int fit = budget > 0 ? static_cast<int>(budget / per_buf) : 0;
    if (fit > 16) fit = 16;
    g.nbuf = chunks < fit ? chunks : fit;
    return chunks;
  };
  int ct = 1;
  for (int d = 1; d * tile_bytes <= 32 * 1024 && d <= g.tiles_per_cta; ++d)
    if (g.tiles_per_cta % d == 0) ct = d;
  int chunks = layout(ct);
  while (g.nbuf < 2 && g.nbuf < chunks && ct > 1) chunks = layout(ct = (ct + 1) / 2);
  if (g.nbuf < 1) g.nbuf = 1;
  if (g.nbuf < 2 && chunks >= 2) g.nbuf = 2;                  // past one wave rather than serial
  return g;
}

// The launch geometry of one decode call: the cluster size (K split) and the shared-memory layout.
// `regs` is the kernel's register count (it bounds the CTAs per SM), `E` the experts side by
// side in the grid (1 for a single weight).  Host code only; the launcher and the host-side
// geometry tests both call it.
struct GeoChoice {
  int cs;
  TmaGeo geo;
  bool fits;          // false: the layout fits no CTA even split 16 ways; nothing may launch
};

template <int BITS>
GeoChoice select_geometry(const Problem& p, bool fold, int regs, int sms, int E) {
  const int units = p.K / Pack<BITS>::kPerUnit;
  const int slabs = (p.N + kSlab - 1) / kSlab;
  const int by_regs = regs > 0 ? 65536 / (((regs + 7) & ~7) * kThreads) : 5;
  const int max_per_sm = by_regs < 1 ? 1 : (by_regs > 5 ? 5 : by_regs);
  // FOLD: one wave when it can be had -- the largest K split (at most the chosen one) whose grid
  // is resident at once; halving stops where a CTA's shared memory would no longer fit (a
  // smaller split stages more activations), and the chosen split stays when no split gives one
  // wave.  FULL keeps the chosen split: it is latency-bound and gains from every extra CTA.
  auto geo_for = [&](int c) {
    return make_geo<BITS>(units, c, p.M, p.group, slabs * c * E, sms, max_per_sm, !fold, p.g_idx != nullptr,
                          p.G);
  };
  // A 16-CTA cluster is used only when it gives one wave; otherwise (and for FULL) at most 8, and
  // at most 4 for several weights side by side (grouped experts), whose grids run many waves:
  // fewer, larger CTAs measured faster there (8 experts x [4096, 14336] 4-bit: T=8 106 -> 82 us,
  // T=1 26 -> 22 us).
  const int cs0 = choose_cluster(p, Pack<BITS>::kPerUnit);
  const int cs_cap = E > 1 ? 4 : 8;
  int cs = cs0 < cs_cap ? cs0 : cs_cap;
  for (int c = cs0; fold && c >= 1; c /= 2) {
    const size_t bytes = (TmaSmem<BITS>::bytes(geo_for(c), p.M) + 1023) & ~static_cast<size_t>(1023);
    if (bytes > 227 * 1024) break;
    int per_sm = static_cast<int>(233472 / (bytes + 1024));
    per_sm = per_sm < max_per_sm ? per_sm : max_per_sm;
    if (static_cast<long long>(slabs) * c * E <= static_cast<long long>(per_sm) * sms) {
      cs = c;
      break;
    }
  }
  TmaGeo geo = geo_for(cs);
  // A layout that does not fit one CTA (a long K range with many tokens stages many activations):
  // widen the split while every warp of a CTA keeps a k-tile of its own; beyond 16 CTAs nothing is
  // launched and the caller takes another path.
  while (TmaSmem<BITS>::bytes(geo, p.M) > kMaxCtaSmem && cs < 16 && units >= 4 * (2 * cs) * kWarps) {
    cs *= 2;
    geo = geo_for(cs);
  }
  return GeoChoice{cs, geo, TmaSmem<BITS>::bytes(geo, p.M) <= kMaxCtaSmem};
}

template <int BITS, int MT, int MX, typename T, bool FOLD, bool GROUPED>
cudaError_t launch_mma(const Problem& p, cudaStream_t stream) {
  Args a;
  a.A = p.A; a.M = p.M; a.K = p.K; a.N = p.N;
  a.qweight = p.qweight; a.qzeros = p.qzeros;
  a.scales = static_cast<const __half*>(p.scales);
  a.g_idx = p.g_idx; a.perm = p.perm; a.group = p.group; a.G = p.G; a.zero_offset = p.zero_offset;
  a.zwords = p.N * BITS / 32;
  a.units = p.K / Pack<BITS>::kPerUnit;
  a.C = p.out; a.status = p.status;
  a.offsets = GROUPED ? p.offsets : nullptr;
  a.rows = p.rows;
  a.experts = GROUPED ? p.E : 0;
  a.il_tiles = p.interleaved ? a.units / 4 : 0;
  a.run_flag = p.run_flag;
  a.run_when = p.run_when;
  const int E = GROUPED ? p.E : 1;                     // weights side by side
  // grid z: expert slots (no more than the rows, each of which belongs to one expert) or token blocks
  const int Z = GROUPED ? (p.E < p.rows ? p.E : p.rows) : (p.tok_split > 1 ? p.tok_split : 1);
  if (Z <= 0) return cudaSuccess;
  Problem pz = p;                                      // the geometry of one token block
  if (!GROUPED && Z > 1) pz.M = MT;
  const int slabs = (p.N + kSlab - 1) / kSlab;
  const int sms = device_info().sm_count;
  auto kern = k_decode_mma<BITS, MT, MX, T, FOLD, GROUPED>;
  // CTAs per SM the registers allow (read once per kernel from its attributes)
  static std::atomic<int> regs_cache{-1};
  int regs = regs_cache.load(std::memory_order_relaxed);
  if (regs < 0) {
    cudaFuncAttributes fa;
    regs = cudaFuncGetAttributes(&fa, kern) == cudaSuccess ? fa.numRegs : 0;
    regs_cache.store(regs, std::memory_order_relaxed);
  }
  const GeoChoice choice = select_geometry<BITS>(pz, FOLD, regs, sms, Z);
  if (!choice.fits) return cudaErrorInvalidConfiguration;
  const int cs = choice.cs;
  const TmaGeo geo = choice.geo;
  if constexpr (MT == 8 && MX > 0) {
    // refills ahead: the runtime-count instantiation, whose warps refill independently, is faster
    // there (measured); the exact one wins when the whole slice is in flight
    const int chunks = (geo.tiles_per_cta + geo.chunk_tiles - 1) / geo.chunk_tiles;
    if (geo.nbuf < chunks) return launch_mma<BITS, MT, 0, T, FOLD, GROUPED>(p, stream);
  }
  CUtensorMap tmW = {};
  if (!p.interleaved) {
    constexpr int ROWS = Pack<BITS>::kRowsPerUnit;
    const cuuint64_t dims[2] = {static_cast<cuuint64_t>(p.N), static_cast<cuuint64_t>(a.units) * ROWS * E};
    const cuuint64_t strides[1] = {static_cast<cuuint64_t>(p.N) * 4};
    const cuuint32_t box[2] = {static_cast<cuuint32_t>(kBoxCols), static_cast<cuuint32_t>(geo.chunk_rows)};
    const cuuint32_t estr[2] = {1, 1};
    if (!encode_tensor_map(&tmW, CU_TENSOR_MAP_DATA_TYPE_INT32, const_cast<int32_t*>(p.qweight), dims,
                           strides, box, estr, CU_TENSOR_MAP_SWIZZLE_128B))
      return cudaErrorInvalidValue;
  }
  const size_t smem = TmaSmem<BITS>::bytes(geo, pz.M);
  // once per device, FOLD only: the full shared-memory carveout (left to the driver, it may pick
  // a smaller one and fit fewer CTAs per SM than the one-wave budget above assumes).  The FULL
  // path keeps the driver's choice: it re-reads scales through L1, which the carveout would shrink.
  static std::atomic<unsigned long long> carveout_set{0};
  const int dev = device_info().device;
  if (FOLD && (dev >= 64 || !(carveout_set.load(std::memory_order_relaxed) & (1ull << dev)))) {
    cudaError_t e = cudaFuncSetAttribute(kern, cudaFuncAttributePreferredSharedMemoryCarveout,
                                         static_cast<int>(cudaSharedmemCarveoutMaxShared));
    if (e != cudaSuccess) return e;
    if (dev < 64) carveout_set.fetch_or(1ull << dev, std::memory_order_relaxed);
  }
  if (smem > 48 * 1024) {
    cudaError_t e = cudaFuncSetAttribute(kern, cudaFuncAttributeMaxDynamicSharedMemorySize,
                                         static_cast<int>(smem));
    if (e != cudaSuccess) return e;
  }
  if (cs > 8) {                                 // 16-CTA clusters are a non-portable size
    static std::atomic<unsigned long long> nonportable_set{0};
    if (dev >= 64 || !(nonportable_set.load(std::memory_order_relaxed) & (1ull << dev))) {
      cudaError_t e = cudaFuncSetAttribute(kern, cudaFuncAttributeNonPortableClusterSizeAllowed, 1);
      if (e != cudaSuccess) return e;
      if (dev < 64) nonportable_set.fetch_or(1ull << dev, std::memory_order_relaxed);
    }
  }
  cudaLaunchConfig_t cfg = {};
  cfg.gridDim = dim3(cs, slabs, Z);
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
  cfg.numAttrs = p.no_pdl ? 1 : 2;   // no_pdl: start only after the previous kernel completed
  return cudaLaunchKernelEx(&cfg, kern, tmW, a, geo);
}

}  // namespace decode
}  // namespace gptq
