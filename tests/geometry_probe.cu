// Host-only probe of the decode kernels' launch geometry, used by tests/test_geometry.py: for
// each problem read from stdin ("bits K N M group fold gidx E regs" per line) it prints the
// cluster split and the shared-memory layout that the launcher would choose, using the library's
// own choose_cluster / make_geo / TmaSmem (no kernel is instantiated and no GPU is needed).  The
// one-wave halving and the widening of a split that does not fit are restated here because they
// need the kernel's register count, which the launcher reads from the compiled kernel; the test
// passes the largest one compiled.  The first column says whether the layout fits one CTA (when it
// does not, nothing is launched: gptq_gemm then takes the tensor-core kernel).
#include <cstdio>

#include "decode.cuh"
#include "decode_mma.cuh"

namespace gptq {
const DeviceInfo& device_info() {
  static DeviceInfo d{0, 152, 10, 3, 232448};
  return d;
}
}  // namespace gptq

using namespace gptq;
using namespace gptq::decode;

template <int BITS>
void probe(int K, int N, int M, int group, bool fold, bool gidx, int E, int regs) {
  Problem p = {};
  p.K = K; p.N = N; p.M = M; p.bits = BITS; p.E = E;
  p.group = group; p.G = K / group;
  const int units = K / Pack<BITS>::kPerUnit, slabs = (N + kSlab - 1) / kSlab, sms = 152;
  const int by_regs = regs > 0 ? 65536 / (((regs + 7) & ~7) * kThreads) : 5;
  const int max_per_sm = by_regs < 1 ? 1 : (by_regs > 5 ? 5 : by_regs);
  auto geo_for = [&](int c) {
    return make_geo<BITS>(units, c, M, group, slabs * c * E, sms, max_per_sm, !fold, gidx, p.G);
  };
  const int cs0 = choose_cluster(p, Pack<BITS>::kPerUnit);
  int cs = cs0 < 8 ? cs0 : 8;
  for (int c = cs0; fold && c >= 1; c /= 2) {
    const size_t bytes = (TmaSmem<BITS>::bytes(geo_for(c), M) + 1023) & ~static_cast<size_t>(1023);
    if (bytes > 227 * 1024) break;
    int per_sm = static_cast<int>(233472 / (bytes + 1024));
    per_sm = per_sm < max_per_sm ? per_sm : max_per_sm;
    if (static_cast<long long>(slabs) * c * E <= static_cast<long long>(per_sm) * sms) {
      cs = c;
      break;
    }
  }
  TmaGeo g = geo_for(cs);
  while (TmaSmem<BITS>::bytes(g, M) > kMaxCtaSmem && cs < 16 && units >= 4 * (2 * cs) * kWarps) {
    cs *= 2;
    g = geo_for(cs);
  }
  const int fits = TmaSmem<BITS>::bytes(g, M) <= kMaxCtaSmem;
  printf("%d %d %d %d %d %d %d %d %d %d %d %d %d %d %d %d %zu\n", fits, cs, g.tiles_per_cta, g.chunk_tiles,
         g.chunk_rows, g.slot_bytes, g.chunk_bytes, g.nbuf, g.max_groups, g.full_groups, g.full_k,
         Pack<BITS>::kPerUnit, Pack<BITS>::kRowsPerUnit, units, slabs, (g.tiles_per_cta + g.chunk_tiles - 1) / g.chunk_tiles,
         TmaSmem<BITS>::bytes(g, M));
}

int main() {
  int bits, K, N, M, group, fold, gidx, E, regs;
  while (scanf("%d %d %d %d %d %d %d %d %d", &bits, &K, &N, &M, &group, &fold, &gidx, &E, &regs) == 9) {
    switch (bits) {
      case 2: probe<2>(K, N, M, group, fold, gidx, E, regs); break;
      case 3: probe<3>(K, N, M, group, fold, gidx, E, regs); break;
      case 4: probe<4>(K, N, M, group, fold, gidx, E, regs); break;
      case 8: probe<8>(K, N, M, group, fold, gidx, E, regs); break;
      default: printf("bad\n");
    }
  }
  return 0;
}
