// Host-only probe of the decode kernels' launch geometry, used by tests/test_geometry.py: for
// each problem read from stdin ("bits K N M group fold gidx E regs" per line) it prints the
// cluster split and the shared-memory layout that the launcher chooses, by calling the
// launcher's own select_geometry (no kernel is instantiated and no GPU is needed).  The register
// count, which the launcher reads from the compiled kernel, is an input; the test passes the
// smallest and the largest one compiled.  The first column says whether the layout fits one CTA
// (when it does not, nothing is launched: gptq_gemm then takes the tensor-core kernel).
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
  static const int32_t dummy = 0;                      // only compared against nullptr
  Problem p = {};
  p.K = K; p.N = N; p.M = M; p.bits = BITS; p.E = E;
  p.group = group; p.G = K / group;
  p.g_idx = gidx ? &dummy : nullptr;
  const int units = K / Pack<BITS>::kPerUnit, slabs = (N + kSlab - 1) / kSlab;
  const GeoChoice c = select_geometry<BITS>(p, fold, regs, device_info().sm_count, E);
  const TmaGeo& g = c.geo;
  printf("%d %d %d %d %d %d %d %d %d %d %d %d %d %d %d %d %zu\n", c.fits ? 1 : 0, c.cs, g.tiles_per_cta,
         g.chunk_tiles, g.chunk_rows, g.slot_bytes, g.chunk_bytes, g.nbuf, g.max_groups, g.full_groups, g.full_k,
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
