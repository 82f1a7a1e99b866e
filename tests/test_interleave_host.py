"""Host checks of gptq_prepack_interleave (no GPU): the interleaved layout is a permutation of the
checkpoint's words, each 32-column block contiguous along K, and the lane fragment the decode
kernel loads (lane = 4 g + t: unit t of the k-tile, the 4 columns of quad (g & 1) * 4 + g / 2)
sits at its place.  Words are tagged with their (row, column) so that a misplaced word shows."""
import numpy as np
import pytest

import gptq_bit_weight_gemm_gb300 as g


@pytest.fixture(scope="module", autouse=True)
def _lib():
    from gptq_bit_weight_gemm_gb300 import build as lib_build
    lib_build.build()


@pytest.mark.parametrize("bits,K,N", [(4, 64, 96), (2, 128, 64), (8, 32, 160), (3, 256, 64)])
def test_interleave_places_every_word(bits, K, N):
    rows = K * bits // 32
    r_idx, c_idx = np.meshgrid(np.arange(rows), np.arange(N), indexing="ij")
    qw = (r_idx * 65536 + c_idx).astype(np.int32)            # each word names its own position
    il = g.prepack_interleave(qw, K=K, N=N, bits=bits)
    assert sorted(il.tolist()) == sorted(qw.ravel().tolist())
    R = 3 if bits == 3 else 1
    T = K // (4 * (32 if bits == 3 else 32 // bits))         # k-tiles of 4 units
    assert il.size == (N // 32) * T * R * 32 * 4
    for cb in range(N // 32):
        block = il[cb * T * R * 128:(cb + 1) * T * R * 128]
        assert set((block & 0xFFFF) // 32) == {cb}             # the block holds its columns only
        for kt in range(T):
            for r in range(R):
                frag = block[(kt * R + r) * 128:(kt * R + r + 1) * 128].reshape(32, 4)
                for lane in range(32):
                    gq, t = lane // 4, lane % 4
                    quad = (gq % 2) * 4 + gq // 2
                    assert list(frag[lane] >> 16) == [(kt * 4 + t) * R + r] * 4
                    assert list(frag[lane] & 0xFFFF) == [cb * 32 + quad * 4 + c for c in range(4)]


def test_interleave_refuses_partial_k_tiles():
    with pytest.raises(g.GPTQError):
        g.prepack_interleave(np.zeros((6, 64), np.int32), K=96, N=64, bits=2)   # 2-bit needs K % 64 == 0
    with pytest.raises(g.GPTQError):
        g.prepack_interleave(np.zeros((6, 64), np.int32), K=64, N=64, bits=3)   # 3-bit needs K % 128 == 0
    with pytest.raises(g.GPTQError):
        g.prepack_interleave(np.zeros((4, 48), np.int32), K=32, N=48, bits=4)   # N % 32 != 0
