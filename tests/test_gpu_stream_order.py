"""A checkpoint written on the stream right before a GEMM: gptq_quantize_rtn rewrites the same
device buffers and gptq_gemm multiplies them at once, with no synchronisation in between, on one
stream.  The GEMM kernels start reading the checkpoint before their dependency wait (programmatic
dependent launch), so this holds only because the writer ends with an ordering step; every
product is checked against the oracle run on the checkpoint the oracle's own writer makes from
the same weights (bit-identical to the GPU writer, see test_quantizer_bit_exact_full)."""
import numpy as np
import pytest
import torch

import gptq_bit_weight_gemm_gb300 as g
import oracle
from helpers import assert_gemm_close, bits16

pytestmark = pytest.mark.gpu
DEV = "cuda"


@pytest.mark.parametrize("bits,group,fmt", [(4, 128, oracle.V2), (3, 128, oracle.V1), (8, 64, oracle.V2)])
def test_quantize_then_gemm_without_synchronize(bits, group, fmt):
    from gptq_bit_weight_gemm_gb300 import build as lib_build
    lib_build.build()
    K, N = 4096, 4096
    G = K // group
    stream = torch.cuda.Stream()
    qw = torch.empty((K * bits // 32, N), dtype=torch.int32, device=DEV)
    qz = torch.empty((G, N * bits // 32), dtype=torch.int32, device=DEV)
    sc = torch.empty((G, N), dtype=torch.float16, device=DEV)
    rng = np.random.default_rng(bits)
    Ws = [(rng.standard_normal((K, N), dtype=np.float32) * np.float32(0.02)) for _ in range(3)]
    As = {M: torch.from_numpy(rng.standard_normal((M, K), dtype=np.float32)).to(torch.float16)
          for M in (1, 16, 64)}
    Wd = [torch.from_numpy(W).to(DEV) for W in Ws]
    Ad = {M: A.to(DEV) for M, A in As.items()}
    torch.cuda.synchronize()
    outs = []
    with torch.cuda.stream(stream):
        for W in Wd:
            g.quantize_rtn(W, bits=bits, group=group, fmt=fmt, out=(qw, qz, sc), stream=stream)
            outs.append({M: g.gemm(A, qw, qz, sc, bits=bits, group=group, fmt=fmt, stream=stream)
                         for M, A in Ad.items()})
    stream.synchronize()
    for W, got in zip(Ws, outs):
        ck = oracle.make_checkpoint(W, bits, group, None, False, fmt)
        for M, A in As.items():
            Cref, B = oracle.gemm(bits16(A), oracle.F16, ck["qweight"], ck["qzeros"], ck["scales"], None,
                                  N, bits, group, fmt)
            assert_gemm_close(got[M], Cref, B, "bits=%d M=%d" % (bits, M))
    assert g.device_status() == 0
