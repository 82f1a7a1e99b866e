"""GPU parity of the decode path on wide matrices with few tokens (at least 64 slabs of 128
columns, M <= 8): against the CPU oracle, element by element -- K splits that end in partial
chunks, group -1, both checkpoint formats, fp16 and bf16, raw checkpoints with degenerate columns
and outlier activations, the act-order prepack through the permutation, one-hot rows, and
determinism."""
import numpy as np
import pytest
import torch

import gptq_bit_weight_gemm_gb300 as g
import gptq_inputs
import oracle
from helpers import assert_gemm_close, bits16, checkpoint, to_device
from test_gpu_edge_numerics import activations, raw_checkpoint

pytestmark = pytest.mark.gpu
DEV = "cuda"


@pytest.fixture(scope="module", autouse=True)
def _built():
    from gptq_bit_weight_gemm_gb300 import build as lib_build
    lib_build.build()
    yield
    assert g.device_status() == 0


CASES = [
    # (bits, group, dtype, K, N, Ms): N >= 64 * 128
    (4, 128, "f16", 1024, 8192, (1, 3, 8)),
    (4, 128, "bf16", 1152, 8320, (1, 8)),       # 36 k-tiles: the last chunk is partial; ragged slab
    (4, -1, "f16", 1024, 8192, (1, 5)),
    (2, 64, "f16", 2048, 8192, (1, 8)),
    (2, 64, "bf16", 1024, 8224, (2, 7)),
    (8, 128, "f16", 512, 8192, (1, 8)),
    (3, 128, "f16", 1024, 8192, (1, 4)),
]


@pytest.mark.parametrize("case", CASES, ids=lambda c: "b%d_g%d_%s_K%d_N%d" % c[:5])
@pytest.mark.parametrize("fmt", ["v2", "v1"])
def test_wide_matches_oracle(case, fmt):
    bits, group, dt, K, N, Ms = case
    wl = gptq_inputs.Workload("wide", K, N, bits, group, dt, Ms, (fmt,), seed=K + N + bits)
    _, ck = checkpoint(wl, fmt)
    qw, qz, sc, _ = to_device(ck)
    for M in Ms:
        A = gptq_inputs.draw_activations(wl, M)
        C = g.gemm(A.to(DEV), qw, qz, sc, bits=bits, group=group, fmt=ck["fmt"])
        torch.cuda.synchronize()
        Cref, B = oracle.gemm(bits16(A), oracle.F16 if dt == "f16" else oracle.BF16, ck["qweight"], ck["qzeros"],
                              ck["scales"], None, N, bits, group, ck["fmt"])
        assert_gemm_close(C, Cref, B, "wide %s %s M=%d" % (case, fmt, M))


@pytest.mark.parametrize("bits,dt", [(4, "f16"), (4, "bf16"), (2, "bf16"), (8, "f16")])
def test_wide_degenerate_columns_and_outliers(bits, dt):
    cols = (0, 1, 127, 128, 4095, 8191)
    ck = raw_checkpoint(1024, 8192, bits, 128, oracle.V2, seed=70 + bits, degenerate_cols=cols)
    qw = torch.from_numpy(ck["qweight"]).to(DEV)
    qz = torch.from_numpy(ck["qzeros"]).to(DEV)
    sc = torch.from_numpy(ck["scales"].view(np.int16)).view(torch.float16).to(DEV)
    for M in (1, 8):
        A = activations(M, 1024, dt, seed=M)
        C = g.gemm(A.to(DEV), qw, qz, sc, bits=bits, group=128, fmt=oracle.V2)
        torch.cuda.synchronize()
        Cref, B = oracle.gemm(bits16(A), oracle.F16 if dt == "f16" else oracle.BF16, ck["qweight"], ck["qzeros"],
                              ck["scales"], None, 8192, bits, 128, oracle.V2)
        assert_gemm_close(C, Cref, B, "wide raw b%d %s M=%d" % (bits, dt, M))
        assert np.all(Cref[:, list(cols)] == 0.0)


def test_wide_act_order_prepacked_and_deterministic():
    wl = gptq_inputs.Workload("wide_act", 1024, 8192, 4, 128, "f16", (1,), ("v2",), seed=9, act_order=True)
    _, ck = checkpoint(wl, "v2")
    qw2, perm = g.prepack_act_order(ck["qweight"], ck["g_idx"], K=wl.K, N=wl.N, bits=4, group=128)
    _, qz, sc, _ = to_device(ck)
    q2, permd = torch.from_numpy(qw2).to(DEV), torch.from_numpy(perm).to(DEV)
    for M in (1, 6):
        A = gptq_inputs.draw_activations(wl, M)
        C = g.gemm_perm(A.to(DEV), permd, q2, qz, sc, bits=4, group=128)
        C2 = g.gemm_perm(A.to(DEV), permd, q2, qz, sc, bits=4, group=128)
        torch.cuda.synchronize()
        assert torch.equal(C.view(torch.int16), C2.view(torch.int16))
        Cref, B = oracle.gemm(bits16(A), oracle.F16, ck["qweight"], ck["qzeros"], ck["scales"], ck["g_idx"], wl.N, 4,
                              128, oracle.V2)
        assert_gemm_close(C, Cref, B, "wide act-order M=%d" % M)


def test_wide_one_hot_rows_bit_exact():
    """One-hot rows make each output a single dequantized weight (exact fp32 product, one rounding)."""
    wl = gptq_inputs.Workload("wide_id", 512, 8192, 4, 64, "f16", (8,), ("v2",), seed=3)
    _, ck = checkpoint(wl, "v2")
    qw, qz, sc, _ = to_device(ck)
    W = g.dequant(qw, qz, sc, K=512, bits=4, group=64)
    rows = np.array([0, 1, 63, 64, 200, 255, 256, 511])
    A = torch.zeros((8, 512), dtype=torch.float16)
    A[np.arange(8), rows] = 1.0
    C = g.gemm(A.to(DEV), qw, qz, sc, bits=4, group=64)
    torch.cuda.synchronize()
    assert torch.equal(C.view(torch.int16), W[torch.from_numpy(rows).to(DEV)].view(torch.int16))
