"""GPU parity of the interleaved-layout decode path (gptq_prepack_interleave + gptq_gemm_interleaved)
against the CPU oracle, and bit-identity with gptq_gemm / gptq_gemm_perm on the checkpoint's own
layout (the same kernel and launch geometry, only the weight copies and fragment addresses
differ).  Shapes end in ragged column slabs (N = 416: a last slab of 32 columns) and split K over
several CTAs; act-order checkpoints are sorted by group, then interleaved, and multiplied through
the permutation."""
import numpy as np
import pytest
import torch

import gptq_bit_weight_gemm_gb300 as g
import gptq_inputs
import oracle
from helpers import assert_gemm_close, bits16, checkpoint, to_device

pytestmark = pytest.mark.gpu
DEV = "cuda"


@pytest.fixture(scope="module", autouse=True)
def _built():
    from gptq_bit_weight_gemm_gb300 import build as lib_build
    lib_build.build()
    yield
    assert g.device_status() == 0


CASES = [
    # (bits, group, dtype, K, N, Ms)
    (4, 128, "f16", 1024, 416, (1, 8, 16, 32)),
    (4, 128, "bf16", 2048, 288, (1, 5, 16)),
    (2, 64, "bf16", 1024, 416, (1, 8, 32)),
    (3, 128, "f16", 1024, 416, (1, 16, 20)),
    (8, 128, "f16", 512, 288, (1, 9, 32)),
    (8, -1, "bf16", 512, 160, (2, 16)),
]


@pytest.mark.parametrize("case", CASES, ids=lambda c: "b%d_g%d_%s_K%d_N%d" % c[:5])
@pytest.mark.parametrize("fmt", ["v2", "v1"])
def test_interleaved_matches_oracle_and_gptq_gemm(case, fmt):
    bits, group, dt, K, N, Ms = case
    wl = gptq_inputs.Workload("il", K, N, bits, group, dt, Ms, (fmt,), seed=K + N + bits)
    _, ck = checkpoint(wl, fmt)
    qw, qz, sc, _ = to_device(ck)
    il = torch.from_numpy(g.prepack_interleave(ck["qweight"], K=K, N=N, bits=bits)).to(DEV)
    for M in Ms:
        A = gptq_inputs.draw_activations(wl, M)
        C = g.gemm_interleaved(A.to(DEV), il, qz, sc, N=N, bits=bits, group=group, fmt=ck["fmt"])
        ref = g.gemm(A.to(DEV), qw, qz, sc, bits=bits, group=group, fmt=ck["fmt"])
        torch.cuda.synchronize()
        assert torch.equal(C.view(torch.int16), ref.view(torch.int16)), M
        Cref, B = oracle.gemm(bits16(A), oracle.F16 if dt == "f16" else oracle.BF16, ck["qweight"], ck["qzeros"],
                              ck["scales"], None, N, bits, group, ck["fmt"])
        assert_gemm_close(C, Cref, B, "interleaved %s M=%d" % (case, M))


@pytest.mark.parametrize("bits,dt,M", [(3, "f16", 16), (4, "bf16", 1), (2, "f16", 8)])
def test_interleaved_act_order(bits, dt, M):
    wl = gptq_inputs.Workload("il_act", 1024, 416, bits, 128, dt, (M,), ("v2",), seed=bits + M, act_order=True)
    _, ck = checkpoint(wl, "v2")
    qw2, perm = g.prepack_act_order(ck["qweight"], ck["g_idx"], K=wl.K, N=wl.N, bits=bits, group=128)
    il = torch.from_numpy(g.prepack_interleave(qw2, K=wl.K, N=wl.N, bits=bits)).to(DEV)
    _, qz, sc, _ = to_device(ck)
    permd = torch.from_numpy(perm).to(DEV)
    A = gptq_inputs.draw_activations(wl, M)
    C = g.gemm_interleaved(A.to(DEV), il, qz, sc, permd, N=wl.N, bits=bits, group=128)
    ref = g.gemm_perm(A.to(DEV), permd, torch.from_numpy(qw2).to(DEV), qz, sc, bits=bits, group=128)
    torch.cuda.synchronize()
    assert torch.equal(C.view(torch.int16), ref.view(torch.int16))
    Cref, B = oracle.gemm(bits16(A), oracle.F16 if dt == "f16" else oracle.BF16, ck["qweight"], ck["qzeros"],
                          ck["scales"], ck["g_idx"], wl.N, bits, 128, oracle.V2)
    assert_gemm_close(C, Cref, B, "interleaved act-order b%d M=%d" % (bits, M))


def test_interleaved_full_size_llama():
    wl = gptq_inputs.WORKLOADS["llama7b_decode_4bit_g128"]
    _, ck = checkpoint(wl, "v2")
    _, qz, sc, _ = to_device(ck)
    il = torch.from_numpy(g.prepack_interleave(ck["qweight"], K=wl.K, N=wl.N, bits=4)).to(DEV)
    for M in (1, 16):
        A = gptq_inputs.draw_activations(wl, M)
        C = g.gemm_interleaved(A.to(DEV), il, qz, sc, N=wl.N, bits=4, group=128)
        torch.cuda.synchronize()
        Cref, B = oracle.gemm(bits16(A), oracle.F16, ck["qweight"], ck["qzeros"], ck["scales"], None, wl.N, 4, 128,
                              oracle.V2)
        assert_gemm_close(C, Cref, B, "interleaved llama M=%d" % M)


def test_interleaved_refuses_unaligned_groups_and_large_m():
    wl = gptq_inputs.Workload("il_bad", 512, 256, 4, 16, "f16", (4,), ("v2",), seed=1)
    _, ck = checkpoint(wl, "v2")
    _, qz, sc, _ = to_device(ck)
    il = torch.from_numpy(g.prepack_interleave(ck["qweight"], K=512, N=256, bits=4)).to(DEV)
    A = torch.zeros((4, 512), dtype=torch.float16, device=DEV)
    with pytest.raises(g.GPTQError) as e:
        g.gemm_interleaved(A, il, qz, sc, N=256, bits=4, group=16)        # group of half a k-tile
    assert e.value.code == -2
    A = torch.zeros((33, 512), dtype=torch.float16, device=DEV)
    with pytest.raises(g.GPTQError) as e:                                  # the decode kernel only
        g.gemm_interleaved(A, il, qz, sc, N=256, bits=4, group=128)
    assert e.value.code == -2
