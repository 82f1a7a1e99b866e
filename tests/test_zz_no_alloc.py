"""gptq_gemm_perm_noalloc: the act-order GEMM for callers that cannot allocate device memory (a
runtime whose allocator already owns the GPU's memory, or code that must not take cudaMalloc's
synchronisation).  Its scratch is a static device buffer inside the library, so it must give the
same result as gptq_gemm_perm with a caller-provided workspace, and stay within the GEMM tolerance
of the oracle -- also on later calls, which find the buffer still holding an earlier call's data.

This file is collected last on purpose; it passes alone in a fresh process as well."""
import ctypes

import numpy as np
import pytest
import torch

import gptq_bit_weight_gemm_gb300 as g
import gptq_inputs
import oracle
from gptq_bit_weight_gemm_gb300 import build as lib_build
from helpers import assert_gemm_close, bits16

pytestmark = pytest.mark.gpu
DEV = "cuda"


def _checkpoint(wl):
    """The act-order checkpoint (oracle writer) and its rows sorted by group (host prepack)."""
    draw = gptq_inputs.draw_weights(wl)
    ck = oracle.make_checkpoint(draw.W, wl.bits, wl.group, draw.g_idx, False, oracle.V2)
    qw2, perm = g.prepack_act_order(ck["qweight"], ck["g_idx"], K=wl.K, N=wl.N, bits=wl.bits,
                                    group=wl.group)
    sc = torch.from_numpy(ck["scales"].view(np.int16)).view(torch.float16).to(DEV)
    return ck, (torch.from_numpy(qw2).to(DEV), torch.from_numpy(ck["qzeros"]).to(DEV), sc,
                torch.from_numpy(perm).to(DEV))


def _noalloc(A, perm, qw, qz, sc, wl):
    M, K = A.shape
    C = torch.full((M, wl.N), float("nan"), dtype=A.dtype, device=DEV)
    p = lambda t: ctypes.c_void_p(t.data_ptr())
    code = g.F16 if A.dtype == torch.float16 else g.BF16
    rc = g.lib().gptq_gemm_perm_noalloc(p(A), M, K, code, p(perm), p(qw), p(qz), p(sc), wl.N, wl.bits,
                                        wl.group, 2, p(C), None)
    assert rc == 0, g.strerror(rc)
    torch.cuda.synchronize()
    return C


@pytest.mark.parametrize("act_dtype", ["f16", "bf16"])
def test_noalloc_matches_oracle_and_gemm_perm_on_consecutive_calls(act_dtype):
    """Calls in a row share the built-in scratch: a 32-token call fills more of it than the 8-token
    call that follows reads, so that second call finds stale data past its own.  Each result must
    be within the GEMM tolerance of the oracle and identical, bit for bit, to gptq_gemm_perm with a
    caller-provided workspace (the same gather and the same deterministic decode)."""
    lib_build.build()
    wl = gptq_inputs.Workload("noalloc", 1024, 544, 4, 128, act_dtype, (8,), ("v2",), seed=17,
                              act_order=True)
    ck, (qw, qz, sc, perm) = _checkpoint(wl)
    for M in (32, 1, 8, 16):
        A = gptq_inputs.draw_activations(wl, M)
        Ad = A.to(DEV)
        C = _noalloc(Ad, perm, qw, qz, sc, wl)
        ref = g.gemm_perm(Ad, perm, qw, qz, sc, bits=wl.bits, group=wl.group)
        torch.cuda.synchronize()
        assert torch.equal(C.view(torch.int16), ref.view(torch.int16)), M
        Cref, B = oracle.gemm(bits16(A), oracle.F16 if act_dtype == "f16" else oracle.BF16, ck["qweight"],
                              ck["qzeros"], ck["scales"], ck["g_idx"], wl.N, wl.bits, wl.group, oracle.V2)
        assert_gemm_close(C, Cref, B, "noalloc M=%d %s" % (M, act_dtype))
    assert g.device_status() == 0


def test_noalloc_rejects_problems_beyond_its_scratch():
    lib_build.build()
    wl = gptq_inputs.Workload("noalloc", 1024, 544, 4, 128, "f16", (8,), ("v2",), seed=17,
                              act_order=True)
    _, (qw, qz, sc, perm) = _checkpoint(wl)
    A = torch.zeros((32, 32768), dtype=torch.float16, device=DEV)   # 2 MiB of gathered activations
    C = torch.empty((32, wl.N), dtype=torch.float16, device=DEV)
    p = lambda t: ctypes.c_void_p(t.data_ptr())
    rc = g.lib().gptq_gemm_perm_noalloc(p(A), 32, 32768, 0, p(perm), p(qw), p(qz), p(sc), wl.N, 4, 128,
                                        2, p(C), None)
    assert rc == -4                            # GPTQ_ERR_WORKSPACE: larger than the built-in scratch
