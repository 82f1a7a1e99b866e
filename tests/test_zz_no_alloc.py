"""gptq_gemm_perm_noalloc: the act-order GEMM for callers that cannot allocate device memory (a
runtime whose allocator already owns the GPU's memory, or code that must not take cudaMalloc's
synchronisation).  Its scratch is a static device buffer inside the library, so it must give the
same result as gptq_gemm_perm with a caller-provided workspace -- also on a second call, which
finds the buffer still holding the first call's data.

This file is collected last on purpose; it passes alone in a fresh process as well."""
import ctypes

import numpy as np
import pytest
import torch

import gptq_bit_weight_gemm_gb300 as g
import gptq_inputs
from gptq_bit_weight_gemm_gb300 import build as lib_build

pytestmark = pytest.mark.gpu
DEV = "cuda"


def _prepacked(wl):
    draw = gptq_inputs.draw_weights(wl)
    W = torch.from_numpy(draw.W).to(DEV)
    gi = torch.from_numpy(draw.g_idx).to(DEV)
    qw, qz, sc = g.quantize_rtn(W, bits=wl.bits, group=wl.group, g_idx=gi)
    qw2, perm = g.prepack_act_order(qw.cpu().numpy(), draw.g_idx, K=wl.K, N=wl.N, bits=wl.bits,
                                    group=wl.group)
    return torch.from_numpy(qw2).to(DEV), qz, sc, torch.from_numpy(perm).to(DEV)


def _noalloc(A, perm, qw, qz, sc, wl):
    M, K = A.shape
    C = torch.full((M, wl.N), float("nan"), dtype=A.dtype, device=DEV)
    p = lambda t: ctypes.c_void_p(t.data_ptr())
    rc = g.lib().gptq_gemm_perm_noalloc(p(A), M, K, 0, p(perm), p(qw), p(qz), p(sc), wl.N, wl.bits,
                                        wl.group, 2, p(C), None)
    assert rc == 0, g.strerror(rc)
    torch.cuda.synchronize()
    return C


def test_noalloc_matches_gemm_perm_on_two_calls():
    lib_build.build()
    wl = gptq_inputs.Workload("noalloc", 1024, 544, 4, 128, "f16", (8,), ("v2",), seed=17,
                              act_order=True)
    qw, qz, sc, perm = _prepacked(wl)
    W = g.dequant(qw, qz, sc, K=wl.K, bits=wl.bits, group=wl.group).float()
    for M in (8, 16):                         # two calls in a row, different tokens
        A = gptq_inputs.draw_activations(wl, M).to(DEV)
        ref = g.gemm_perm(A, perm, qw, qz, sc, bits=wl.bits, group=wl.group)
        C = _noalloc(A, perm, qw, qz, sc, wl)
        B = A[:, perm.long()].float().abs() @ W.abs()          # sum_k |a_k w_k|
        err = (C.float() - ref.float()).abs()
        assert torch.isfinite(C).all()
        assert bool((err <= 2e-3 * B + 1e-3).all()), float(err.max())
    assert g.device_status() == 0


def test_noalloc_rejects_problems_beyond_its_scratch():
    lib_build.build()
    wl = gptq_inputs.Workload("noalloc", 1024, 544, 4, 128, "f16", (8,), ("v2",), seed=17,
                              act_order=True)
    qw, qz, sc, perm = _prepacked(wl)
    A = torch.zeros((32, 32768), dtype=torch.float16, device=DEV)   # 2 MiB of gathered activations
    C = torch.empty((32, wl.N), dtype=torch.float16, device=DEV)
    p = lambda t: ctypes.c_void_p(t.data_ptr())
    rc = g.lib().gptq_gemm_perm_noalloc(p(A), 32, 32768, 0, p(perm), p(qw), p(qz), p(sc), wl.N, 4, 128,
                                        2, p(C), None)
    assert rc == -4                            # GPTQ_ERR_WORKSPACE: larger than the built-in scratch
