"""Shared test helpers: seeded checkpoints (written by the oracle), device copies, tolerance.

The GEMM acceptance rule is the one the task states for every element:
    |C - C_ref| <= 2e-3 * sum_k |A[m,k] * w[k,n]| + 1e-3
with C_ref the oracle's fp32 result; dequantized weights must match bit for bit.
"""
import functools

import numpy as np

import gptq_inputs
import oracle

RTOL_SUM = 2e-3
ATOL = 1e-3
FMT = {"v1": oracle.V1, "v2": oracle.V2}


def dtype_code(wl):
    return oracle.F16 if wl.act_dtype == "f16" else oracle.BF16


@functools.lru_cache(maxsize=16)
def checkpoint(wl, fmt="v2"):
    """(draw, checkpoint dict) for a workload, quantized and packed by the oracle."""
    draw = gptq_inputs.draw_weights(wl)
    ck = oracle.make_checkpoint(draw.W, wl.bits, wl.group, draw.g_idx, wl.sym, FMT[fmt])
    return draw, ck


def to_device(ck, device="cuda"):
    import torch
    qw = torch.from_numpy(ck["qweight"]).to(device)
    qz = torch.from_numpy(ck["qzeros"]).to(device)
    sc = torch.from_numpy(ck["scales"].view(np.int16)).view(torch.float16).to(device)
    gi = None if ck["g_idx"] is None else torch.from_numpy(ck["g_idx"]).to(device)
    return qw, qz, sc, gi


def bits16(t):
    import torch
    return t.detach().cpu().contiguous().view(torch.int16).numpy().view(np.uint16)


def assert_gemm_close(C, Cref, B, what=""):
    C = np.asarray(C, dtype=np.float64)
    err = np.abs(C - Cref)
    bound = RTOL_SUM * B + ATOL
    bad = ~(err <= bound)
    if bad.any():
        idx = np.argwhere(bad)[:5]
        raise AssertionError("%s: %d elements outside 2e-3*sum|a*w| + 1e-3, e.g. %s (max err %g)" % (
            what, int(bad.sum()), [(tuple(i), float(C[tuple(i)]), float(Cref[tuple(i)])) for i in idx],
            float(err.max())))
