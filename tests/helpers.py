"""Shared test helpers: seeded checkpoints (written by the oracle), device copies, tolerance.

The GEMM acceptance rule, for every element:
    |C - C_ref| <= 2e-3 * sum_k |A[m,k] * w[k,n]| + 1e-3 + ulp/2
with C_ref the oracle's fp32 result and ulp/2 half a unit in the last place of C's dtype (the
one rounding of the result to A's dtype); dequantized weights must match bit for bit.
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


def out_half_ulp(Cref, tol, dtype):
    """Half a unit in the last place of the output dtype (fp16 / bf16) at the magnitude of the
    reference result plus its tolerance: the error of rounding an exact result once to C's dtype."""
    import torch
    mant, emin = {torch.float16: (10, -14), torch.bfloat16: (7, -126)}[dtype]
    mag = np.abs(np.asarray(Cref, dtype=np.float64)) + tol
    e = np.floor(np.log2(np.maximum(mag, np.finfo(np.float64).tiny)))
    return np.exp2(np.maximum(e, emin) - mant) / 2


def assert_gemm_close(C, Cref, B, what=""):
    """C: the library's result as a torch tensor in its output dtype (A's dtype, fp16 or bf16).

    Accept iff |C - C_ref| <= 2e-3 * B + 1e-3 + h element-wise, where h is half a unit in the last
    place of C's dtype at |C_ref|: C is the fp32 result rounded once to that dtype, and that one
    rounding alone may move it by h (2^-9 relative for bf16 -- as much as the 2e-3 bound itself
    when one product dominates the sum, so the bound is taken on top of it)."""
    Cn = np.asarray(C.detach().float().cpu().numpy(), dtype=np.float64)
    tol = RTOL_SUM * np.asarray(B, dtype=np.float64) + ATOL
    err = np.abs(Cn - Cref)
    bound = tol + out_half_ulp(Cref, tol, C.dtype)
    bad = ~(err <= bound)
    if bad.any():
        idx = np.argwhere(bad)[:5]
        raise AssertionError("%s: %d elements outside 2e-3*sum|a*w| + 1e-3 + ulp/2, e.g. %s (max err %g)" % (
            what, int(bad.sum()), [(tuple(int(j) for j in i), float(Cn[tuple(i)]), float(Cref[tuple(i)]))
                                   for i in idx], float(err.max())))
