"""GPU parity for long K at many tokens, where the decode kernels' staged activations outgrow one
CTA's shared memory at the usual K split: the launcher widens the split (up to 16-CTA clusters),
runs 17..32 tokens as two 16-token blocks when one 32-token block fits no CTA, and where even that
does not fit, gptq_gemm runs the tensor-core kernel while the decode-only calls (gptq_gemm_perm,
gptq_gemm_grouped) refuse the shape with GPTQ_ERR_SHAPE.  Shapes follow the down projections of
70B- and 405B-class models (K = 28672, 53248) on a narrow column slice, and K = 98304 for the
refusal."""
import numpy as np
import pytest
import torch

import gptq_bit_weight_gemm_gb300 as g
import gptq_inputs
import oracle
from helpers import assert_gemm_close, bits16

pytestmark = pytest.mark.gpu

DEV = "cuda"
BASE = gptq_inputs.WORKLOADS["llama7b_decode_4bit_g128"]


@pytest.fixture(scope="module", autouse=True)
def _built():
    from gptq_bit_weight_gemm_gb300 import build as lib_build
    lib_build.build()
    assert torch.cuda.is_available()
    yield
    assert g.device_status() == 0


def _checkpoint(K, N, bits, group):
    import dataclasses
    wl = dataclasses.replace(BASE.resized(K, N, (32,), name="long_k_%d_%d_b%d_g%d" % (K, N, bits, group)),
                             bits=bits, group=group)
    draw = gptq_inputs.draw_weights(wl)
    return wl, oracle.make_checkpoint(draw.W, bits, group, None, False, oracle.V2)


def _dev(ck):
    return (torch.from_numpy(ck["qweight"]).to(DEV), torch.from_numpy(ck["qzeros"]).to(DEV),
            torch.from_numpy(ck["scales"].view(np.int16)).view(torch.float16).to(DEV))


@pytest.mark.parametrize("K,bits,group", [
    (16384, 4, 32),      # the usual 8-way split would need 248 KB per CTA: widened to 16
    (28672, 4, 128),     # 70B-class down projection
    (28672, 8, 128),
    (53248, 2, 128),     # 405B-class: two 16-token blocks at a 16-way split
])
def test_gemm_long_k_many_tokens(K, bits, group):
    N, M = 256, 32
    wl, ck = _checkpoint(K, N, bits, group)
    A = gptq_inputs.draw_activations(wl, M)
    qw, qz, sc = _dev(ck)
    C = g.gemm(A.to(DEV), qw, qz, sc, bits=bits, group=group, fmt=g.V2)
    torch.cuda.synchronize()
    Cref, B = oracle.gemm(bits16(A), oracle.F16, ck["qweight"], ck["qzeros"], ck["scales"], None, N, bits,
                          group, oracle.V2)
    assert_gemm_close(C, Cref, B, "K=%d bits=%d group=%d" % (K, bits, group))


@pytest.mark.parametrize("sort_rows", [True, False], ids=["sorted", "per_row"])
def test_gemm_long_k_act_order_on_the_tensor_core_fallback(sort_rows):
    """K = 53248 at 32 tokens fits no 32-token decode layout; the call runs two 16-token blocks or,
    where those do not fit either, the tensor-core kernel.  With act-order it must match the oracle
    both on rows sorted by group on the device (4-column repack strips) and with the per-row-group
    kernels (g_idx)."""
    K, N, M, bits, group = 53248, 256, 32, 4, 128
    import dataclasses
    wl = dataclasses.replace(BASE.resized(K, N, (M,), name="long_k_act"), bits=bits, group=group,
                             act_order=True)
    draw = gptq_inputs.draw_weights(wl)
    ck = oracle.make_checkpoint(draw.W, bits, group, draw.g_idx, False, oracle.V2)
    A = gptq_inputs.draw_activations(wl, M)
    qw, qz, sc = _dev(ck)
    assert g.act_order_workspace_size(M, K, N, bits, group) > 0
    C = g.gemm(A.to(DEV), qw, qz, sc, torch.from_numpy(ck["g_idx"]).to(DEV), bits=bits, group=group,
               fmt=g.V2, sort_rows=sort_rows)
    torch.cuda.synchronize()
    Cref, B = oracle.gemm(bits16(A), oracle.F16, ck["qweight"], ck["qzeros"], ck["scales"], ck["g_idx"], N,
                          bits, group, oracle.V2)
    assert_gemm_close(C, Cref, B, "K=%d act-order" % K)


def test_gemm_perm_long_k_runs_as_two_token_blocks():
    """K = 53248 at 32 tokens: one 32-token block fits no CTA, two 16-token blocks do; the
    decode-only call runs them and matches the oracle."""
    K, N, M, bits, group = 53248, 256, 32, 2, 128
    wl, ck = _checkpoint(K, N, bits, group)
    A = gptq_inputs.draw_activations(wl, M)
    qw, qz, sc = _dev(ck)
    perm = torch.arange(K, dtype=torch.int32, device=DEV)
    C = g.gemm_perm(A.to(DEV), perm, qw, qz, sc, bits=bits, group=group, fmt=g.V2)
    torch.cuda.synchronize()
    Cref, B = oracle.gemm(bits16(A), oracle.F16, ck["qweight"], ck["qzeros"], ck["scales"], None, N, bits,
                          group, oracle.V2)
    assert_gemm_close(C, Cref, B, "gemm_perm K=%d M=%d" % (K, M))


def test_decode_only_calls_refuse_what_fits_no_cta():
    K, N, M, bits, group = 98304, 256, 32, 2, 128
    wl, ck = _checkpoint(K, N, bits, group)
    A = gptq_inputs.draw_activations(wl, M).to(DEV)
    qw, qz, sc = _dev(ck)
    perm = torch.arange(K, dtype=torch.int32, device=DEV)
    with pytest.raises(g.GPTQError) as e:
        g.gemm_perm(A, perm, qw, qz, sc, bits=bits, group=group)
    assert e.value.code == -2
    offsets = torch.tensor([0, M], dtype=torch.int32, device=DEV)
    with pytest.raises(g.GPTQError) as e:
        g.gemm_grouped(A, offsets, qw[None], qz[None], sc[None], bits=bits, group=group, max_m=M)
    assert e.value.code == -2


def test_host_buffer_call_where_the_decode_kernels_decline():
    """gptq_gemm_host with page-locked C: the decode kernels would write C in place, but at K =
    98304 and 32 tokens they take no layout; the call then copies C back from the tensor-core
    kernel's result in C_dev."""
    K, N, M, bits, group = 98304, 256, 32, 2, 128
    wl, ck = _checkpoint(K, N, bits, group)
    A = gptq_inputs.draw_activations(wl, M)
    qw, qz, sc = _dev(ck)
    A_host = A.contiguous().pin_memory()
    C_host = torch.empty((M, N), dtype=A.dtype).pin_memory()
    A_dev = torch.empty((M, K), dtype=A.dtype, device=DEV)
    C_dev = torch.empty((M, N), dtype=A.dtype, device=DEV)
    g.gemm_host(A_host, A_dev, qw, qz, sc, bits=bits, group=group, C_dev=C_dev, C_host=C_host)
    Cref, B = oracle.gemm(bits16(A), oracle.F16, ck["qweight"], ck["qzeros"], ck["scales"], None, N, bits,
                          group, oracle.V2)
    assert_gemm_close(C_host, Cref, B, "host buffers, K=%d" % K)
    assert torch.equal(C_host.view(torch.int16), C_dev.cpu().view(torch.int16))
