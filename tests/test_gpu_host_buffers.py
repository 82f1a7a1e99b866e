"""GPU parity of gptq_gemm_host: gptq_gemm (page "增强 vLLM 对 GPTQv2 格式的支持：分析与实现",
section "调整细节：根据格式选择处理方式") with the activations read from host memory and the result
written to host memory inside the call.  Checked against the oracle at the GEMM's tolerance, and
against gptq_gemm on device buffers bit for bit (the same kernels run); page-locked and pageable
host memory; the decode and tensor-core kernels, fp16 and bf16, act-order."""
import pytest
import torch

import gptq_bit_weight_gemm_gb300 as g
import gptq_inputs
import oracle
from helpers import assert_gemm_close, bits16, checkpoint, dtype_code, to_device

pytestmark = pytest.mark.gpu

DEV = "cuda"


@pytest.fixture(scope="module", autouse=True)
def _built():
    from gptq_bit_weight_gemm_gb300 import build as lib_build
    lib_build.build()
    assert torch.cuda.is_available()
    yield
    assert g.device_status() == 0


CASES = [
    # (bits, group, dtype, M, K, N, act_order)
    (4, 128, "f16", 1, 1024, 544, False),
    (3, 128, "bf16", 7, 640, 416, False),
    (2, 64, "f16", 32, 512, 288, False),
    (8, 128, "bf16", 48, 384, 160, False),
    (4, 64, "f16", 2, 512, 352, True),
]


@pytest.mark.parametrize("case", CASES, ids=lambda c: "b%d_g%d_%s_M%d_K%d_N%d_ao%d" % c)
@pytest.mark.parametrize("pinned", [True, False], ids=["pinned", "pageable"])
def test_host_buffers_match_oracle_and_device_call(case, pinned):
    bits, group, dt, M, K, N, act_order = case
    wl = gptq_inputs.Workload("host", K, N, bits, group, dt, (M,), ("v2",), seed=M * 7 + bits,
                              act_order=act_order)
    _, ck = checkpoint(wl, "v2")
    qw, qz, sc, gi = to_device(ck)
    A = gptq_inputs.draw_activations(wl, M)
    A_host = A.contiguous()
    C_host = torch.empty((M, N), dtype=A.dtype)
    if pinned:
        A_host = A_host.pin_memory()
        C_host = C_host.pin_memory()
    A_dev = torch.empty((M, K), dtype=A.dtype, device=DEV)
    C_dev = torch.empty((M, N), dtype=A.dtype, device=DEV)
    size = g.act_order_workspace_size(M, K, N, bits, group) if act_order else 0
    if size == 0 and A.dtype == torch.bfloat16:
        size = g.workspace_size(M, K, N, bits, group)
    ws = torch.empty(max(size, 1), dtype=torch.uint8, device=DEV) if size else None
    out = g.gemm_host(A_host, A_dev, qw, qz, sc, gi, bits=bits, group=group, C_dev=C_dev, C_host=C_host,
                      workspace=ws)
    assert out.data_ptr() == C_host.data_ptr()
    Cref, B = oracle.gemm(bits16(A), dtype_code(wl), ck["qweight"], ck["qzeros"], ck["scales"], ck["g_idx"],
                          N, bits, group, ck["fmt"])
    assert_gemm_close(C_host, Cref, B, "gemm_host %s" % (case,))
    C_ref_dev = g.gemm(A.to(DEV), qw, qz, sc, gi, bits=bits, group=group, workspace=ws)
    torch.cuda.synchronize()
    assert torch.equal(C_host.view(torch.int16), C_ref_dev.cpu().view(torch.int16))


def test_empty_problem_and_validation_errors():
    K, N, bits, group = 256, 128, 4, 64
    wl = gptq_inputs.Workload("host", K, N, bits, group, "f16", (1,), ("v2",), seed=3)
    _, ck = checkpoint(wl, "v2")
    qw, qz, sc, _ = to_device(ck)
    A_dev = torch.empty((1, K), dtype=torch.float16, device=DEV)
    C_dev = torch.empty((1, N), dtype=torch.float16, device=DEV)
    # M = 0: nothing to do
    out = g.gemm_host(torch.empty((0, K), dtype=torch.float16), A_dev, qw, qz, sc, bits=bits, group=group,
                      C_dev=C_dev, C_host=torch.empty((0, N), dtype=torch.float16))
    assert out.numel() == 0
    # a group size that does not divide K: gptq_gemm's own check, reported through the host call
    # before anything is copied (the staging buffer keeps its contents)
    A_dev.fill_(-3.0)
    with pytest.raises(g.GPTQError):
        g.gemm_host(torch.ones((1, K), dtype=torch.float16), A_dev, qw, qz, sc, bits=bits, group=96,
                    C_dev=C_dev, C_host=torch.empty((1, N), dtype=torch.float16))
    torch.cuda.synchronize()
    assert bool((A_dev == -3.0).all())
    # staging buffers of the wrong dtype or size are refused before the call
    with pytest.raises(TypeError):
        g.gemm_host(torch.ones((1, K), dtype=torch.float16), A_dev.to(torch.bfloat16), qw, qz, sc, bits=bits,
                    group=group, C_dev=C_dev, C_host=torch.empty((1, N), dtype=torch.float16))
    with pytest.raises(ValueError):
        g.gemm_host(torch.ones((2, K), dtype=torch.float16), A_dev, qw, qz, sc, bits=bits, group=group,
                    C_dev=C_dev, C_host=torch.empty((2, N), dtype=torch.float16))
    assert g.device_status() == 0


@pytest.mark.parametrize("named_stream", [False, True], ids=["default_stream", "captured_plan"])
def test_prepared_call_reruns_on_new_host_contents(named_stream):
    """HostGemm prepares the call once (on a named stream: a captured graph); each call takes the
    host buffer's current contents."""
    K, N, bits, group = 1024, 544, 4, 128
    stream = torch.cuda.Stream() if named_stream else None
    wl = gptq_inputs.Workload("host", K, N, bits, group, "f16", (3,), ("v2",), seed=11)
    _, ck = checkpoint(wl, "v2")
    qw, qz, sc, _ = to_device(ck)
    A_host = torch.empty((3, K), dtype=torch.float16).pin_memory()
    C_host = torch.empty((3, N), dtype=torch.float16).pin_memory()
    A_dev = torch.empty((3, K), dtype=torch.float16, device=DEV)
    C_dev = torch.empty((3, N), dtype=torch.float16, device=DEV)
    call = g.HostGemm(A_host, A_dev, qw, qz, sc, bits=bits, group=group, C_dev=C_dev, C_host=C_host,
                      stream=stream)
    assert (call._plan is not None) == named_stream
    for seed in (1, 2, 3):
        wl_s = gptq_inputs.Workload("host", K, N, bits, group, "f16", (3,), ("v2",), seed=seed)
        A = gptq_inputs.draw_activations(wl_s, 3)
        A_host.copy_(A)
        out = call()
        assert out is C_host
        Cref, B = oracle.gemm(bits16(A), dtype_code(wl), ck["qweight"], ck["qzeros"], ck["scales"], None,
                              N, bits, group, ck["fmt"])
        assert_gemm_close(C_host, Cref, B, "prepared call, activations %d" % seed)


@pytest.mark.parametrize("case", [(4, 128, "f16", 16, 1024, 544), (8, 128, "bf16", 48, 384, 160),
                                  (2, 64, "bf16", 5, 512, 288)], ids=lambda c: "b%d_g%d_%s_M%d_K%d_N%d" % c)
def test_captured_plan_matches_the_direct_call(case):
    """The captured plan replays exactly gptq_gemm_host's work: the same bits, for the decode and
    the tensor-core kernels (bf16 prefill with its workspace), run after run."""
    bits, group, dt, M, K, N = case
    wl = gptq_inputs.Workload("host", K, N, bits, group, dt, (M,), ("v2",), seed=M + bits)
    _, ck = checkpoint(wl, "v2")
    qw, qz, sc, _ = to_device(ck)
    A = gptq_inputs.draw_activations(wl, M)
    A_host = A.contiguous().pin_memory()
    C_host = torch.empty((M, N), dtype=A.dtype).pin_memory()
    A_dev = torch.empty((M, K), dtype=A.dtype, device=DEV)
    C_dev = torch.empty((M, N), dtype=A.dtype, device=DEV)
    size = g.workspace_size(M, K, N, bits, group) if A.dtype == torch.bfloat16 else 0
    ws = torch.empty(size, dtype=torch.uint8, device=DEV) if size else None
    stream = torch.cuda.Stream()
    direct = g.gemm_host(A_host, A_dev, qw, qz, sc, bits=bits, group=group, C_dev=C_dev,
                         C_host=torch.empty((M, N), dtype=A.dtype).pin_memory(), workspace=ws, stream=stream).clone()
    call = g.HostGemm(A_host, A_dev, qw, qz, sc, bits=bits, group=group, C_dev=C_dev, C_host=C_host, workspace=ws,
                      stream=stream)
    assert call._plan is not None
    for _ in range(3):
        C_host.zero_()
        call()
        assert torch.equal(C_host.view(torch.int16), direct.view(torch.int16))
    Cref, B = oracle.gemm(bits16(A), dtype_code(wl), ck["qweight"], ck["qzeros"], ck["scales"], None, N, bits,
                          group, ck["fmt"])
    assert_gemm_close(C_host, Cref, B, "captured plan %s" % (case,))
    call.close()
