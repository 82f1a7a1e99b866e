"""GPU parity: the CUDA library (through the C ABI) against the CPU oracle on the same seeded
inputs.  Dequantized weights and quantizer outputs must match bit for bit; GEMM outputs must be
within |C - C_ref| <= 2e-3 * sum_k |a*w| + 1e-3 of the oracle's fp32 result, element by element.

Sizes: every workload at its full size (decode workloads compared on every output, the
M = 4096 prefill workloads on sampled rows), plus oracle-sized cases that span several tiles
and end in ragged tails, and the degenerate cases (M = 0, one tile, out-of-range g_idx)."""
import numpy as np
import pytest
import torch

import gptq_bit_weight_gemm_gb300 as g
import gptq_inputs
import oracle
from helpers import FMT, assert_gemm_close, bits16, checkpoint, dtype_code, to_device

pytestmark = pytest.mark.gpu

WL = gptq_inputs.WORKLOADS
DEV = "cuda"


@pytest.fixture(scope="module", autouse=True)
def _built():
    from gptq_bit_weight_gemm_gb300 import build as lib_build
    lib_build.build()
    assert torch.cuda.is_available()
    yield
    assert g.device_status() == 0


def _gpu_gemm(wl, ck, A):
    qw, qz, sc, gi = to_device(ck)
    C = g.gemm(A.to(DEV), qw, qz, sc, gi, bits=wl.bits, group=wl.group, fmt=ck["fmt"])
    torch.cuda.synchronize()
    return C


def _oracle_gemm(wl, ck, A, rows=None):
    return oracle.gemm(bits16(A), dtype_code(wl), ck["qweight"], ck["qzeros"], ck["scales"],
                       ck["g_idx"], wl.N, wl.bits, wl.group, ck["fmt"], rows=rows)


# ------------------------------------------------------------------------------ dequant
@pytest.mark.parametrize("name", list(WL))
@pytest.mark.parametrize("fmt", ["v2", "v1"])
def test_dequant_bit_exact_full(name, fmt):
    wl = WL[name]
    _, ck = checkpoint(wl, fmt)
    qw, qz, sc, gi = to_device(ck)
    w32 = oracle.dequant_f32(ck["qweight"], ck["qzeros"], ck["scales"], ck["g_idx"], wl.K, wl.N,
                             wl.bits, wl.group, FMT[fmt])
    for dt, code in ((torch.float16, oracle.F16), (torch.bfloat16, oracle.BF16)):
        W = g.dequant(qw, qz, sc, gi, K=wl.K, bits=wl.bits, group=wl.group, fmt=FMT[fmt], dtype=dt)
        ref = oracle.round_to(w32, code)
        got = bits16(W)
        if not np.array_equal(got, ref):
            bad = np.argwhere(got != ref)[:5]
            raise AssertionError("%s %s %s: %d mismatches, e.g. %s" % (
                name, fmt, dt, int((got != ref).sum()), bad.tolist()))


# ------------------------------------------------------------------------------ quantizer
@pytest.mark.parametrize("name", list(WL))
@pytest.mark.parametrize("fmt", ["v2", "v1"])
def test_quantizer_bit_exact_full(name, fmt):
    wl = WL[name]
    draw, ck = checkpoint(wl, fmt)
    gi = None if draw.g_idx is None else torch.from_numpy(draw.g_idx).to(DEV)
    qw, qz, sc = g.quantize_rtn(torch.from_numpy(draw.W).to(DEV), bits=wl.bits, group=wl.group,
                                g_idx=gi, sym=wl.sym, fmt=FMT[fmt])
    assert np.array_equal(bits16(sc), ck["scales"]), name
    assert np.array_equal(qz.cpu().numpy(), ck["qzeros"]), name
    assert np.array_equal(qw.cpu().numpy(), ck["qweight"]), name


# ------------------------------------------------------------------------------ GEMM, full size
DECODE_CASES = [(n, M, f) for n in WL for M in WL[n].Ms for f in WL[n].fmts if M <= 16]


@pytest.mark.parametrize("name,M,fmt", DECODE_CASES)
def test_decode_gemm_full(name, M, fmt):
    wl = WL[name]
    _, ck = checkpoint(wl, fmt)
    A = gptq_inputs.draw_activations(wl, M)
    C = _gpu_gemm(wl, ck, A)
    Cref, B = _oracle_gemm(wl, ck, A)
    assert_gemm_close(C, Cref, B, "%s M=%d %s" % (name, M, fmt))


LARGE_CASES = [(n, M, f) for n in WL for M in WL[n].Ms for f in WL[n].fmts if M > 16]


@pytest.mark.parametrize("name,M,fmt", LARGE_CASES)
def test_large_m_gemm_full_sampled_rows(name, M, fmt):
    wl = WL[name]
    _, ck = checkpoint(wl, fmt)
    A = gptq_inputs.draw_activations(wl, M)
    C = _gpu_gemm(wl, ck, A)
    rng = np.random.default_rng(M)
    fixed = [0, 1, 127, 128, 255, M // 2, M - 1]
    rows = np.unique(np.concatenate([[r for r in fixed if r < M],
                                     rng.choice(M, size=min(M, 24), replace=False)])).astype(np.int32)
    Cref, B = _oracle_gemm(wl, ck, A, rows=rows)
    assert_gemm_close(C[torch.from_numpy(rows).long().to(DEV)], Cref, B,
                      "%s M=%d %s" % (name, M, fmt))


# ------------------------------------------------------------------------------ GEMM, oracle-sized
SMALL = [
    # (bits, group, act_order, dtype, M, K, N)
    (4, 128, False, "f16", 1, 512, 352),
    (4, 64, False, "bf16", 3, 256, 160),
    (2, 64, False, "bf16", 7, 1024, 544),
    (3, 128, True, "f16", 16, 640, 416),
    (3, 32, False, "bf16", 5, 96, 96),
    (8, 128, False, "f16", 9, 384, 288),
    (8, 128, False, "bf16", 2, 384, 288),
    (8, -1, False, "bf16", 12, 256, 224),
    (4, -1, False, "f16", 16, 1024, 1056),
    (2, 16, True, "f16", 4, 512, 128),
    (4, 16, False, "f16", 6, 64, 64),
    (4, 128, False, "bf16", 37, 640, 800),
    (4, 128, True, "f16", 130, 512, 544),
    (8, 128, False, "bf16", 200, 384, 288),
    (2, 64, False, "f16", 300, 576, 800),
    (3, 128, True, "bf16", 129, 1024, 288),
    (4, -1, False, "bf16", 257, 256, 1024),
    (4, 128, False, "f16", 24, 640, 416),
    (2, 64, False, "bf16", 32, 512, 288),
    (3, 128, True, "f16", 20, 640, 288),
    (8, 128, False, "bf16", 31, 384, 160),
    # narrow and deep: 16-CTA clusters
    (4, 128, False, "f16", 1, 4096, 256),
    (2, 64, False, "bf16", 8, 4096, 640),
    (3, 128, True, "f16", 4, 4096, 128),
]


@pytest.mark.parametrize("case", SMALL, ids=lambda c: "b%d_g%d_%s_%s_M%d_K%d_N%d" % (
    c[0], c[1], "act" if c[2] else "seq", c[3], c[4], c[5], c[6]))
@pytest.mark.parametrize("fmt", ["v2", "v1"])
def test_gemm_oracle_sized(case, fmt):
    bits, group, act, dt, M, K, N = case
    wl = gptq_inputs.Workload("small", K, N, bits, group, dt, (M,), (fmt,), seed=M * 7 + bits,
                              act_order=act, sym=(bits == 8 and group == -1))
    _, ck = checkpoint(wl, fmt)
    A = gptq_inputs.draw_activations(wl, M)
    C = _gpu_gemm(wl, ck, A)
    Cref, B = _oracle_gemm(wl, ck, A)
    assert_gemm_close(C, Cref, B, str(case))


# ------------------------------------------------------------------------------ pins on the GPU
def test_identity_gives_dequant_bit_exact():
    """gemm(A = I) equals gptq_dequant bit for bit (fp32 accumulation of one nonzero term).  The
    tensor-core kernel multiplies the weight rounded to fp16 for both activation types, so with
    bf16 activations its identity product is that fp16 weight rounded to bf16 (computed here by
    the oracle); the decode kernel's folded path keeps the exact product and matches the bf16
    dequant itself."""
    wl = WL["tiny_4bit_g64"]
    for fmt in ("v2", "v1"):
        _, ck = checkpoint(wl, fmt)
        qw, qz, sc, gi = to_device(ck)
        for dt in (torch.float16, torch.bfloat16):
            I = torch.eye(wl.K, dtype=dt, device=DEV)
            C = g.gemm(I, qw, qz, sc, bits=wl.bits, group=wl.group, fmt=FMT[fmt])
            W = g.dequant(qw, qz, sc, K=wl.K, bits=wl.bits, group=wl.group, fmt=FMT[fmt], dtype=dt)
            if dt == torch.float16:
                assert torch.equal(C.view(torch.int16), W.view(torch.int16)), (fmt, dt)
            else:
                w16 = oracle.dequant(ck["qweight"], ck["qzeros"], ck["scales"], None, wl.K, wl.N, wl.bits,
                                     wl.group, FMT[fmt], oracle.F16)
                exp = oracle.round_to(oracle.to_double(w16, oracle.F16).astype(np.float32), oracle.BF16)
                assert np.array_equal(bits16(C), exp), (fmt, dt)
            for M in (1, 5, 16):   # one-hot rows through the decode kernel
                C1 = g.gemm(I[:M].contiguous(), qw, qz, sc, bits=wl.bits, group=wl.group,
                            fmt=FMT[fmt])
                assert torch.equal(C1.view(torch.int16), W[:M].view(torch.int16)), (fmt, dt, M)


def test_v1_and_v2_give_identical_results():
    """Zeros >= 1 encode the same dequantization in both formats: identical bits on the GPU."""
    wl = WL["llama7b_decode_4bit_g128"]
    _, c2 = checkpoint(wl, "v2")
    _, c1 = checkpoint(wl, "v1")
    assert c2["zero"].min() >= 1
    for M in (1, 16, 64):
        A = gptq_inputs.draw_activations(wl, M).to(DEV)
        outs = []
        for ck in (c1, c2):
            qw, qz, sc, _ = to_device(ck)
            outs.append(g.gemm(A, qw, qz, sc, bits=4, group=128, fmt=ck["fmt"]))
        assert torch.equal(outs[0], outs[1]), M


def test_act_order_permutation_invariance():
    wl = WL["act_order_3bit_g128"].resized(1024, 416, (16,))
    draw, ck = checkpoint(wl, "v2")
    A = gptq_inputs.draw_activations(wl, 16)
    C = _gpu_gemm(wl, ck, A)
    p = np.random.default_rng(1).permutation(wl.K)
    ck_p = dict(ck)
    ck_p["qweight"] = oracle.pack_k(ck["q"][p], wl.bits)
    ck_p["g_idx"] = np.ascontiguousarray(ck["g_idx"][p])
    A_p = A[:, torch.from_numpy(p)].contiguous()
    C_p = _gpu_gemm(wl, ck_p, A_p)
    Cref, B = _oracle_gemm(wl, ck, A)
    assert_gemm_close(C_p, Cref, B, "permuted")
    assert_gemm_close(C, Cref, B, "original")
    qw, qz, sc, gi = to_device(ck)
    qwp, _, _, gip = to_device(ck_p)
    W = g.dequant(qw, qz, sc, gi, K=wl.K, bits=3, group=128, fmt=2)
    Wp = g.dequant(qwp, qz, sc, gip, K=wl.K, bits=3, group=128, fmt=2)
    assert torch.equal(Wp.view(torch.int16), W[torch.from_numpy(p).to(DEV)].view(torch.int16))


# ------------------------------------------------------------------------------ prepacked act-order
PERM_CASES = [
    # (bits, group, dtype, M, K, N): act-order checkpoints, rows sorted by group on the host
    (3, 128, "f16", 16, 640, 416),
    (3, 128, "bf16", 20, 640, 288),
    (2, 16, "f16", 4, 512, 128),
    (2, 64, "bf16", 13, 1024, 160),
    (4, 128, "f16", 1, 1024, 544),
    (4, 64, "bf16", 8, 512, 352),
    (8, 128, "f16", 32, 384, 288),
    (8, 128, "bf16", 3, 384, 160),
]


def _gemm_perm(wl, ck, A):
    qw2, perm = g.prepack_act_order(ck["qweight"], ck["g_idx"], K=wl.K, N=wl.N, bits=wl.bits,
                                    group=wl.group)
    _, qz, sc, _ = to_device(ck)
    C = g.gemm_perm(A.to(DEV), torch.from_numpy(perm).to(DEV), torch.from_numpy(qw2).to(DEV), qz, sc,
                    bits=wl.bits, group=wl.group, fmt=ck["fmt"])
    torch.cuda.synchronize()
    return C


@pytest.mark.parametrize("case", PERM_CASES, ids=lambda c: "b%d_g%d_%s_M%d_K%d_N%d" % c)
@pytest.mark.parametrize("fmt", ["v2", "v1"])
def test_gemm_perm_prepacked_act_order(case, fmt):
    """A[:, perm] @ W_prepacked equals the act-order GEMM of the original checkpoint."""
    bits, group, dt, M, K, N = case
    wl = gptq_inputs.Workload("small", K, N, bits, group, dt, (M,), (fmt,), seed=M * 11 + bits,
                              act_order=True)
    _, ck = checkpoint(wl, fmt)
    A = gptq_inputs.draw_activations(wl, M)
    C = _gemm_perm(wl, ck, A)
    Cref, B = _oracle_gemm(wl, ck, A)
    assert_gemm_close(C, Cref, B, str(case))


def test_gemm_perm_full_size_act_order():
    wl = WL["act_order_3bit_g128"]
    _, ck = checkpoint(wl, "v2")
    A = gptq_inputs.draw_activations(wl, 16)
    C = _gemm_perm(wl, ck, A)
    Cref, B = _oracle_gemm(wl, ck, A)
    assert_gemm_close(C, Cref, B, "act_order_3bit_g128 prepacked")
    assert g.device_status() == 0


# ------------------------------------------------------------------------------ edge cases
def test_m0_leaves_output_untouched():
    wl = WL["tiny_4bit_g64"]
    _, ck = checkpoint(wl, "v2")
    qw, qz, sc, _ = to_device(ck)
    A = torch.empty((0, wl.K), dtype=torch.float16, device=DEV)
    C = g.gemm(A, qw, qz, sc, bits=4, group=64)
    assert C.shape == (0, wl.N)


def test_outputs_fully_written_and_guard_band_intact():
    for M in (3, 16, 77):
        wl = gptq_inputs.Workload("guard", 256, 352, 4, 64, "bf16", (M,), ("v2",), seed=M)
        _, ck = checkpoint(wl, "v2")
        qw, qz, sc, _ = to_device(ck)
        A = gptq_inputs.draw_activations(wl, M).to(DEV)
        buf = torch.full((M + 8, wl.N), float("nan"), dtype=torch.bfloat16, device=DEV)
        buf[M:] = 7.0
        C = g.gemm(A, qw, qz, sc, bits=4, group=64, out=buf[:M])
        torch.cuda.synchronize()
        assert torch.isfinite(C.float()).all(), M
        assert (buf[M:].float() == 7.0).all(), M


def test_deterministic():
    wl = WL["llama7b_decode_4bit_g128"]
    _, ck = checkpoint(wl, "v2")
    qw, qz, sc, _ = to_device(ck)
    for M in (1, 16, 200):
        A = gptq_inputs.draw_activations(wl, M).to(DEV)
        C1 = g.gemm(A, qw, qz, sc, bits=4, group=128)
        C2 = g.gemm(A, qw, qz, sc, bits=4, group=128)
        assert torch.equal(C1.view(torch.int16), C2.view(torch.int16)), M


def test_out_of_range_g_idx_is_clamped_and_flagged():
    wl = gptq_inputs.Workload("gidx", 256, 128, 4, 64, "f16", (4,), ("v2",), seed=3, act_order=True)
    draw, ck = checkpoint(wl, "v2")
    bad = ck["g_idx"].copy()
    bad[5] = 99
    bad[200] = -3
    qw, qz, sc, _ = to_device(ck)
    A = gptq_inputs.draw_activations(wl, 4)
    assert g.device_status() == 0
    C = g.gemm(A.to(DEV), qw, qz, sc, torch.from_numpy(bad).to(DEV), bits=4, group=64)
    assert g.device_status() & g.DEV_GIDX_RANGE
    clamped = np.clip(bad, 0, wl.G - 1).astype(np.int32)
    Cref, B = oracle.gemm(bits16(A), oracle.F16, ck["qweight"], ck["qzeros"], ck["scales"], clamped,
                          wl.N, 4, 64, oracle.V2)
    assert_gemm_close(C, Cref, B, "clamped g_idx")
    assert g.device_status() == 0


def test_misaligned_pointer_rejected():
    wl = WL["tiny_4bit_g64"]
    _, ck = checkpoint(wl, "v2")
    qw, qz, sc, _ = to_device(ck)
    A = torch.zeros((2, wl.K + 1), dtype=torch.float16, device=DEV)[:, 1:]
    with pytest.raises(ValueError):          # the binding refuses non-contiguous views
        g.gemm(A, qw, qz, sc, bits=4, group=64)
    flat = torch.zeros(wl.K * 2 + 1, dtype=torch.float16, device=DEV)[1:].view(2, wl.K)
    with pytest.raises(g.GPTQError) as e:    # the C ABI refuses the 2-byte offset
        g.gemm(flat, qw, qz, sc, bits=4, group=64)
    assert e.value.code == -3


# ------------------------------------------------------------------------------ failure detection
def test_bounded_wait_times_out_and_context_survives():
    """A bounded wait on a phase nothing completes gives up, flags GPTQ_DEV_TIMEOUT, and the
    context stays usable (no trap, no fault)."""
    assert g.device_status() == 0
    waited, status = g.selftest_wait_timeout(50_000_000)
    assert waited == 1
    assert status & g.DEV_TIMEOUT
    assert g.device_status() == 0          # read-and-clear
    wl = WL["tiny_4bit_g64"]
    _, ck = checkpoint(wl, "v2")
    A = gptq_inputs.draw_activations(wl, 64)
    C = _gpu_gemm(wl, ck, A)
    Cref, B = _oracle_gemm(wl, ck, A)
    assert_gemm_close(C, Cref, B, "after timeout self-test")
