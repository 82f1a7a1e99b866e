"""GPU parity on the checkpoints that stress the arithmetic: every GEMM path against the CPU
oracle, element by element, at |C - C_ref| <= 2e-3 * sum_k |a*w| + 1e-3 + ulp/2 (helpers.py).

The seeded N(0, 0.02) workloads give groups whose codes spread over the whole range, so
|q - zero| is large on average and sum_k |a*w| is far from zero.  These cases do the opposite:

* degenerate groups: every code equal to its zero, so the group dequantizes to exactly 0 (page
  "增强 vLLM 对 GPTQv2 格式的支持：分析与实现", section "LLM 的权重量化": w = (q - zero) * scale).
  A column made of such groups has sum_k |a*w| = 0, so the GEMM must return 0 within the
  absolute 1e-3 -- whatever the scale and however large the activations.  (GPTQv1 cannot store
  the zero 0 of a zero-range group, so there the pruned columns dequantize to -scale.)  They come two ways:
  pruned (all-zero) columns and blocks through the round-to-nearest writer (a zero-range group
  gets scale 1), and raw codes planted equal to the zero under a large scale;
* activations with outlier channels (|a| of 1e2 to 1e3 on 1% of the k);
* raw checkpoints: uniformly random codes, stored zeros and fp16 scales (some of them fp16
  subnormals), packed by the oracle's writer -- including the GPTQv1 stored field 2^b - 1,
  whose runtime zero is 2^b (section "从 GPTQv1 到 GPTQv2": runtime zero = stored + 1);
* one-hot activation rows, which make every GEMM output a single dequantized weight, so each
  path must reproduce gptq_dequant bit for bit.

Every path runs: the decode kernel with the per-group scale factored out (2/4/8-bit, 3-bit
fp16, groups aligned to its k-tiles), the per-weight dequantizing decode (act-order g_idx,
bf16 3/8-bit, unaligned groups), the tensor-core kernel (M > 32, with and without g_idx), the
standalone dequant, the prepacked act-order GEMM and the grouped (mixture-of-experts) GEMM;
fp16 and bf16; M = 1, 16, 32 and 130."""
import numpy as np
import pytest
import torch

import gptq_bit_weight_gemm_gb300 as g
import gptq_inputs
import oracle
from helpers import assert_gemm_close, bits16

pytestmark = pytest.mark.gpu
DEV = "cuda"
TDT = {"f16": torch.float16, "bf16": torch.bfloat16}
ODT = {"f16": oracle.F16, "bf16": oracle.BF16}


@pytest.fixture(scope="module", autouse=True)
def _built():
    from gptq_bit_weight_gemm_gb300 import build as lib_build
    lib_build.build()
    assert torch.cuda.is_available()
    yield
    assert g.device_status() == 0


# ------------------------------------------------------------------------------ inputs
def raw_checkpoint(K, N, bits, group, fmt, seed, *, act_order=False, degenerate_cols=(),
                   subnormal_frac=0.1):
    """A checkpoint of uniformly random codes, stored zeros and scales, packed by the oracle.

    degenerate_cols: every code of these columns equals its group's runtime zero (the column
    dequantizes to 0); their scales are drawn large (2 to 16) so that a path which does not
    cancel the zero exactly shows it.  The stored zeros of those columns stay below 2^b - 1 in
    GPTQv1 (a runtime zero of 2^b is no code)."""
    rng = np.random.default_rng(seed)
    G = 1 if group == -1 else K // group
    top = (1 << bits) - 1
    q = rng.integers(0, top + 1, size=(K, N)).astype(np.uint8)
    stored = rng.integers(0, top + 1, size=(G, N)).astype(np.int32)
    stored[:, 0] = top                                   # the largest stored field in column 0
    # scales: fp16 in [2^(-3-b), 2^(1-b)) with random mantissas (so |w| < 2 and the outputs stay
    # inside the fp16 range even with the outlier activations), some of them fp16 subnormals
    e = rng.integers(12 - bits, 16 - bits, size=(G, N))
    m = rng.integers(0, 1024, size=(G, N))
    sbits = ((e << 10) | m).astype(np.uint16)
    sub = rng.random((G, N)) < subnormal_frac
    sbits[sub] = rng.integers(1, 1024, size=int(sub.sum())).astype(np.uint16)
    g_idx = None
    if act_order:
        g_idx = (rng.permutation(K) // (K // G)).astype(np.int32)
    rows_group = g_idx if g_idx is not None else np.arange(K) // (K // G)
    for n in degenerate_cols:
        stored[:, n] = np.minimum(stored[:, n], top - 1) if fmt == oracle.V1 else stored[:, n]
        zero = stored[:, n] + (1 if fmt == oracle.V1 else 0)
        q[:, n] = zero[rows_group]
        sbits[:, n] = ((rng.integers(16, 19, size=G) << 10) | rng.integers(0, 1024, size=G)).astype(np.uint16)
    return {"qweight": oracle.pack_k(q, bits), "qzeros": oracle.pack_n(stored, bits), "scales": sbits,
            "g_idx": g_idx, "bits": bits, "group": group, "fmt": fmt, "K": K, "N": N}


def quantized_checkpoint(K, N, bits, group, fmt, seed, *, sym=False, zero_cols=(), zero_blocks=()):
    """N(0, 0.02) weights through the oracle's round-to-nearest writer, with pruned (all-zero)
    columns and all-zero (group, column) blocks: those groups have range 0, get scale 1 and
    every code equal to the zero."""
    rng = np.random.default_rng(seed)
    W = rng.standard_normal((K, N), dtype=np.float32) * np.float32(0.02)
    rows = K if group == -1 else group
    for n in zero_cols:
        W[:, n] = 0.0
    for gi, n in zero_blocks:
        W[gi * rows:(gi + 1) * rows, n] = 0.0
    ck = oracle.make_checkpoint(W, bits, group, None, sym, fmt)
    ck.update(K=K, N=N)
    return ck


def activations(M, K, dtype, seed, outliers=True):
    """N(0, 1) activations; with outliers, 1% of the k carry |a| of 1e2 to 1e3 in every row."""
    rng = np.random.default_rng(seed)
    a = rng.standard_normal((M, K), dtype=np.float32)
    if outliers:
        ks = rng.choice(K, size=max(1, K // 100), replace=False)
        a[:, ks] *= rng.uniform(100.0, 1000.0, size=ks.size).astype(np.float32)
    return torch.from_numpy(a).to(TDT[dtype])


def dev(ck):
    qw = torch.from_numpy(ck["qweight"]).to(DEV)
    qz = torch.from_numpy(ck["qzeros"]).to(DEV)
    sc = torch.from_numpy(ck["scales"].view(np.int16)).view(torch.float16).to(DEV)
    gi = None if ck["g_idx"] is None else torch.from_numpy(ck["g_idx"]).to(DEV)
    return qw, qz, sc, gi


def check_gemm(ck, A, dtype, what):
    """The GEMM against the oracle; act-order checkpoints both on rows sorted by group on the device
    and with per-row groups."""
    qw, qz, sc, gi = dev(ck)
    Cref, B = oracle.gemm(bits16(A), ODT[dtype], ck["qweight"], ck["qzeros"], ck["scales"], ck["g_idx"],
                          ck["N"], ck["bits"], ck["group"], ck["fmt"])
    for sort_rows in ((True, False) if gi is not None else (True,)):
        C = g.gemm(A.to(DEV), qw, qz, sc, gi, bits=ck["bits"], group=ck["group"], fmt=ck["fmt"],
                   sort_rows=sort_rows)
        torch.cuda.synchronize()
        assert_gemm_close(C, Cref, B, "%s sort_rows=%s" % (what, sort_rows))
    return C, Cref, B


# ------------------------------------------------------------------------------ raw checkpoints
RAW = [(bits, dt, fmt, act) for bits in (2, 3, 4, 8) for dt in ("f16", "bf16")
       for fmt in ("v2", "v1") for act in (False, True)]
MS = (1, 16, 32, 130)
DEGENERATE = (1, 2, 77, 128, 255, 300, 415)


def _raw(bits, dt, fmt, act):
    f = oracle.V1 if fmt == "v1" else oracle.V2
    seed = 1000 + 100 * bits + 10 * (dt == "bf16") + 2 * (fmt == "v1") + act
    return raw_checkpoint(1024, 416, bits, 128, f, seed, act_order=act, degenerate_cols=DEGENERATE)


@pytest.mark.parametrize("bits,dt,fmt,act", RAW)
def test_raw_checkpoint_gemm_with_outliers_and_degenerate_columns(bits, dt, fmt, act):
    ck = _raw(bits, dt, fmt, act)
    for M in MS:
        A = activations(M, ck["K"], dt, seed=7 * M + bits)
        C, Cref, B = check_gemm(ck, A, dt, "b%d %s %s act=%s M=%d" % (bits, dt, fmt, act, M))
        # the degenerate columns are exactly zero in the oracle and within 1e-3 on the GPU
        assert np.all(Cref[:, list(DEGENERATE)] == 0.0) and np.all(B[:, list(DEGENERATE)] == 0.0)


@pytest.mark.parametrize("bits,dt,fmt,act", RAW)
def test_raw_checkpoint_dequant_and_one_hot_rows_bit_exact(bits, dt, fmt, act):
    """gptq_dequant equals the oracle bit for bit, and one-hot rows of A through every GEMM path
    (M = 1, 16, 32 decode; 130 tensor-core) reproduce those rows of the dequantized weight.

    The GEMMs multiply in fp16 for both activation types.  The per-weight and tensor-core paths
    (act-order with per-row groups, M > 32) multiply the weight rounded to fp16, so with bf16
    outputs a one-hot row gives that fp16 weight rounded again to bf16; the folded decode path
    (also act-order on rows sorted by group on the device) keeps the exact product
    (q - zero) * scale in fp32 and rounds it once.  Act-order runs both ways."""
    ck = _raw(bits, dt, fmt, act)
    qw, qz, sc, gi = dev(ck)
    K, N = ck["K"], ck["N"]
    ref = oracle.dequant(ck["qweight"], ck["qzeros"], ck["scales"], ck["g_idx"], K, N, bits, 128,
                         ck["fmt"], ODT[dt])
    ref_via_f16 = ref
    if dt == "bf16":
        w16 = oracle.dequant(ck["qweight"], ck["qzeros"], ck["scales"], ck["g_idx"], K, N, bits, 128,
                             ck["fmt"], oracle.F16)
        ref_via_f16 = oracle.round_to(oracle.to_double(w16, oracle.F16).astype(np.float32), oracle.BF16)
    W = g.dequant(qw, qz, sc, gi, K=K, bits=bits, group=128, fmt=ck["fmt"], dtype=TDT[dt])
    got = bits16(W)
    assert np.array_equal(got, ref), "dequant: %d mismatches" % int((got != ref).sum())
    rng = np.random.default_rng(bits)
    for M in MS:
        rows = np.sort(rng.choice(K, size=M, replace=False))
        A = torch.zeros((M, K), dtype=TDT[dt])
        A[np.arange(M), rows] = 1.0
        for sort_rows in ((True, False) if act else (True,)):
            C = g.gemm(A.to(DEV), qw, qz, sc, gi, bits=bits, group=128, fmt=ck["fmt"], sort_rows=sort_rows)
            torch.cuda.synchronize()
            c = bits16(C)
            # -0 and +0 both represent an exact zero
            per_weight = (act and not sort_rows) or M > 32
            exp = (ref_via_f16 if per_weight else ref)[rows]
            same = (c == exp) | (((c & 0x7FFF) == 0) & ((exp & 0x7FFF) == 0))
            assert same.all(), "M=%d sort_rows=%s: %d of %d outputs differ from dequant" % (
                M, sort_rows, int((~same).sum()), same.size)


# ------------------------------------------------------------------------------ quantizer-made degenerate groups
QUANT = [
    # (bits, group, sym, dtype): every folded decode flavour and its per-weight counterpart
    (4, 128, False, "f16"), (4, 128, False, "bf16"), (2, 64, False, "f16"), (2, 64, False, "bf16"),
    (8, 128, True, "f16"), (8, 128, True, "bf16"), (3, 128, False, "f16"), (3, 128, False, "bf16"),
    (4, -1, False, "f16"), (4, 32, False, "bf16"), (4, 16, False, "f16"),
]


@pytest.mark.parametrize("bits,group,sym,dt", QUANT)
@pytest.mark.parametrize("fmt", ["v2", "v1"])
def test_pruned_columns_and_zero_blocks(bits, group, sym, dt, fmt):
    f = oracle.V1 if fmt == "v1" else oracle.V2
    zero_cols = (0, 5, 130, 400)
    G = 1 if group == -1 else 2048 // group
    zero_blocks = [(gi, n) for gi in range(0, G, 2) for n in (7, 64, 200)]
    ck = quantized_checkpoint(2048, 416, bits, group, f, seed=31 + bits, sym=sym, zero_cols=zero_cols,
                              zero_blocks=zero_blocks)
    for M in MS:
        A = activations(M, 2048, dt, seed=M + 3)
        _, Cref, B = check_gemm(ck, A, dt, "b%d g%d %s %s M=%d" % (bits, group, dt, fmt, M))
        if f == oracle.V2:
            # v2 stores the zero 0 of a zero-range group; v1 cannot (it stores clamp(0 - 1) = 0 and
            # adds 1), so there the pruned columns dequantize to -scale, not 0
            assert np.all(Cref[:, list(zero_cols)] == 0.0)


# ------------------------------------------------------------------------------ other entry points
@pytest.mark.parametrize("bits,dt", [(4, "f16"), (4, "bf16"), (3, "f16"), (2, "bf16"), (8, "f16")])
def test_prepacked_act_order_degenerate_columns(bits, dt):
    ck = raw_checkpoint(1024, 416, bits, 128, oracle.V2, seed=50 + bits, act_order=True,
                        degenerate_cols=DEGENERATE)
    qw2, perm = g.prepack_act_order(ck["qweight"], ck["g_idx"], K=1024, N=416, bits=bits, group=128)
    _, qz, sc, _ = dev(ck)
    for M in (1, 16, 32):
        A = activations(M, 1024, dt, seed=M)
        C = g.gemm_perm(A.to(DEV), torch.from_numpy(perm).to(DEV), torch.from_numpy(qw2).to(DEV), qz, sc,
                        bits=bits, group=128, fmt=oracle.V2)
        torch.cuda.synchronize()
        Cref, B = oracle.gemm(bits16(A), ODT[dt], ck["qweight"], ck["qzeros"], ck["scales"], ck["g_idx"],
                              416, bits, 128, oracle.V2)
        assert_gemm_close(C, Cref, B, "prepacked b%d %s M=%d" % (bits, dt, M))


@pytest.mark.parametrize("dt", ["f16", "bf16"])
def test_grouped_degenerate_experts(dt):
    cks = [raw_checkpoint(512, 288, 4, 64, oracle.V2, seed=90 + e, degenerate_cols=(0, 31, 100, 287))
           for e in range(3)]
    stack = lambda key: np.stack([c[key] for c in cks])
    offsets = np.array([0, 5, 5, 21], np.int32)
    A = activations(21, 512, dt, seed=4)
    C = g.gemm_grouped(A.to(DEV), torch.from_numpy(offsets).to(DEV), torch.from_numpy(stack("qweight")).to(DEV),
                       torch.from_numpy(stack("qzeros")).to(DEV),
                       torch.from_numpy(stack("scales").view(np.int16)).view(torch.float16).to(DEV),
                       bits=4, group=64, max_m=16, fmt=oracle.V2)
    torch.cuda.synchronize()
    Cref, B = oracle.gemm_grouped(bits16(A), ODT[dt], offsets, stack("qweight"), stack("qzeros"),
                                  stack("scales"), 288, 4, 64, oracle.V2)
    assert_gemm_close(C, Cref, B, "grouped %s" % dt)
