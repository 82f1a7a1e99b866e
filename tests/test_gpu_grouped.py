"""GPU parity of the grouped (mixture-of-experts) GEMM, gptq_gemm_grouped, against the CPU
oracle's gemm_grouped on the same seeded inputs (page "4.3 Weight-only INT4 量化：GPTQ、AWQ 与
Marlin Kernel", section 7: a MoE model's expert weights are GPTQ checkpoints like any other).

Every row an expert owns must be within |C - C_ref| <= 2e-3 * sum_k |a*w| + 1e-3 of the
oracle's fp32 result; rows no expert owns, and the rows of an expert whose range is flagged,
must keep the sentinel they held before the call.  Sizes: oracle-sized cases over every width,
format and dtype with ragged column tails, empty experts and experts that fill the token tile,
plus the full Mixtral-shaped expert layer (8 experts x [4096, 14336]) compared on every row."""
import dataclasses

import numpy as np
import pytest
import torch

import gptq_bit_weight_gemm_gb300 as g
import gptq_inputs
import oracle
from helpers import FMT, assert_gemm_close, bits16

pytestmark = pytest.mark.gpu

DEV = "cuda"
MOE = gptq_inputs.MOE_WORKLOADS["moe_mixtral_4bit_g128"]
SENTINEL = {torch.float16: 0x7E00, torch.bfloat16: 0x7FC0}     # a quiet NaN of each format


@pytest.fixture(scope="module", autouse=True)
def _built():
    from gptq_bit_weight_gemm_gb300 import build as lib_build
    lib_build.build()
    assert torch.cuda.is_available()
    yield
    assert g.device_status() == 0


def _dtype(mw):
    return torch.float16 if mw.act_dtype == "f16" else torch.bfloat16


def _experts(mw, fmt):
    """Every expert's checkpoint, written by the oracle, stacked expert-first."""
    cks = [oracle.make_checkpoint(gptq_inputs.draw_expert_weights(mw, e), mw.bits, mw.group, None,
                                  False, FMT[fmt]) for e in range(mw.E)]
    return (np.stack([c["qweight"] for c in cks]), np.stack([c["qzeros"] for c in cks]),
            np.stack([c["scales"] for c in cks]))


def _gpu(mw, fmt, A, offsets, max_m, ck):
    qw, qz, sc = ck
    dt = _dtype(mw)
    fill = int(np.array(SENTINEL[dt], np.uint16).view(np.int16))
    C = torch.full((A.shape[0], mw.N), fill, dtype=torch.int16, device=DEV).view(dt)
    g.gemm_grouped(A.to(DEV), torch.from_numpy(offsets).to(DEV), torch.from_numpy(qw).to(DEV),
                   torch.from_numpy(qz).to(DEV),
                   torch.from_numpy(sc.view(np.int16)).view(torch.float16).to(DEV),
                   bits=mw.bits, group=mw.group, max_m=max_m, fmt=FMT[fmt], out=C)
    torch.cuda.synchronize()
    return C


def _compare(mw, fmt, A, offsets, C, ck, skip=()):
    qw, qz, sc = ck
    code = oracle.F16 if mw.act_dtype == "f16" else oracle.BF16
    Cref, B = oracle.gemm_grouped(bits16(A), code, offsets, qw, qz, sc, mw.N, mw.bits, mw.group,
                                  FMT[fmt])
    got = bits16(C)
    sentinel = SENTINEL[_dtype(mw)]
    owned = np.zeros(A.shape[0], bool)
    for e in range(mw.E):
        lo, hi = int(offsets[e]), int(offsets[e + 1])
        if e in skip or hi <= lo:
            continue
        owned[lo:hi] = True
        assert_gemm_close(C[lo:hi], Cref[lo:hi], B[lo:hi],
                          "%s %s expert %d rows %d..%d" % (mw.name, fmt, e, lo, hi))
    assert np.all(got[~owned] == sentinel), "rows outside every expert's range were written"


def _grouped_rows(mw, T):
    r = gptq_inputs.draw_routing(mw, T)
    A = gptq_inputs.draw_token_activations(mw, T)[torch.from_numpy(r.row_token).long()]
    return A.contiguous(), r.offsets


def _case(E, K, N, bits, group, act, topk=2):
    return dataclasses.replace(MOE, name="moe_%dx%dx%d_b%d_g%d_%s" % (E, K, N, bits, group, act), E=E,
                               K=K, N=N, bits=bits, group=group, act_dtype=act, topk=topk)


# (workload, tokens, max_m): several slabs with ragged last slabs (N % 128 != 0), K splits over
# clusters, every width, both dtypes, one group per column, and token tiles 1, 8, 16 and 32
SMALL = [
    (_case(3, 512, 320, 4, 128, "f16"), 5, 8),
    (_case(8, 1024, 256, 2, 64, "bf16"), 8, 8),
    (_case(4, 768, 384, 3, 128, "f16"), 6, 16),
    (_case(4, 512, 256, 8, -1, "bf16"), 6, 8),
    (_case(6, 512, 192, 4, 32, "f16", topk=1), 4, 1),
    (_case(4, 1024, 640, 4, 128, "bf16", topk=4), 24, 32),
    (_case(5, 512, 256, 3, 64, "bf16"), 7, 16),
    (_case(3, 2048, 128, 8, 128, "f16"), 3, 8),
]


@pytest.mark.parametrize("mw,T,max_m", SMALL, ids=lambda v: v.name if hasattr(v, "name") else str(v))
@pytest.mark.parametrize("fmt", ["v2", "v1"])
def test_grouped_small(mw, T, max_m, fmt):
    A, offsets = _grouped_rows(mw, T)
    if mw.topk == 1 and max_m == 1:                   # one token per expert at most
        offsets = np.minimum(np.arange(mw.E + 1), T).astype(np.int32)
        A = A[:T]
    assert np.diff(offsets).max() <= max_m
    ck = _experts(mw, fmt)
    C = _gpu(mw, fmt, A, offsets, max_m, ck)
    _compare(mw, fmt, A, offsets, C, ck)


def test_grouped_full_tile_and_unowned_rows():
    """Experts holding exactly max_m rows, empty experts between them, and trailing rows that
    no expert owns (they keep the sentinel)."""
    mw = _case(5, 1024, 384, 4, 128, "f16")
    offsets = np.array([0, 16, 16, 32, 32, 40], np.int32)
    A = gptq_inputs.draw_token_activations(dataclasses.replace(mw, K=1024), 44)
    ck = _experts(mw, "v2")
    C = _gpu(mw, "v2", A, offsets, 16, ck)
    _compare(mw, "v2", A, offsets, C, ck)


@pytest.mark.parametrize("offsets,rows,bad", [
    ([0, 3, 4, 4], 5, 0),        # expert 0 holds 3 rows, more than max_m = 2
    ([0, 2, 1, 1], 3, 1),        # expert 1's range is decreasing
    ([0, 2, 9], 4, 1),           # expert 1's range ends past the last row
])
def test_grouped_flags_bad_ranges(offsets, rows, bad):
    """A bad range is skipped (its rows keep the sentinel), flagged in the status word, and the
    other experts are still computed."""
    E = len(offsets) - 1
    mw = _case(E, 512, 256, 4, 128, "f16")
    offsets = np.array(offsets, np.int32)
    A = gptq_inputs.draw_token_activations(mw, rows)
    ck = _experts(mw, "v2")
    assert g.device_status() == 0
    C = _gpu(mw, "v2", A, offsets, 2, ck)
    assert g.device_status() & g.DEV_EXPERT_ROWS
    good = offsets.copy()
    _compare(mw, "v2", A, good, C, ck, skip=(bad,))
    lo, hi = int(offsets[bad]), int(offsets[bad + 1])
    if hi > lo:
        assert np.all(bits16(C)[lo:min(hi, rows)] == SENTINEL[torch.float16])


def test_grouped_flags_bad_ranges_with_fewer_rows_than_experts():
    """Fewer rows than experts: the grid then holds one slot per row, and slot z takes the z-th
    expert that holds rows.  Malformed ranges (expert 2 ends past the rows, expert 3 decreases)
    are skipped and flagged; the one valid expert is computed and the other rows keep the
    sentinel."""
    E, rows = 6, 3
    mw = _case(E, 512, 256, 4, 128, "f16")
    offsets = np.array([0, 1, 1, 5, 3, 3, 3], np.int32)
    A = gptq_inputs.draw_token_activations(mw, rows)
    ck = _experts(mw, "v2")
    assert g.device_status() == 0
    C = _gpu(mw, "v2", A, offsets, 2, ck)
    assert g.device_status() & g.DEV_EXPERT_ROWS
    _compare(mw, "v2", A, np.array([0, 1, 1, 1, 1, 1, 1], np.int32), C, ck)


@pytest.mark.parametrize("T", MOE.Ts)
def test_grouped_full_size(T):
    """The Mixtral-shaped expert layer at full size: 8 experts x [4096, 14336], 4-bit g128,
    T tokens routed to 2 experts each; every output compared."""
    A, offsets = _grouped_rows(MOE, T)
    max_m = 1 if np.diff(offsets).max() <= 1 else 8
    ck = _experts(MOE, "v2")
    C = _gpu(MOE, "v2", A, offsets, max_m, ck)
    _compare(MOE, "v2", A, offsets, C, ck)


@pytest.mark.parametrize("max_m", [8, 16, 32])
@pytest.mark.parametrize("bits,group,act", [(4, 128, "f16"), (2, 64, "bf16"), (3, 128, "bf16")])
def test_grouped_one_row_in_a_wide_tile(max_m, bits, group, act):
    """One row per expert through the run-time token-count kernels (tile 8, 16 or 32) on a shape
    that runs 16-CTA clusters with two k-tiles per CTA, where the staged activations are smaller
    than a token's 128 partial sums: the one-token reduction must not pass through them."""
    mw = _case(2, 1024, 256, bits, group, act)
    A = gptq_inputs.draw_token_activations(mw, 2)
    offsets = np.array([0, 1, 2], np.int32)
    ck = _experts(mw, "v2")
    C = _gpu(mw, "v2", A, offsets, max_m, ck)
    _compare(mw, "v2", A, offsets, C, ck)
