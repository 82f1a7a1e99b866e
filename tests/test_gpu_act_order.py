"""GPU parity of gptq_gemm on act-order checkpoints (page "增强 vLLM 对 GPTQv2 格式的支持：分析与实现",
section "LLM 的权重量化": the quantization groups are the row sets {k : g_idx[k] == g}).

With a workspace of gptq_gemm_act_order_workspace_size bytes the call sorts the rows by group on the
device, rewrites the packed weight in that order and runs the group-wise kernels; a device flag
sends g_idx whose groups are not all of `group` rows to the per-row-group kernels.  Checked here:
  * the device's sorted row order and sorted packed weight equal the host prepack's, bit for bit
    (integer work), for every width;
  * both paths (sorted rows, and per-row groups with sort_rows=False) against the oracle, on the
    decode kernel (M <= 32, one token and several), the tensor-core kernel (M > 32, ragged), fp16
    and bf16, v1 and v2;
  * g_idx with unequal groups (flag 0: the per-row-group kernels run, in the same stream order),
    and with an entry out of range (clamped and flagged, as without the workspace);
  * repeated calls give identical bits;
  * gptq_prepack_act_order_device (the same sort and repack, once, into caller buffers) equals the
    host prepack bit for bit, a gptq_gemm_perm issued right after it on the stream meets the
    oracle, and g_idx it cannot sort leaves its outputs unwritten and raises GPTQ_DEV_GIDX_GROUPS."""
import ctypes

import numpy as np
import pytest
import torch

import gptq_bit_weight_gemm_gb300 as g
import gptq_inputs
import oracle
from helpers import FMT, assert_gemm_close, bits16, checkpoint, dtype_code, to_device

pytestmark = pytest.mark.gpu

DEV = "cuda"


@pytest.fixture(scope="module", autouse=True)
def _built():
    from gptq_bit_weight_gemm_gb300 import build as lib_build
    lib_build.build()
    assert torch.cuda.is_available()
    yield
    assert g.device_status() == 0


def _up(x):
    return (x + 255) // 256 * 256


def _layout(K, N, bits):
    """Offsets of the flag, the sorted row order and the sorted packed weight in the workspace
    (the code positions sit between the last two)."""
    perm = 256
    qweight = perm + 2 * _up(K * 4)
    return 0, perm, qweight, qweight + _up(K * bits // 32 * N * 4)


def _wl(bits, group, dt, M, K, N, fmt="v2", seed=0):
    return gptq_inputs.Workload("act", K, N, bits, group, dt, (M,), (fmt,), seed=seed or (M * 13 + bits),
                                act_order=True)


def _oracle(wl, ck, A, g_idx=None):
    return oracle.gemm(bits16(A), dtype_code(wl), ck["qweight"], ck["qzeros"], ck["scales"],
                       ck["g_idx"] if g_idx is None else g_idx, wl.N, wl.bits, wl.group, ck["fmt"])


def _gemm(wl, ck, A, g_idx=None, sort_rows=True, workspace=None):
    qw, qz, sc, gi = to_device(ck)
    if g_idx is not None:
        gi = torch.from_numpy(g_idx).to(DEV)
    C = g.gemm(A.to(DEV), qw, qz, sc, gi, bits=wl.bits, group=wl.group, fmt=ck["fmt"],
               sort_rows=sort_rows, workspace=workspace)
    torch.cuda.synchronize()
    return C


@pytest.mark.parametrize("bits,group,K,N", [
    (2, 64, 1024, 160), (3, 128, 640, 416), (4, 32, 512, 96), (8, 128, 384, 288),
    # long K: the repack's column strip narrows to 16, 8 and 4 columns
    (4, 128, 16384, 64), (3, 128, 40960, 64), (4, 128, 53248, 32), (8, 128, 20480, 32)])
def test_device_sort_matches_host_prepack(bits, group, K, N):
    wl = _wl(bits, group, "f16", 5, K, N)
    _, ck = checkpoint(wl, "v2")
    size = g.act_order_workspace_size(5, K, N, bits, group)
    assert size > 0
    ws = torch.zeros(size, dtype=torch.uint8, device=DEV)
    A = gptq_inputs.draw_activations(wl, 5)
    C = _gemm(wl, ck, A, workspace=ws)
    qw_host, perm_host = g.prepack_act_order(ck["qweight"], ck["g_idx"], K=K, N=N, bits=bits, group=group)
    f, p, q, end = _layout(K, N, bits)
    raw = ws.cpu().numpy()
    assert raw[f:f + 4].view(np.int32)[0] == 1
    assert np.array_equal(raw[p:p + 4 * K].view(np.int32), perm_host)
    assert np.array_equal(raw[q:q + qw_host.nbytes].view(np.int32).reshape(qw_host.shape), qw_host)
    Cref, B = _oracle(wl, ck, A)
    assert_gemm_close(C, Cref, B, "sorted rows b%d" % bits)


@pytest.mark.parametrize("bits,group,K,N", [
    (2, 64, 1024, 160), (3, 128, 640, 416), (4, 32, 512, 96), (8, 128, 384, 288), (4, 128, 16384, 64),
    (3, 128, 5120, 1024)])
def test_device_prepack_matches_host_prepack(bits, group, K, N):
    wl = _wl(bits, group, "f16", 4, K, N, seed=bits * 7 + 1)
    _, ck = checkpoint(wl, "v2")
    qw, qz, sc, gi = to_device(ck)
    qw_dev, perm_dev = g.prepack_act_order_device(qw, gi, K=K, N=N, bits=bits, group=group)
    # the very next call on the stream uses them (the prepack ends with an ordering step)
    A = gptq_inputs.draw_activations(wl, 4)
    C = g.gemm_perm(A.to(DEV), perm_dev, qw_dev, qz, sc, bits=bits, group=group, fmt=ck["fmt"])
    torch.cuda.synchronize()
    qw_host, perm_host = g.prepack_act_order(ck["qweight"], ck["g_idx"], K=K, N=N, bits=bits, group=group)
    assert np.array_equal(perm_dev.cpu().numpy(), perm_host)
    assert np.array_equal(qw_dev.cpu().numpy(), qw_host)
    Cref, B = _oracle(wl, ck, A)
    assert_gemm_close(C, Cref, B, "device prepack b%d" % bits)


@pytest.mark.parametrize("case", ["unequal_groups", "entry_out_of_range"])
def test_device_prepack_leaves_outputs_for_unusable_g_idx(case):
    bits, group, K, N = 4, 128, 1024, 160
    wl = _wl(bits, group, "f16", 1, K, N)
    _, ck = checkpoint(wl, "v2")
    bad = ck["g_idx"].copy()
    if case == "unequal_groups":
        bad[np.flatnonzero(bad == 1)[0]] = 0                       # group 0: group + 1 rows
    else:
        bad[5] = K // group                                         # G: outside [0, G)
    qw = torch.from_numpy(ck["qweight"]).to(DEV)
    gi = torch.from_numpy(bad).to(DEV)
    out = torch.full_like(qw, 0x5A5A5A5A)
    perm = torch.full((K,), -7, dtype=torch.int32, device=DEV)
    ws = torch.empty(g.prepack_act_order_device_workspace_size(K, bits, group), dtype=torch.uint8, device=DEV)
    p = lambda t: ctypes.c_void_p(t.data_ptr())
    rc = g.lib().gptq_prepack_act_order_device(p(qw), p(gi), K, N, bits, group, p(out), p(perm), p(ws),
                                               ws.numel(), None)
    assert rc == 0, g.strerror(rc)
    assert g.device_status() == g.DEV_GIDX_GROUPS
    assert bool((out == 0x5A5A5A5A).all()) and bool((perm == -7).all())


CASES = [
    # (bits, group, dtype, M, K, N): decode (one token: A gathered while staging; several: gathered
    # into the workspace) and tensor-core (M > 32, ragged tiles)
    (3, 128, "f16", 1, 1024, 416),
    (3, 128, "bf16", 16, 640, 288),
    (4, 128, "f16", 8, 1024, 544),
    (4, 64, "bf16", 32, 512, 352),
    (2, 64, "bf16", 3, 1024, 160),
    (8, 128, "f16", 20, 384, 288),
    (8, 64, "bf16", 1, 512, 160),
    (4, 128, "f16", 130, 512, 544),
    (3, 128, "bf16", 129, 1024, 288),
    (2, 128, "f16", 300, 768, 256),
    (8, 128, "bf16", 65, 384, 160),
]


@pytest.mark.parametrize("case", CASES, ids=lambda c: "b%d_g%d_%s_M%d_K%d_N%d" % c)
@pytest.mark.parametrize("fmt", ["v2", "v1"])
@pytest.mark.parametrize("sort_rows", [True, False], ids=["sorted", "per_row"])
def test_act_order_gemm_both_paths(case, fmt, sort_rows):
    bits, group, dt, M, K, N = case
    wl = _wl(bits, group, dt, M, K, N, fmt)
    _, ck = checkpoint(wl, fmt)
    assert g.act_order_workspace_size(M, K, N, bits, group) > 0
    A = gptq_inputs.draw_activations(wl, M)
    C = _gemm(wl, ck, A, sort_rows=sort_rows)
    Cref, B = _oracle(wl, ck, A)
    assert_gemm_close(C, Cref, B, "%s %s sort_rows=%s" % (case, fmt, sort_rows))


@pytest.mark.parametrize("M,dt", [(1, "f16"), (12, "bf16"), (80, "f16"), (33, "bf16")])
def test_unequal_groups_take_the_per_row_kernels(M, dt):
    """Groups of unequal size (each row drawn into a random group) cannot be sorted into groups of
    `group` rows: the device flag is 0 and the per-row-group kernels give the result."""
    K, N, bits, group = 512, 160, 4, 64
    wl = _wl(bits, group, dt, M, K, N)
    _, ck = checkpoint(wl, "v2")
    rng = np.random.default_rng(M)
    g_uneven = rng.integers(0, K // group, size=K).astype(np.int32)
    assert np.bincount(g_uneven, minlength=K // group).max() != group
    ck_u = oracle.make_checkpoint(gptq_inputs.draw_weights(wl).W, bits, group, g_uneven, False, oracle.V2)
    size = g.act_order_workspace_size(M, K, N, bits, group)
    ws = torch.full((size,), 0x7F, dtype=torch.uint8, device=DEV)
    A = gptq_inputs.draw_activations(wl, M)
    C = _gemm(wl, ck_u, A, workspace=ws)
    assert ws[:4].cpu().numpy().view(np.int32)[0] == 0
    Cref, B = _oracle(wl, ck_u, A)
    assert_gemm_close(C, Cref, B, "unequal groups M=%d" % M)
    assert g.device_status() == 0


@pytest.mark.parametrize("M", [1, 6, 40])
def test_out_of_range_entry_is_clamped_and_flagged_with_workspace(M):
    K, N, bits, group = 256, 128, 4, 64
    wl = _wl(bits, group, "f16", M, K, N)
    _, ck = checkpoint(wl, "v2")
    bad = ck["g_idx"].copy()
    bad[5] = 99
    bad[200] = -3
    A = gptq_inputs.draw_activations(wl, M)
    assert g.device_status() == 0
    C = _gemm(wl, ck, A, g_idx=bad)
    assert g.device_status() & g.DEV_GIDX_RANGE
    clamped = np.clip(bad, 0, K // group - 1).astype(np.int32)
    Cref, B = _oracle(wl, ck, A, g_idx=clamped)
    assert_gemm_close(C, Cref, B, "clamped g_idx M=%d" % M)
    assert g.device_status() == 0


def test_full_size_act_order_both_paths_and_deterministic():
    wl = gptq_inputs.WORKLOADS["act_order_3bit_g128"]
    _, ck = checkpoint(wl, "v2")
    A = gptq_inputs.draw_activations(wl, 16)
    Cref, B = _oracle(wl, ck, A)
    C1 = _gemm(wl, ck, A)
    C2 = _gemm(wl, ck, A)
    assert torch.equal(C1.view(torch.int16), C2.view(torch.int16))
    assert_gemm_close(C1, Cref, B, "act_order_3bit_g128 sorted rows")
    C3 = _gemm(wl, ck, A, sort_rows=False)
    assert_gemm_close(C3, Cref, B, "act_order_3bit_g128 per-row groups")

