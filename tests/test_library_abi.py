"""The C-ABI library: it loads, exports every function include/gptq.h declares, and its host-only
paths (argument validation, the v1 -> v2 zero repack, error strings) behave as documented.
No compute call is made here: these tests run without a GPU."""
import ctypes
import os
import shutil
import subprocess

import numpy as np
import pytest

import gptq_bit_weight_gemm_gb300 as g
import oracle
from gptq_bit_weight_gemm_gb300 import build as lib_build

ROOT = os.path.dirname(os.path.dirname(os.path.abspath(__file__)))


@pytest.fixture(scope="module")
def lib():
    lib_build.build()
    return g.lib()


def test_exports_every_declared_symbol(lib):
    declared = g.header_functions()
    assert declared == sorted(["gptq_dequant", "gptq_gemm", "gptq_gemm_workspace_size",
                               "gptq_repack_zeros_v1_to_v2", "gptq_quantize_rtn",
                               "gptq_get_device_status", "gptq_strerror",
                               "gptq_selftest_wait_timeout", "gptq_prepack_act_order",
                               "gptq_prepack_act_order_device", "gptq_prepack_act_order_device_workspace_size",
                               "gptq_gemm_perm", "gptq_gemm_perm_workspace_size",
                               "gptq_gemm_perm_noalloc", "gptq_gemm_grouped",
                               "gptq_prepack_interleave", "gptq_gemm_interleaved",
                               "gptq_gemm_act_order_workspace_size", "gptq_gemm_host",
                               "gptq_host_plan_create", "gptq_host_plan_run", "gptq_host_plan_destroy"])
    for name in declared:
        assert hasattr(lib, name), name


def test_strerror_and_workspace(lib):
    for code in range(0, -9, -1):
        assert g.strerror(code).startswith(g._STATUS[code])
    assert g.workspace_size(1, 4096, 11008, 4, 128) == 8192 + 256        # fp16 copy of A + row scale
    assert g.workspace_size(4096, 4096, 14336, 4, 128) == 4096 * 4096 * 2 + 4096 * 4
    assert g.workspace_size(0, 4096, 11008, 4, 128) == 0


P = ctypes.c_void_p
FAKE = P(0x10000)   # never dereferenced: validation fails before any device work


@pytest.mark.parametrize("kw,code", [
    (dict(bits=5), -1), (dict(bits=1), -1), (dict(fmt=3), -1), (dict(dtype=2), -1),
    (dict(K=48), -2), (dict(N=40), -2), (dict(group=96), -2), (dict(group=0), -2),
    (dict(group=-1, g_idx=FAKE), -2), (dict(M=-1), -2),
    (dict(qweight=P(0x10004)), -3), (dict(A=P(0x10008)), -3),
    (dict(qweight=None), -1),
])
def test_gemm_validation_without_gpu(lib, kw, code):
    a = dict(A=FAKE, M=1, K=256, dtype=0, qweight=FAKE, qzeros=FAKE, scales=FAKE, g_idx=None,
             N=256, bits=4, group=128, fmt=2, C=FAKE)
    a.update(kw)
    rc = lib.gptq_gemm(a["A"], a["M"], a["K"], a["dtype"], a["qweight"], a["qzeros"], a["scales"],
                       a["g_idx"], a["N"], a["bits"], a["group"], a["fmt"], a["C"], None, 0, None)
    assert rc == code


def test_gemm_m0_is_noop(lib):
    rc = lib.gptq_gemm(None, 0, 256, 0, FAKE, FAKE, FAKE, None, 256, 4, 128, 2, None, None, 0, None)
    assert rc == 0


def test_selftest_validation_without_gpu(lib):
    assert lib.gptq_selftest_wait_timeout(0, FAKE, None) == -1
    assert lib.gptq_selftest_wait_timeout(100, None, None) == -1
    assert lib.gptq_selftest_wait_timeout(100, P(0x10002), None) == -3


def test_dequant_and_quantize_validation_without_gpu(lib):
    assert lib.gptq_dequant(FAKE, FAKE, FAKE, None, 256, 256, 4, 128, 2, 5, FAKE, None) == -1
    assert lib.gptq_dequant(FAKE, FAKE, FAKE, None, 256, 256, 4, 100, 2, 0, FAKE, None) == -2
    assert lib.gptq_dequant(FAKE, FAKE, FAKE, None, 256, 256, 4, 128, 2, 0, P(0x10002), None) == -3
    assert lib.gptq_quantize_rtn(FAKE, 256, 256, 4, 128, None, 2, 2, FAKE, FAKE, FAKE, None) == -1
    assert lib.gptq_quantize_rtn(None, 256, 256, 4, 128, None, 0, 2, FAKE, FAKE, FAKE, None) == -1


@pytest.mark.parametrize("bits", [2, 3, 4, 8])
def test_host_repack_matches_oracle(lib, bits):
    rng = np.random.default_rng(bits)
    G, N = 7, 96
    z = rng.integers(0, (1 << bits) - 1, (G, N)).astype(np.int32)   # never 2^b - 1
    qz_v1 = oracle.pack_n(z, bits)
    got = g.repack_zeros_v1_to_v2(qz_v1, N, bits)
    assert np.array_equal(got, oracle.repack_v1_to_v2(qz_v1, G, N, bits))
    assert np.array_equal(oracle.unpack_n(got, G, N, bits), z + 1)


@pytest.mark.parametrize("bits", [2, 3, 4, 8])
def test_host_repack_overflow(lib, bits):
    z = np.zeros((2, 64), np.int32)
    z[1, 37] = (1 << bits) - 1
    qz = oracle.pack_n(z, bits)
    before = qz.copy()
    rc = lib.gptq_repack_zeros_v1_to_v2(qz.ctypes.data_as(P), qz.ctypes.data_as(P), 2, 64, bits)
    assert rc == -5
    assert np.array_equal(qz, before)    # left unchanged (in place)
    with pytest.raises(g.GPTQError):
        g.repack_zeros_v1_to_v2(qz, 64, bits)


def test_host_repack_in_place(lib):
    z = np.arange(64, dtype=np.int32).reshape(1, 64) % 15
    qz = oracle.pack_n(z, 4)
    rc = lib.gptq_repack_zeros_v1_to_v2(qz.ctypes.data_as(P), qz.ctypes.data_as(P), 1, 64, 4)
    assert rc == 0
    assert np.array_equal(oracle.unpack_n(qz, 1, 64, 4), z + 1)


def _act_order_checkpoint(bits, K=256, N=64, group=32, seed=0):
    rng = np.random.default_rng(seed)
    W = (rng.standard_normal((K, N)) * 0.02).astype(np.float32)
    g_idx = (rng.permutation(K) // group).astype(np.int32)
    return oracle.make_checkpoint(W, bits, group, g_idx=g_idx), g_idx


@pytest.mark.parametrize("bits", [2, 3, 4, 8])
def test_prepack_act_order_matches_oracle(lib, bits):
    """Row k' of the prepacked checkpoint, read with contiguous groups, dequantizes exactly like
    row perm[k'] of the act-order original (the oracle reads both)."""
    K, N, group = 256, 64, 32
    ck, g_idx = _act_order_checkpoint(bits, K, N, group)
    qw2, perm = g.prepack_act_order(ck["qweight"], g_idx, K=K, N=N, bits=bits, group=group)
    assert sorted(perm.tolist()) == list(range(K))
    assert np.all(np.diff(g_idx[perm]) >= 0)                       # groups now contiguous
    assert np.all(np.diff(perm[g_idx[perm] == 3]) > 0)             # stable inside a group
    w_orig = oracle.dequant(ck["qweight"], ck["qzeros"], ck["scales"], g_idx, K, N, bits, group, 2, 0)
    w_new = oracle.dequant(qw2, ck["qzeros"], ck["scales"], None, K, N, bits, group, 2, 0)
    assert np.array_equal(w_new, w_orig[perm])
    assert np.array_equal(oracle.unpack_k(qw2, K, N, bits), ck["q"][perm])


def test_prepack_act_order_validation(lib):
    K, N, group = 256, 64, 32
    ck, g_idx = _act_order_checkpoint(4, K, N, group)
    qw = ck["qweight"]
    bad = g_idx.copy()
    bad[np.flatnonzero(g_idx == 1)[0]] = 0                         # group 0: group + 1 rows
    for gi, code in ((bad, -2), (np.full(K, 8, np.int32), -2), (np.full(K, -1, np.int32), -2)):
        out, perm = np.empty_like(qw), np.empty(K, np.int32)
        rc = lib.gptq_prepack_act_order(qw.ctypes.data_as(P), gi.ctypes.data_as(P), K, N, 4, group,
                                        out.ctypes.data_as(P), perm.ctypes.data_as(P))
        assert rc == code
    out, perm = np.empty_like(qw), np.empty(K, np.int32)
    assert lib.gptq_prepack_act_order(qw.ctypes.data_as(P), g_idx.ctypes.data_as(P), K, N, 4, 48,
                                      out.ctypes.data_as(P), perm.ctypes.data_as(P)) == -2
    assert lib.gptq_prepack_act_order(None, g_idx.ctypes.data_as(P), K, N, 4, group,
                                      out.ctypes.data_as(P), perm.ctypes.data_as(P)) == -1


@pytest.mark.parametrize("kw,code", [
    (dict(M=33), -2), (dict(M=-1), -2), (dict(group=-1), -2), (dict(perm=None), -1),
    (dict(perm=P(0x10004)), -3), (dict(bits=5), -1), (dict(K=48), -2),
    (dict(M=4), -4), (dict(M=4, ws=FAKE, ws_bytes=4 * 256 * 2 - 1), -4),
    (dict(M=4, ws=P(0x10008), ws_bytes=4 * 256 * 2), -3),
])
def test_gemm_perm_validation_without_gpu(lib, kw, code):
    a = dict(A=FAKE, M=1, K=256, dtype=0, perm=FAKE, qweight=FAKE, qzeros=FAKE, scales=FAKE,
             N=256, bits=4, group=128, fmt=2, C=FAKE, ws=None, ws_bytes=0)
    a.update(kw)
    rc = lib.gptq_gemm_perm(a["A"], a["M"], a["K"], a["dtype"], a["perm"], a["qweight"], a["qzeros"],
                            a["scales"], a["N"], a["bits"], a["group"], a["fmt"], a["C"], a["ws"],
                            a["ws_bytes"], None)
    assert rc == code


@pytest.mark.parametrize("kw,code", [
    (dict(max_m=0), -2), (dict(max_m=33), -2), (dict(E=-1), -2), (dict(E=65536), -2),
    (dict(rows=-1), -2), (dict(offsets=None), -1), (dict(A=None), -1), (dict(C=None), -1),
    (dict(offsets=P(0x10002)), -3), (dict(A=P(0x10008)), -3), (dict(bits=5), -1),
    (dict(fmt=3), -1), (dict(dtype=2), -1), (dict(K=48), -2), (dict(group=100), -2),
    (dict(rows=0), 0), (dict(E=0), 0),
])
def test_gemm_grouped_validation_without_gpu(lib, kw, code):
    a = dict(A=FAKE, rows=16, K=256, dtype=0, offsets=FAKE, E=4, max_m=8, qweight=FAKE,
             qzeros=FAKE, scales=FAKE, N=256, bits=4, group=128, fmt=2, C=FAKE)
    a.update(kw)
    rc = lib.gptq_gemm_grouped(a["A"], a["rows"], a["K"], a["dtype"], a["offsets"], a["E"], a["max_m"],
                               a["qweight"], a["qzeros"], a["scales"], a["N"], a["bits"], a["group"],
                               a["fmt"], a["C"], None)
    assert rc == code


def test_act_order_workspace_size(lib):
    # flag (256) + row order and code positions (K * 4 each) + sorted packed weight + the
    # tensor-core workspace for M x K
    assert g.act_order_workspace_size(16, 5120, 13824, 3, 128) == (256 + 2 * 20480 + 5120 * 3 // 32 * 13824 * 4
                                                                   + 16 * 5120 * 2 + 256)
    assert g.act_order_workspace_size(1, 4096, 11008, 4, 128) == (256 + 2 * 16384 + 4096 // 8 * 11008 * 4
                                                                  + 8192 + 256)
    assert g.act_order_workspace_size(3, 96, 32, 8, 32) == 256 + 2 * 512 + 24 * 32 * 4 + 768 + 256
    assert g.act_order_workspace_size(4, 512, 128, 2, 16) == 0      # groups of 16 rows at 2 bits (not whole k-tiles)
    assert g.act_order_workspace_size(4, 1024, 128, 3, 64) == 0     # 3-bit groups must be multiples of 128
    assert g.act_order_workspace_size(4, 4096, 128, 4, 1) == 0      # 4096 groups: the sort's 520 KB
    assert g.act_order_workspace_size(4, 131072, 128, 4, 128) == 0  # a 4-column strip of 256 KB
    assert g.act_order_workspace_size(0, 512, 128, 4, 64) == 0
    assert g.act_order_workspace_size(4, 500, 128, 4, 64) == 0      # group does not divide K


def test_prepack_act_order_device_workspace_size(lib):
    # the sort's flag (256) + each sorted row's code position (K * 4, rounded up to 256)
    assert g.prepack_act_order_device_workspace_size(5120, 3, 128) == 256 + 20480
    assert g.prepack_act_order_device_workspace_size(96, 8, 32) == 256 + 512
    assert g.prepack_act_order_device_workspace_size(512, 2, 16) == 256 + 2048   # any group size
    assert g.prepack_act_order_device_workspace_size(4096, 4, 1) == 0     # 4096 groups: the sort's 520 KB
    assert g.prepack_act_order_device_workspace_size(131072, 4, 128) == 0  # a 4-column strip of 256 KB
    assert g.prepack_act_order_device_workspace_size(500, 4, 100) == 0     # K not a multiple of 32
    assert g.prepack_act_order_device_workspace_size(512, 4, 100) == 0     # group does not divide K
    assert g.prepack_act_order_device_workspace_size(512, 5, 64) == 0
    assert g.prepack_act_order_device_workspace_size(512, 4, 0) == 0


@pytest.mark.parametrize("kw,code", [
    (dict(qweight=None), -1), (dict(g_idx=None), -1), (dict(out=None), -1), (dict(perm=None), -1),
    (dict(ws=None), -1), (dict(bits=5), -1), (dict(K=48), -2), (dict(N=48), -2), (dict(group=100), -2),
    (dict(group=0), -2), (dict(K=4096, group=1), -2), (dict(ws_bytes=256 + 1024 - 1), -4),
    (dict(perm=P(0x30008)), -3), (dict(out=P(0x20008)), -3), (dict(g_idx=P(0x40002)), -3),
    (dict(ws=P(0x50008)), -3),
    (dict(out=P(0x10000 + 256 * 64 * 4 // 8 - 16)), -1),   # the last 16 bytes of qweight
])
def test_prepack_act_order_device_validation_without_gpu(lib, kw, code):
    a = dict(qweight=FAKE, g_idx=P(0x40000), K=256, N=64, bits=4, group=32, out=P(0x20000),
             perm=P(0x30000), ws=P(0x50000), ws_bytes=4096)
    a.update(kw)
    rc = lib.gptq_prepack_act_order_device(a["qweight"], a["g_idx"], a["K"], a["N"], a["bits"], a["group"],
                                           a["out"], a["perm"], a["ws"], a["ws_bytes"], None)
    assert rc == code


def test_gemm_perm_workspace_size(lib):
    assert g.gemm_perm_workspace_size(1, 4096) == 0
    assert g.gemm_perm_workspace_size(0, 4096) == 0
    assert g.gemm_perm_workspace_size(16, 5120) == 16 * 5120 * 2
    assert g.gemm_perm_workspace_size(3, 96) == 768        # 576 rounded up to 256


def test_product_does_not_import_oracle():
    import os
    import re
    pkg = os.path.dirname(g.__file__)
    for root, _, files in os.walk(pkg):
        for f in files:
            if f.endswith((".py", ".cu", ".cuh", ".h")):
                text = open(os.path.join(root, f)).read()
                assert not re.search(r"^\s*(import|from)\s+oracle\b", text, re.M), f
                assert "gptq_oracle" not in text, f


C_CONSUMER = r"""
#include <stdio.h>
#include <string.h>
#include "gptq.h"

int main(void) {
  int32_t qz[2][8];
  int rc, i;
  /* host-only entry points, called from plain C */
  for (i = 0; i < 8; ++i) qz[0][i] = 0x11111111;          /* 4-bit v1 zeros 1..1 */
  rc = gptq_repack_zeros_v1_to_v2(qz[0], qz[1], 1, 64, 4);
  if (rc != GPTQ_OK || qz[1][0] != 0x22222222) { printf("repack %d %x\n", rc, qz[1][0]); return 1; }
  /* validation happens before any device work */
  if (gptq_gemm(NULL, 1, 256, GPTQ_F16, NULL, NULL, NULL, NULL, 256, 4, 128, GPTQ_FMT_V2, NULL, NULL, 0,
                NULL) != GPTQ_ERR_ARG) return 2;
  if (gptq_gemm_grouped(NULL, 0, 256, GPTQ_F16, NULL, 1, 8, NULL, NULL, NULL, 256, 4, 128,
                        GPTQ_FMT_V2, NULL, NULL) != GPTQ_ERR_ARG) return 3;
  if (gptq_gemm_workspace_size(1, 4096, 11008, 4, 128) != 8448) return 4;
  /* the host-buffer call: a NULL host or staging pointer, and the empty problem */
  if (gptq_gemm_host(NULL, NULL, 1, 256, GPTQ_F16, NULL, NULL, NULL, NULL, 256, 4, 128, GPTQ_FMT_V2,
                     NULL, NULL, NULL, 0, NULL) != GPTQ_ERR_ARG) return 6;
  if (gptq_gemm_host(NULL, NULL, 0, 256, GPTQ_F16, NULL, NULL, NULL, NULL, 256, 4, 128, GPTQ_FMT_V2,
                     NULL, NULL, NULL, 0, NULL) != GPTQ_OK) return 7;
  if (gptq_gemm_host(NULL, NULL, 1, 0, GPTQ_F16, NULL, NULL, NULL, NULL, 256, 4, 128, GPTQ_FMT_V2,
                     NULL, NULL, NULL, 0, NULL) != GPTQ_ERR_SHAPE) return 8;
  /* the prepared call: a NULL plan slot or the legacy default stream is refused first */
  {
    gptq_host_plan* plan = (gptq_host_plan*)1;
    if (gptq_host_plan_create(NULL, NULL, NULL, 1, 256, GPTQ_F16, NULL, NULL, NULL, NULL, 256, 4, 128,
                              GPTQ_FMT_V2, NULL, NULL, NULL, 0, NULL) != GPTQ_ERR_ARG) return 9;
    if (gptq_host_plan_create(&plan, NULL, NULL, 1, 256, GPTQ_F16, NULL, NULL, NULL, NULL, 256, 4, 128,
                              GPTQ_FMT_V2, NULL, NULL, NULL, 0, NULL) != GPTQ_ERR_ARG || plan != NULL) return 10;
    if (gptq_host_plan_run(NULL) != GPTQ_ERR_ARG) return 11;
    if (gptq_host_plan_destroy(NULL) != GPTQ_OK) return 12;
  }
  if (strlen(gptq_strerror(GPTQ_ERR_SHAPE)) == 0) return 5;
  printf("c consumer ok\n");
  return 0;
}
"""


@pytest.mark.skipif(shutil.which("gcc") is None, reason="needs gcc")
def test_header_is_plain_c_and_links(lib, tmp_path):
    """The boundary is a C ABI: a C99 program (no C++ compiler) includes include/gptq.h, links the
    built library and calls its host entry points and argument checks."""
    src = tmp_path / "consumer.c"
    src.write_text(C_CONSUMER)
    exe = tmp_path / "consumer"
    libdir = os.path.dirname(g.LIB_PATH)
    subprocess.run(["gcc", "-std=c99", "-Wall", "-Werror", "-I", os.path.join(ROOT, "include"), str(src),
                    "-o", str(exe), "-L", libdir, "-l:" + os.path.basename(g.LIB_PATH),
                    "-Wl,-rpath," + libdir], check=True)
    r = subprocess.run([str(exe)], capture_output=True, text=True)
    assert r.returncode == 0 and "c consumer ok" in r.stdout, (r.returncode, r.stdout, r.stderr)
