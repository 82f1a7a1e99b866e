"""Host-side launch geometry of the decode kernels, checked without a GPU.

tests/geometry_probe.cu is compiled against the library's headers (nvcc, host code only) and asks
the launcher's own geometry selection (select_geometry in decode_mma.cuh) for the cluster split
and shared-memory layout of a sweep of problems: every width, K up to 53248,
N with ragged slabs, 1 to 32 tokens, groups from 32 rows to one per column, the scale-folding and
the per-weight dequant paths, act-order, grouped launches of 8 experts, and two token blocks side
by side (17..32 tokens as two 16-token blocks).  Every layout must:
  - fit one CTA's shared memory (227 KB),
  - keep TMA boxes within the hardware's 256 rows, in 1024-byte aligned slots of 32 columns,
  - cover the whole K range with its CTAs and every chunk of a CTA with buffers,
  - stage the scale/zero constants of every group a CTA's K range touches (recomputed here from
    the split rule the kernel uses), and the per-k data of the dequant path within its 24 KB.
A layout that cannot fit even split 16 ways is refused before any launch (gptq_gemm then runs the
tensor-core kernel); that may only happen for K beyond 28672.
"""
import itertools
import os
import shutil
import subprocess
import tempfile

import pytest

ROOT = os.path.dirname(os.path.dirname(os.path.abspath(__file__)))
CSRC = os.path.join(ROOT, "gptq_bit_weight_gemm_gb300", "csrc")
SMEM_PER_CTA = 227 * 1024
PER = {2: 16, 3: 32, 4: 8, 8: 4}


@pytest.fixture(scope="module")
def probe():
    nvcc = shutil.which("nvcc") or "/usr/local/cuda/bin/nvcc"
    if not os.path.exists(nvcc):
        pytest.skip("needs nvcc")
    tmp = tempfile.mkdtemp(prefix="geometry_probe_")
    exe = os.path.join(tmp, "probe")
    subprocess.run([nvcc, "-gencode", "arch=compute_103a,code=sm_103a", "-std=c++17",
                    "--expt-relaxed-constexpr", "-I", os.path.join(ROOT, "include"), "-I", CSRC,
                    os.path.join(ROOT, "tests", "geometry_probe.cu"), "-o", exe], check=True)
    yield exe
    shutil.rmtree(tmp, ignore_errors=True)


def _problems():
    for bits, K, N, M in itertools.product((2, 3, 4, 8), (256, 512, 1024, 4096, 5120, 8192, 16384, 28672,
                                                          53248),
                                           (128, 384, 4096, 11008, 14336), (1, 2, 5, 8, 9, 16, 17, 32)):
        for group in (32, 64, 128, K):
            if K % group:
                continue
            foldable = group % (4 * PER[bits]) == 0
            for fold, gidx in ((True, False), (False, False), (False, True)):
                if fold and not foldable:
                    continue
                for E in (1, 2, 8):    # 2: two 16-token blocks side by side (the token split)
                    if gidx and E > 1:
                        continue
                    for regs in (64, 216):    # the decode kernels compile to 64 .. 214 registers
                        yield bits, K, N, M, group, int(fold), int(gidx), E, regs


def _split(total, parts, idx):
    return total * idx // parts, total * (idx + 1) // parts


def test_launch_geometry_fits_and_covers(probe):
    probs = list(_problems())
    out = subprocess.run([probe], input="".join("%d %d %d %d %d %d %d %d %d\n" % p for p in probs),
                         capture_output=True, text=True, check=True).stdout.split("\n")
    assert len([l for l in out if l]) == len(probs)
    bad, refused = [], []
    for p, line in zip(probs, out):
        bits, K, N, M, group, fold, gidx, E, regs = p
        (fits, cs, tpc, ct, crows, slot, cbytes, nbuf, maxg, fullg, fullk, per, rows, units, slabs, chunks,
         smem) = map(int, line.split())
        if not fits:
            # refused (nothing launched): only where no wider split exists
            refused.append(p)
            if not ((cs == 16 or units < 4 * 2 * cs * 4) and smem > SMEM_PER_CTA):
                bad.append((p, line, ["refused although a wider split remained"]))
            continue
        G = K // group
        tiles_total = (units + 3) // 4
        checks = {
            "cluster size": cs in (1, 2, 4, 8, 16),
            "K covered": tpc * cs >= tiles_total and tpc == (tiles_total + cs - 1) // cs,
            "box rows <= 256": 1 <= crows <= 256 and crows == ct * 4 * rows,
            "slot 1024-aligned": slot % 1024 == 0 and slot >= crows * 128 and cbytes == 4 * slot,
            "buffers": 1 <= nbuf <= 16 and nbuf <= max(chunks, 2) and chunks * ct >= tpc,
            "shared memory": smem <= SMEM_PER_CTA,
        }
        if fold:
            need = 0
            for r in range(cs):
                b, e = _split(tiles_total, cs, r)
                if e > b:
                    need = max(need, min((e * 4 * per - 1) // group, G - 1) - (b * 4 * per) // group + 1)
            checks["group constants"] = maxg >= need
        elif fullg:
            checks["dequant staging"] = fullg * 128 * 4 + fullk * 2 <= 24 * 1024 and \
                (fullg == G if gidx else fullg >= 1)
        failed = [k for k, ok in checks.items() if not ok]
        if failed:
            bad.append((p, line, failed))
    assert not bad, "%d layouts break a rule, e.g. %s" % (len(bad), bad[:3])
    # every K up to 28672 (70B-class down projections) keeps the decode kernels at any token count
    assert not [p for p in refused if p[1] <= 28672], [p for p in refused if p[1] <= 28672][:5]
