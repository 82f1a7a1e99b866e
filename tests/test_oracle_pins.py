"""Pins for the CPU oracle: checks against what the page and mathematics fix, not against
the oracle itself.

Page: "增强 vLLM 对 GPTQv2 格式的支持：分析与实现" (xxxxyu.github.io):
  section "LLM 的权重量化"          -- quantizer, inverse, symmetric zero;
  section "从 GPTQv1 到 GPTQv2"      -- v1 stores clamp(zero - 1) (+1 at run time), v2 stores
                                       zero; v1 -> v2 lossless; INT2 v1 range [0,3] -> [1,3];
  section "调整细节：根据格式选择处理方式" -- zero_offset = use_v2_format ? 0 : 1; 16 two-bit
                                       codes per int32 word.

Page: "4.3 Weight-only INT4 量化：GPTQ、AWQ 与 Marlin Kernel", section 7 -- the expert weights
  of a MoE model are GPTQ checkpoints like any other (the grouped GEMM).

Kinds of pin used (each check below names its kind):
  golden     hand-worked values in tests/golden/ (with their derivation);
  closed     closed forms and invariants (error bound, losslessness, permutation invariance);
  library    a special case that reduces to numpy / torch (fp16/bf16 rounding, float64 matmul);
  brute      tiny inputs recomputed in pure Python from an independent big-integer packer
             and exact (math.fsum) sums.

Every check is a function of an ``Oracle`` object so that ``test_planted_mistakes`` can run
the same suite against copies of the oracle with a mistake planted in them, and show that
each plausible mistake fails at least one pin.
"""
import itertools
import json
import math
import os
import shutil
import subprocess
import tempfile

import numpy as np
import pytest
import torch

import oracle
from oracle import F16, BF16, V1, V2

GOLDEN = os.path.join(os.path.dirname(os.path.abspath(__file__)), "golden")


def _golden(name):
    with open(os.path.join(GOLDEN, name)) as f:
        return json.load(f)


def _py_pack_stream(codes, bits):
    """Independent packer: one big integer, code i shifted to bit b*i, cut into words."""
    acc = 0
    for i, c in enumerate(codes):
        acc |= int(c) << (bits * i)
    nwords = len(codes) * bits // 32
    return [((acc >> (32 * w)) & 0xFFFFFFFF) for w in range(nwords)]


def _as_i32(words):
    return np.array(words, dtype=np.uint32).view(np.int32)


def _py_pack_k(q, bits):
    K, N = q.shape
    out = np.zeros((K * bits // 32, N), np.int32)
    for n in range(N):
        out[:, n] = _as_i32(_py_pack_stream(q[:, n], bits))
    return out


def _py_pack_n(z, bits):
    G, N = z.shape
    out = np.zeros((G, N * bits // 32), np.int32)
    for g in range(G):
        out[g, :] = _as_i32(_py_pack_stream(z[g, :], bits))
    return out


def _rows_for(length, bits):
    """Smallest multiple of `length` that fills whole words (3-bit: multiples of 32)."""
    r = length
    while (r * bits) % 32 or (bits == 3 and r % 32):
        r += length
    return r


# ----------------------------------------------------------------------------- checks
def check_hand_worked_groups(orc):
    """golden: scale, zero, codes and w_hat of hand-worked groups, v1 and v2."""
    for g in _golden("hand_worked_groups.json")["groups"]:
        bits, w = g["bits"], np.array(g["w"], np.float32)
        K = _rows_for(len(w), bits)
        N = 32 if bits == 3 else 32 // bits
        col = np.resize(w, K)
        W = np.repeat(col[:, None], N, axis=1)
        q, zero, scale = orc.quantize_rtn(W, bits, K, None, g["sym"])
        s = orc.to_double(scale, F16)
        assert np.all(s == g["scale"]), (g["name"], s[0, 0])
        assert np.all(zero == g["zero"]), (g["name"], zero[0, 0])
        assert np.array_equal(q[: len(w), 0], np.array(g["q"])), (g["name"], q[: len(w), 0])
        for fmt, key in ((V2, "w_hat_v2"), (V1, "w_hat_v1")):
            stored = orc.store_zeros(zero, bits, fmt)
            if fmt == V1:
                assert np.all(stored == g["v1_stored_zero"]), (g["name"], stored[0, 0])
            w_hat = orc.dequant_f32(orc.pack_k(q, bits), orc.pack_n(stored, bits), scale, None,
                                    K, N, bits, K, fmt)
            assert np.array_equal(w_hat[: len(w), 0], np.array(g[key], np.float32)), \
                (g["name"], fmt, w_hat[: len(w), 0])


def check_symmetric_zero(orc):
    """golden/closed: symmetric zero = round((2^b - 1)/2) for every width."""
    zs = _golden("hand_worked_groups.json")["symmetric_zeros"]
    rng = np.random.default_rng(11)
    for bits in (2, 3, 4, 8):
        W = rng.standard_normal((128, 32), dtype=np.float32)
        _, zero, _ = orc.quantize_rtn(W, bits, 32, None, True)
        assert np.all(zero == zs[str(bits)]), (bits, np.unique(zero))


def check_packed_words(orc):
    """golden: words packed from listed codes, and codes unpacked from listed words."""
    for c in _golden("packed_words.json")["cases"]:
        bits, codes = c["bits"], np.array(c["codes"], np.uint8)
        words = _as_i32([int(x, 16) for x in c["words"]])
        K = len(codes)
        got = orc.pack_k(codes.reshape(K, 1), bits)[:, 0]
        assert np.array_equal(got, words), (bits, [hex(x) for x in got.view(np.uint32)])
        assert np.array_equal(orc.unpack_k(words.reshape(-1, 1), K, 1, bits)[:, 0], codes)
        got_n = orc.pack_n(codes.reshape(1, K).astype(np.int32), bits)[0]
        assert np.array_equal(got_n, words), bits
        assert np.array_equal(orc.unpack_n(words.reshape(1, -1), 1, K, bits)[0], codes)


def check_pack_exhaustive(orc):
    """brute: every code at every position, both directions, against the big-int packer."""
    for bits in (2, 3, 4, 8):
        per = 32 if bits == 3 else 32 // bits       # codes per packing unit
        L = 1 << bits
        K = per * 2
        q = np.array([[(k + n) % L for n in range(L)] for k in range(K)], np.uint8)
        qw = orc.pack_k(q, bits)
        assert np.array_equal(qw, _py_pack_k(q, bits)), bits
        assert np.array_equal(orc.unpack_k(qw, K, L, bits), q), bits
        z = q.T.astype(np.int32).copy()            # [L, K]: codes along N
        qz = orc.pack_n(z, bits)
        assert np.array_equal(qz, _py_pack_n(z, bits)), bits
        assert np.array_equal(orc.unpack_n(qz, L, K, bits), z), bits


def check_v1_v2_lossless(orc):
    """closed: v1 -> v2 repack returns z for every z in [1, 2^b-1]; z = 0 becomes 1 under v1;
    a v1 field of 2^b - 1 cannot be repacked."""
    for bits in (2, 3, 4, 8):
        maxq = (1 << bits) - 1
        N = 32 * max(1, (maxq + 1) // 32)
        z = (np.arange(N) % maxq + 1).astype(np.int32).reshape(1, N)     # 1..maxq
        v1 = orc.pack_n(orc.store_zeros(z, bits, V1), bits)
        v2 = orc.pack_n(orc.store_zeros(z, bits, V2), bits)
        assert np.array_equal(orc.repack_v1_to_v2(v1, 1, N, bits), v2), bits
        zero0 = np.zeros((1, N), np.int32)
        assert np.all(orc.store_zeros(zero0, bits, V1) == 0)
        bad = orc.pack_n(np.full((1, N), maxq, np.int32), bits)
        with pytest.raises(oracle.OracleError):
            orc.repack_v1_to_v2(bad, 1, N, bits)
    # INT2: the runtime zeros a v1 checkpoint can express are exactly {1, 2, 3}
    z = np.array([[0, 1, 2, 3] * 8], np.int32)
    stored = orc.store_zeros(z, 2, V1)
    q = np.zeros((16, 32), np.uint8)
    s = np.full((1, 32), 0x3C00, np.uint16)                               # scale 1.0
    w = orc.dequant_f32(orc.pack_k(q, 2), orc.pack_n(stored, 2), s, None, 16, 32, 2, 16, V1)
    assert sorted(set((-w[0]).astype(int).tolist())) == [1, 2, 3]


def check_v1_v2_same_dequant(orc):
    """closed: the v1 and v2 encodings of the same zeros (all >= 1) dequantize identically,
    and a v1 checkpoint read as v2 is off by exactly one step."""
    rng = np.random.default_rng(5)
    for bits in (2, 3, 4, 8):
        K, N, group = 128, 64, 32
        G = K // group
        q = rng.integers(0, 1 << bits, (K, N)).astype(np.uint8)
        z = rng.integers(1, 1 << bits, (G, N)).astype(np.int32)
        s = orc.round_to(rng.uniform(1e-3, 1e-1, (G, N)).astype(np.float32), F16)
        qw = orc.pack_k(q, bits)
        w2 = orc.dequant_f32(qw, orc.pack_n(orc.store_zeros(z, bits, V2), bits), s, None, K, N,
                             bits, group, V2)
        qz1 = orc.pack_n(orc.store_zeros(z, bits, V1), bits)
        w1 = orc.dequant_f32(qw, qz1, s, None, K, N, bits, group, V1)
        assert np.array_equal(w1, w2), bits
        w1_as_v2 = orc.dequant_f32(qw, qz1, s, None, K, N, bits, group, V2)
        step = np.repeat(orc.to_double(s, F16), group, axis=0)
        assert np.array_equal(w1_as_v2.astype(np.float64) - w2, step), bits


def check_quantize_error_bound(orc):
    """closed: |w - w_hat| <= scale/2 for codes that were not clamped; with the stored (fp16)
    scale, |w - w_hat| <= scale/2 + (2^b - 1)|scale - scale32| for every asymmetric entry of
    a group whose zero was not clamped."""
    rng = np.random.default_rng(7)
    for bits in (2, 3, 4, 8):
        K, N, group = 256, 64, 32
        G = K // group
        W = (rng.standard_normal((K, N), dtype=np.float32) * np.float32(0.02))
        q, zero, sc = orc.quantize_rtn(W, bits, group, None, False)
        s = np.repeat(orc.to_double(sc, F16), group, axis=0)
        w_hat = orc.dequant_f32(orc.pack_k(q, bits), orc.pack_n(zero, bits), sc, None, K, N, bits,
                                group, V2).astype(np.float64)
        err = np.abs(W.astype(np.float64) - w_hat)
        maxq = (1 << bits) - 1
        free = (q > 0) & (q < maxq)
        assert np.all(err[free] <= s[free] / 2 * (1 + 2.0 ** -20)), bits
        Wg = W.reshape(G, group, N)
        s32 = ((Wg.max(axis=1) - Wg.min(axis=1)) / np.float32(maxq)).astype(np.float64)
        zfree = np.repeat((zero > 0) & (zero < maxq), group, axis=0)
        bound = s / 2 + maxq * np.abs(s - np.repeat(s32, group, axis=0))
        assert np.all(err[zfree] <= bound[zfree] * (1 + 2.0 ** -20)), bits


def check_fp16_bf16_rounding(orc):
    """library: fp16 rounding equals numpy's float32 -> float16 cast, bf16 rounding equals
    torch's float32 -> bfloat16 cast (both round to nearest, ties to even), including ties,
    subnormals and overflow; the decoders equal numpy / torch on all 65536 patterns."""
    rng = np.random.default_rng(3)
    x = np.concatenate([
        rng.standard_normal(20000).astype(np.float32) * np.float32(10.0) ** rng.integers(-9, 6, 20000).astype(np.float32),
        np.array([0.0, -0.0, 65504.0, 65519.996, 65520.0, -65520.0, 1e-8, 2.0 ** -25, 3 * 2.0 ** -26,
                  2.0 ** -24, 1e30, -1e30, 3.0e38], np.float32),
    ])
    h = np.arange(0x7C00, dtype=np.uint32).astype(np.uint16).view(np.float16).astype(np.float32)
    mid = ((h[:-1].astype(np.float64) + h[1:].astype(np.float64)) / 2).astype(np.float32)
    x = np.concatenate([x, mid, -mid])
    with np.errstate(over="ignore"):
        ref16 = x.astype(np.float16).view(np.uint16)
    assert np.array_equal(orc.round_to(x, F16), ref16)
    bf = torch.from_numpy(x).to(torch.bfloat16).view(torch.int16).numpy().view(np.uint16)
    assert np.array_equal(orc.round_to(x, BF16), bf)
    allp = np.arange(65536, dtype=np.uint32).astype(np.uint16)
    ref16 = allp.view(np.float16).astype(np.float64)
    got16 = orc.to_double(allp, F16)
    assert np.array_equal(np.isnan(got16), np.isnan(ref16))
    ok = ~np.isnan(ref16)
    assert np.array_equal(got16[ok], ref16[ok]) and np.array_equal(np.signbit(got16[ok]), np.signbit(ref16[ok]))
    refbf = torch.from_numpy(allp.view(np.int16)).view(torch.bfloat16).double().numpy()
    gotbf = orc.to_double(allp, BF16)
    ok = ~np.isnan(refbf)
    assert np.array_equal(gotbf[ok], refbf[ok]) and np.array_equal(np.isnan(gotbf), np.isnan(refbf))


def check_gemm_vs_float64(orc):
    """library: the fp32 triple loop agrees with numpy's float64 matmul within fp32 summation
    error, and the bound B equals |A| @ |W| in float64."""
    rng = np.random.default_rng(9)
    for dtype, bits, group, act in ((F16, 4, 64, False), (BF16, 3, 128, True), (F16, 8, -1, False)):
        M, K, N = 6, 512, 96
        G = oracle.n_groups(K, group)
        q = rng.integers(0, 1 << bits, (K, N)).astype(np.uint8)
        z = rng.integers(0, 1 << bits, (G, N)).astype(np.int32)
        s = orc.round_to(rng.uniform(1e-3, 5e-2, (G, N)).astype(np.float32), F16)
        gi = rng.integers(0, G, K).astype(np.int32) if act else None
        qw, qz = orc.pack_k(q, bits), orc.pack_n(z, bits)
        A = orc.round_to(rng.standard_normal((M, K)).astype(np.float32), dtype)
        C, B = orc.gemm(A, dtype, qw, qz, s, gi, N, bits, group, V2)
        W = orc.dequant_f32(qw, qz, s, gi, K, N, bits, group, V2).astype(np.float64)
        A64 = orc.to_double(A, dtype)
        ref = A64 @ W
        absb = np.abs(A64) @ np.abs(W)
        assert np.allclose(B, absb, rtol=1e-12, atol=0), dtype
        assert np.all(np.abs(C - ref) <= 1.01 * K * 2.0 ** -24 * absb + 1e-30), dtype
        # rows selection returns the same rows
        C2, _ = orc.gemm(A, dtype, qw, qz, s, gi, N, bits, group, V2, rows=np.array([4, 1]))
        assert np.array_equal(C2, C[[4, 1]])


def check_identity_and_one_hot(orc):
    """closed: A = I gives C = w32 exactly; one-hot rows of A select single rows of W."""
    rng = np.random.default_rng(13)
    K, N, bits, group = 64, 32, 4, 32
    G = K // group
    q = rng.integers(0, 16, (K, N)).astype(np.uint8)
    z = rng.integers(0, 16, (G, N)).astype(np.int32)
    s = orc.round_to(rng.uniform(1e-3, 5e-2, (G, N)).astype(np.float32), F16)
    qw, qz = orc.pack_k(q, bits), orc.pack_n(z, bits)
    W = orc.dequant_f32(qw, qz, s, None, K, N, bits, group, V1)
    for dtype in (F16, BF16):
        I = orc.round_to(np.eye(K, dtype=np.float32), dtype)
        C, B = orc.gemm(I, dtype, qw, qz, s, None, N, bits, group, V1)
        assert np.array_equal(C, W) and np.array_equal(B, np.abs(W).astype(np.float64))
        two = np.zeros((3, K), np.float32)
        two[0, 5] = 2.0
        two[1, 63] = -0.5
        two[2, 0] = 1.0
        C, _ = orc.gemm(orc.round_to(two, dtype), dtype, qw, qz, s, None, N, bits, group, V1)
        assert np.array_equal(C, np.stack([2 * W[5], -0.5 * W[63], W[0]]))


def check_group_index_forms(orc):
    """closed: g_idx = k // group gives the same weights as no g_idx; group = -1 is one group;
    permuting K rows of (A's columns, codes, g_idx) together permutes W's rows and leaves C
    within fp32 reordering error (act-order invariance)."""
    rng = np.random.default_rng(17)
    K, N, bits, group = 256, 64, 3, 64
    G = K // group
    q = rng.integers(0, 8, (K, N)).astype(np.uint8)
    z = rng.integers(0, 8, (G, N)).astype(np.int32)
    s = orc.round_to(rng.uniform(1e-3, 5e-2, (G, N)).astype(np.float32), F16)
    qw, qz = orc.pack_k(q, bits), orc.pack_n(z, bits)
    plain = orc.dequant_f32(qw, qz, s, None, K, N, bits, group, V2)
    explicit = orc.dequant_f32(qw, qz, s, (np.arange(K) // group).astype(np.int32), K, N, bits,
                               group, V2)
    assert np.array_equal(plain, explicit)
    one = orc.dequant_f32(qw, qz[:1], s[:1], None, K, N, bits, -1, V2)
    ref = (q.astype(np.float64) - z[0]) * orc.to_double(s[0], F16)
    assert np.array_equal(one, ref.astype(np.float32))
    gi = rng.integers(0, G, K).astype(np.int32)
    A = orc.round_to(rng.standard_normal((4, K)).astype(np.float32), F16)
    C, B = orc.gemm(A, F16, qw, qz, s, gi, N, bits, group, V2)
    W = orc.dequant_f32(qw, qz, s, gi, K, N, bits, group, V2)
    p = rng.permutation(K)
    qw_p = orc.pack_k(q[p], bits)
    W_p = orc.dequant_f32(qw_p, qz, s, gi[p], K, N, bits, group, V2)
    assert np.array_equal(W_p, W[p])
    C_p, _ = orc.gemm(np.ascontiguousarray(A[:, p]), F16, qw_p, qz, s, gi[p], N, bits, group, V2)
    assert np.all(np.abs(C_p - C) <= 2 * K * 2.0 ** -24 * B)


def check_brute_force_tiny(orc):
    """brute: M in {1,2,3}, K in {32,64,96}, N in {32,64}; every width x format x act-order x
    dtype.  Checkpoints are built from chosen codes, zeros and scales with the independent
    big-int packer; every weight and every sum is recomputed in pure Python (exact products,
    math.fsum)."""
    rng = np.random.default_rng(21)
    shapes = list(itertools.product((1, 2, 3), (32, 64, 96), (32, 64)))
    combos = list(itertools.product((2, 3, 4, 8), (V1, V2), (False, True), (F16, BF16)))
    for i, (bits, fmt, act, dtype) in enumerate(combos):
        M, K, N = shapes[i % len(shapes)]
        group = (32, -1, K)[i % 3] if not act else 32
        G = oracle.n_groups(K, group)
        L = 1 << bits
        q = rng.integers(0, L, (K, N)).astype(np.uint8)
        stored = rng.integers(0, L, (G, N)).astype(np.int32)
        s16 = rng.uniform(1e-3, 1e-1, (G, N)).astype(np.float16)
        s = s16.view(np.uint16)
        gi = rng.integers(0, G, K).astype(np.int32) if act else None
        a32 = rng.standard_normal((M, K)).astype(np.float32)
        if dtype == F16:
            A = a32.astype(np.float16).view(np.uint16)
            a64 = A.view(np.float16).astype(np.float64)
        else:
            t = torch.from_numpy(a32).to(torch.bfloat16)
            A = t.view(torch.int16).numpy().view(np.uint16)
            a64 = t.double().numpy()
        qw, qz = _py_pack_k(q, bits), _py_pack_n(stored, bits)
        off = 1 if fmt == V1 else 0
        w = [[0.0] * N for _ in range(K)]
        for k in range(K):
            g = int(gi[k]) if act else (0 if group == -1 else k // group)
            for n in range(N):
                w[k][n] = (int(q[k, n]) - (int(stored[g, n]) + off)) * float(s16[g, n])
        W = orc.dequant_f32(qw, qz, s, gi, K, N, bits, group, fmt)
        assert np.array_equal(W, np.array(w, np.float32)), (bits, fmt, act)
        Wr = orc.dequant(qw, qz, s, gi, K, N, bits, group, fmt, dtype)
        if dtype == F16:
            ref = np.array(w).astype(np.float16).view(np.uint16)
        else:
            ref = torch.tensor(w, dtype=torch.float64).to(torch.bfloat16).view(torch.int16).numpy().view(np.uint16)
        assert np.array_equal(Wr, ref), (bits, fmt, act, dtype)
        C, B = orc.gemm(A, dtype, qw, qz, s, gi, N, bits, group, fmt)
        for m in range(M):
            for n in range(N):
                terms = [float(a64[m, k]) * w[k][n] for k in range(K)]
                exact = math.fsum(terms)
                babs = math.fsum(abs(t) for t in terms)
                assert abs(B[m, n] - babs) <= 1e-12 * babs, (bits, fmt, act, dtype)
                assert abs(float(C[m, n]) - exact) <= 1.01 * K * 2.0 ** -24 * babs, \
                    (bits, fmt, act, dtype, m, n, float(C[m, n]), exact)


def check_grouped(orc):
    """brute + closed: the grouped (mixture-of-experts) GEMM.  Three experts (one without
    rows) plus a row no expert owns, every width x format x dtype; each expert's checkpoint is
    built from chosen codes with the independent packer and every sum recomputed with math.fsum.
    Then: one expert equals gemm() bit for bit, and reordering the experts (moving their row
    blocks with them) leaves every row bit-identical."""
    rng = np.random.default_rng(31)
    K, N, group = 64, 32, 32
    offsets = np.array([0, 2, 2, 5], np.int32)           # expert 1 has no rows; row 5 none
    rows = 6
    for bits, fmt, dtype in itertools.product((2, 3, 4, 8), (V1, V2), (F16, BF16)):
        E, G, L = 3, K // group, 1 << bits
        q = rng.integers(0, L, (E, K, N)).astype(np.uint8)
        stored = rng.integers(0, L, (E, G, N)).astype(np.int32)
        s16 = rng.uniform(1e-3, 1e-1, (E, G, N)).astype(np.float16)
        a32 = rng.standard_normal((rows, K)).astype(np.float32)
        if dtype == F16:
            A = a32.astype(np.float16).view(np.uint16)
            a64 = A.view(np.float16).astype(np.float64)
        else:
            t = torch.from_numpy(a32).to(torch.bfloat16)
            A = t.view(torch.int16).numpy().view(np.uint16)
            a64 = t.double().numpy()
        qw = np.stack([_py_pack_k(q[e], bits) for e in range(E)])
        qz = np.stack([_py_pack_n(stored[e], bits) for e in range(E)])
        sc = s16.view(np.uint16)
        off = 1 if fmt == V1 else 0
        C, B = orc.gemm_grouped(A, dtype, offsets, qw, qz, sc, N, bits, group, fmt)
        owner = [None] * rows
        for e in range(E):
            for r in range(offsets[e], offsets[e + 1]):
                owner[r] = e
        for r in range(rows):
            e = owner[r]
            if e is None:
                assert np.all(np.isnan(C[r])) and np.all(np.isnan(B[r])), (bits, fmt, r)
                continue
            for n in range(N):
                terms = [float(a64[r, k]) * (int(q[e, k, n]) - (int(stored[e, k // group, n]) + off))
                         * float(s16[e, k // group, n]) for k in range(K)]
                exact = math.fsum(terms)
                babs = math.fsum(abs(x) for x in terms)
                assert abs(B[r, n] - babs) <= 1e-12 * babs, (bits, fmt, dtype, r, n)
                assert abs(float(C[r, n]) - exact) <= 1.01 * K * 2.0 ** -24 * babs, \
                    (bits, fmt, dtype, r, n, float(C[r, n]), exact)
        # one expert: the plain GEMM
        C1, B1 = orc.gemm_grouped(A[:4], dtype, np.array([0, 4], np.int32), qw[:1], qz[:1], sc[:1],
                                  N, bits, group, fmt)
        Cg, Bg = orc.gemm(A[:4], dtype, qw[0], qz[0], sc[0], None, N, bits, group, fmt)
        assert np.array_equal(C1, Cg) and np.array_equal(B1, Bg), (bits, fmt, dtype)
        # experts in the order (2, 0, 1): rows 2..4 first, then 0..1
        perm = [2, 0, 1]
        blocks = [A[offsets[e]:offsets[e + 1]] for e in perm]
        A2 = np.concatenate(blocks + [A[5:]])
        off2 = np.concatenate([[0], np.cumsum([len(b) for b in blocks])]).astype(np.int32)
        C2, _ = orc.gemm_grouped(A2, dtype, off2, qw[perm], qz[perm], sc[perm], N, bits, group, fmt)
        assert np.array_equal(C2[:3], C[2:5]) and np.array_equal(C2[3:5], C[0:2]), (bits, fmt, dtype)


PIN_CHECKS = [
    check_hand_worked_groups,
    check_symmetric_zero,
    check_packed_words,
    check_pack_exhaustive,
    check_v1_v2_lossless,
    check_v1_v2_same_dequant,
    check_quantize_error_bound,
    check_fp16_bf16_rounding,
    check_gemm_vs_float64,
    check_identity_and_one_hot,
    check_group_index_forms,
    check_brute_force_tiny,
    check_grouped,
]


@pytest.mark.parametrize("check", PIN_CHECKS, ids=lambda c: c.__name__[6:])
def test_oracle_pin(check):
    check(oracle.default())


# ----------------------------------------------------------------------------- mutations
# Plausible mistakes, planted in copies of the oracle on the CPU: each must fail a pin.
MUTATIONS = [
    ("v1 offset inverted", "fmt == OR_FMT_V2 ? 0 : 1;", "fmt == OR_FMT_V2 ? 1 : 0;"),
    ("MSB-first bit order", "code |= ((word >> (pos % 32)) & 1u) << t;",
     "code |= ((word >> (pos % 32)) & 1u) << (bits - 1 - t);"),
    ("zero dropped", "(double)(q - z) * s", "(double)(q) * s"),
    ("zero sign flipped", "(double)(q - z) * s", "(double)(z - q) * s"),
    ("group index k % group", "(int)(k / group);", "(int)(k % group);"),
    ("activation k reversed", "A[m * K + k], a_dtype", "A[m * K + (K - 1 - k)], a_dtype"),
    ("round half up", "return rint(x / quantum) * quantum;",
     "return floor(x / quantum + 0.5) * quantum;"),
    ("zero sign in quantizer", "z = -rintf(wmin[i] / s[i]);", "z = rintf(wmin[i] / s[i]);"),
    ("v1 stores zero + 1", "fmt == OR_FMT_V1 ? zero[i] - 1 : zero[i];",
     "fmt == OR_FMT_V1 ? zero[i] + 1 : zero[i];"),
    ("symmetric zero floor", "z = rintf(maxq / 2.0f);", "z = floorf(maxq / 2.0f);"),
    ("bf16 with 7 significant bits", "or_round_sig(x, 8, -126)", "or_round_sig(x, 7, -126)"),
    ("fp16 subnormal scale", "ldexp((double)f, -24)", "ldexp((double)f, -25)"),
    ("bound without abs", "b[n] += fabs((double)a * (double)w[n]);", "b[n] += (double)a * (double)w[n];"),
    ("qzeros row stride N", "qzeros + (int64_t)g * zwords, 1, bits, n)",
     "qzeros + (int64_t)g * N, 1, bits, n)"),
    ("repack adds nothing", "or_stream_put(out + g * words, 1, bits, n, f + 1);",
     "or_stream_put(out + g * words, 1, bits, n, f);"),
    ("scale from fp32 not fp16", "s[i] = (float)oracle_half_to_double(h);", "s[i] = s32;"),
    ("min/max over wrong column", "if (w > wmax[(int64_t)g * N + n]) wmax[(int64_t)g * N + n] = w;",
     "if (w > wmax[(int64_t)g * N]) wmax[(int64_t)g * N] = w;"),
]


def _build_mutant(src, old, new, tmpdir, idx):
    assert src.count(old) == 1, old
    path = os.path.join(tmpdir, "mutant%d.c" % idx)
    with open(path, "w") as f:
        f.write(src.replace(old, new))
    lib = os.path.join(tmpdir, "libmutant%d.so" % idx)
    subprocess.run(["gcc", *oracle.build.CFLAGS, path, "-o", lib, "-lm"], check=True,
                   stderr=subprocess.DEVNULL)
    return oracle.Oracle(oracle.load_library(lib))


@pytest.mark.skipif(shutil.which("gcc") is None, reason="needs gcc")
def test_planted_mistakes_fail_a_pin():
    with open(oracle.build.SRC) as f:
        src = f.read()
    tmpdir = tempfile.mkdtemp(prefix="oracle_mutants_")
    try:
        survivors = []
        for idx, (what, old, new) in enumerate(MUTATIONS):
            orc = _build_mutant(src, old, new, tmpdir, idx)
            caught = False
            for check in PIN_CHECKS:
                try:
                    check(orc)
                except (AssertionError, oracle.OracleError, ValueError, IndexError):
                    caught = True
                    break
            if not caught:
                survivors.append(what)
        assert not survivors, "planted mistakes that no pin caught: %s" % survivors
    finally:
        shutil.rmtree(tmpdir, ignore_errors=True)


# Plausible mistakes in the grouped composition (Python), planted in copies of its source.
GROUPED_MUTATIONS = [
    ("previous expert's weight", "qweight[e], qzeros[e], scales[e]", "qweight[e - 1], qzeros[e - 1], scales[e - 1]"),
    ("expert 0's scales for all", "qzeros[e], scales[e]", "qzeros[e], scales[0]"),
    ("row range shifted", "lo, hi = int(offsets[e]), int(offsets[e + 1])",
     "lo, hi = int(offsets[e]) + 1, int(offsets[e + 1]) + 1"),
    ("format ignored", "None, N, bits, group, fmt)", "None, N, bits, group, V2)"),
]


def test_planted_mistakes_in_grouped_fail_a_pin():
    import inspect
    import textwrap
    src = textwrap.dedent(inspect.getsource(oracle.Oracle.gemm_grouped))
    survivors = []
    for what, old, new in GROUPED_MUTATIONS:
        assert src.count(old) == 1, old
        ns = {"np": np, "_c": oracle._c, "V2": V2}
        exec(src.replace(old, new), ns)
        orc = oracle.Oracle(oracle.default()._lib)
        orc.gemm_grouped = ns["gemm_grouped"].__get__(orc)
        try:
            check_grouped(orc)
            survivors.append(what)
        except (AssertionError, oracle.OracleError, ValueError, IndexError):
            pass
    assert not survivors, "planted mistakes that no pin caught: %s" % survivors
