"""CPU oracle for the GPTQ mixed-precision GEMM -- TEST INFRASTRUCTURE ONLY.

Only the test suite, the smoke check and the benchmark's CPU-baseline leg may import this
package.  The product library never imports, links or runs it, and it never imports the
product library: the two share no code.

The arithmetic lives in ``gptq_oracle.c`` (plain single-threaded C, written from the page
"增强 vLLM 对 GPTQv2 格式的支持：分析与实现", sections "LLM 的权重量化", "从 GPTQv1 到
GPTQv2" and "调整细节：根据格式选择处理方式").  This module only marshals numpy arrays
to and from it.

Conventions: 16-bit floats travel as ``uint16`` bit patterns with a dtype code
(``F16 = 0``, ``BF16 = 1``); packed words are ``int32`` arrays; ``fmt`` is ``V1 = 1``
(zero stored as clamp(zero - 1), plus one at run time) or ``V2 = 2`` (zero stored as is).

Every function here is pinned by ``tests/test_oracle_pins.py`` (hand-worked groups,
packed words, closed forms, library routines and brute force); no function is
"parity unpinned" except the bit layout of real-world checkpoints, of which there are
none to compare against.
"""
import ctypes
import numpy as np

from . import build as _build

F16, BF16 = 0, 1
V1, V2 = 1, 2


class OracleError(RuntimeError):
    pass


_SIGS = {
    "oracle_unpack_k": "PIIIP",
    "oracle_unpack_n": "PIIIP",
    "oracle_pack_k": "PIIIP",
    "oracle_pack_n": "PIIIP",
    "oracle_dequant_f32": "PPPPIIIIIP",
    "oracle_dequant": "PPPPIIIIIIP",
    "oracle_gemm_w32": "PIIIPIPIPP",
    "oracle_gemm": "PIIIPPPPIIIIPIPP",
    "oracle_repack_v1_to_v2": "PPIII",
    "oracle_quantize_rtn": "PIIIIPIPPP",
    "oracle_store_zeros": "PLIIP",
}
_CT = {"P": ctypes.c_void_p, "I": ctypes.c_int, "L": ctypes.c_int64}


def load_library(path):
    """Open an oracle shared library and declare its signatures."""
    lib = ctypes.CDLL(path)
    for name, args in _SIGS.items():
        fn = getattr(lib, name)
        fn.argtypes = [_CT[c] for c in args]
        fn.restype = ctypes.c_int
    for name in ("oracle_half_to_double_array", "oracle_bf16_to_double_array",
                 "oracle_float_to_half_array", "oracle_float_to_bf16_array"):
        fn = getattr(lib, name)
        fn.argtypes = [ctypes.c_void_p, ctypes.c_int64, ctypes.c_void_p]
        fn.restype = None
    return lib


_lib = None


def _load():
    global _lib
    if _lib is None:
        _lib = load_library(_build.build())
    return _lib


def _p(a):
    return None if a is None else a.ctypes.data_as(ctypes.c_void_p)


def _c(a, dtype):
    return None if a is None else np.ascontiguousarray(a, dtype=dtype)


def _check(rc, what):
    if rc != 0:
        raise OracleError("%s failed with code %d" % (what, rc))


def n_groups(K, group):
    return 1 if group == -1 else K // group


class Oracle:
    """The oracle's functions bound to one compiled copy of gptq_oracle.c."""

    def __init__(self, lib):
        self._lib = lib

    # ---------------------------------------------------------------- 16-bit float formats
    def to_double(self, bits16, dtype):
        """Decode fp16 / bf16 bit patterns to float64."""
        x = _c(bits16, np.uint16)
        out = np.empty(x.shape, np.float64)
        fn = (self._lib.oracle_half_to_double_array if dtype == F16
              else self._lib.oracle_bf16_to_double_array)
        fn(_p(x), x.size, _p(out))
        return out

    def round_to(self, x, dtype):
        """Round float32 values to fp16 / bf16 (nearest, ties to even); return bit patterns."""
        x = _c(x, np.float32)
        out = np.empty(x.shape, np.uint16)
        fn = (self._lib.oracle_float_to_half_array if dtype == F16
              else self._lib.oracle_float_to_bf16_array)
        fn(_p(x), x.size, _p(out))
        return out

    # ---------------------------------------------------------------- packing
    def unpack_k(self, qweight, K, N, bits):
        qw = _c(qweight, np.int32)
        q = np.empty((K, N), np.uint8)
        _check(self._lib.oracle_unpack_k(_p(qw), K, N, bits, _p(q)), "unpack_k")
        return q

    def unpack_n(self, qzeros, G, N, bits):
        qz = _c(qzeros, np.int32)
        z = np.empty((G, N), np.int32)
        _check(self._lib.oracle_unpack_n(_p(qz), G, N, bits, _p(z)), "unpack_n")
        return z

    def pack_k(self, q, bits):
        q = _c(q, np.uint8)
        K, N = q.shape
        out = np.empty((K * bits // 32, N), np.int32)
        _check(self._lib.oracle_pack_k(_p(q), K, N, bits, _p(out)), "pack_k")
        return out

    def pack_n(self, z, bits):
        z = _c(z, np.int32)
        G, N = z.shape
        out = np.empty((G, N * bits // 32), np.int32)
        _check(self._lib.oracle_pack_n(_p(z), G, N, bits, _p(out)), "pack_n")
        return out

    # ---------------------------------------------------------------- dequant / GEMM
    def dequant_f32(self, qweight, qzeros, scales, g_idx, K, N, bits, group, fmt):
        """Exact fp32 dequantized weights w32[K, N] = (q - zero) * scale."""
        qw, qz = _c(qweight, np.int32), _c(qzeros, np.int32)
        sc, gi = _c(scales, np.uint16), _c(g_idx, np.int32)
        out = np.empty((K, N), np.float32)
        _check(self._lib.oracle_dequant_f32(_p(qw), _p(qz), _p(sc), _p(gi), K, N, bits, group,
                                          fmt, _p(out)), "dequant_f32")
        return out

    def dequant(self, qweight, qzeros, scales, g_idx, K, N, bits, group, fmt, out_dtype):
        """Dequantized weights rounded once to fp16/bf16 (uint16 bit patterns)."""
        qw, qz = _c(qweight, np.int32), _c(qzeros, np.int32)
        sc, gi = _c(scales, np.uint16), _c(g_idx, np.int32)
        out = np.empty((K, N), np.uint16)
        _check(self._lib.oracle_dequant(_p(qw), _p(qz), _p(sc), _p(gi), K, N, bits, group, fmt,
                                      out_dtype, _p(out)), "dequant")
        return out

    def gemm_w32(self, A, a_dtype, w32, rows=None):
        """C = A @ w32 in fp32 (k ascending) and the bound B = sum_k |A * w32|, for `rows`."""
        A = _c(A, np.uint16)
        w = _c(w32, np.float32)
        M, K = A.shape
        N = w.shape[1]
        r = None if rows is None else _c(rows, np.int32)
        nr = M if r is None else r.size
        C = np.empty((nr, N), np.float32)
        B = np.empty((nr, N), np.float64)
        _check(self._lib.oracle_gemm_w32(_p(A), M, K, a_dtype, _p(w), N, _p(r), nr, _p(C), _p(B)),
               "gemm_w32")
        return C, B

    def gemm(self, A, a_dtype, qweight, qzeros, scales, g_idx, N, bits, group, fmt, rows=None):
        """Reference C = A @ dequant_f32(...) (fp32, k ascending) and its bound B."""
        A = _c(A, np.uint16)
        M, K = A.shape
        qw, qz = _c(qweight, np.int32), _c(qzeros, np.int32)
        sc, gi = _c(scales, np.uint16), _c(g_idx, np.int32)
        r = None if rows is None else _c(rows, np.int32)
        nr = M if r is None else r.size
        C = np.empty((nr, N), np.float32)
        B = np.empty((nr, N), np.float64)
        _check(self._lib.oracle_gemm(_p(A), M, K, a_dtype, _p(qw), _p(qz), _p(sc), _p(gi), N, bits,
                                   group, fmt, _p(r), nr, _p(C), _p(B)), "gemm")
        return C, B

    def gemm_grouped(self, A, a_dtype, offsets, qweight, qzeros, scales, N, bits, group, fmt):
        """Mixture-of-experts reference: expert e multiplies rows [offsets[e], offsets[e + 1]) of
        A by its own dequantized weight, exactly as gemm() does for one weight (page "4.3
        Weight-only INT4 量化：GPTQ、AWQ 与 Marlin Kernel", section 7: the expert weights of a
        MoE model are GPTQ checkpoints like any other).  qweight, qzeros and scales are indexed
        by expert first.  Returns (C, B) over every row of A; rows no expert owns stay NaN."""
        A = _c(A, np.uint16)
        rows = A.shape[0]
        C = np.full((rows, N), np.nan, np.float32)
        B = np.full((rows, N), np.nan, np.float64)
        for e in range(len(offsets) - 1):
            lo, hi = int(offsets[e]), int(offsets[e + 1])
            if hi > lo:
                C[lo:hi], B[lo:hi] = self.gemm(A[lo:hi], a_dtype, qweight[e], qzeros[e], scales[e],
                                               None, N, bits, group, fmt)
        return C, B

    def repack_v1_to_v2(self, qz_v1, G, N, bits):
        qz = _c(qz_v1, np.int32)
        out = np.empty_like(qz)
        rc = self._lib.oracle_repack_v1_to_v2(_p(qz), _p(out), G, N, bits)
        _check(rc, "repack_v1_to_v2")
        return out

    # ---------------------------------------------------------------- checkpoint writer
    def quantize_rtn(self, W, bits, group, g_idx=None, sym=False):
        """Round-to-nearest quantizer: returns (q[K,N] uint8, zero[G,N] int32, scale[G,N] fp16 bits)."""
        W = _c(W, np.float32)
        K, N = W.shape
        G = n_groups(K, group)
        gi = _c(g_idx, np.int32)
        q = np.empty((K, N), np.uint8)
        z = np.empty((G, N), np.int32)
        s = np.empty((G, N), np.uint16)
        _check(self._lib.oracle_quantize_rtn(_p(W), K, N, bits, group, _p(gi), int(sym), _p(q),
                                           _p(z), _p(s)), "quantize_rtn")
        return q, z, s

    def store_zeros(self, zero, bits, fmt):
        """Zeros as a checkpoint stores them: v2 exact, v1 clamp(zero - 1)."""
        z = _c(zero, np.int32)
        out = np.empty_like(z)
        _check(self._lib.oracle_store_zeros(_p(z), z.size, bits, fmt, _p(out)), "store_zeros")
        return out

    def make_checkpoint(self, W, bits, group, g_idx=None, sym=False, fmt=V2):
        """Quantize W and pack it as a GPTQ checkpoint of format `fmt`.

        Returns a dict with qweight [K*bits/32, N], qzeros [G, N*bits/32], scales [G, N]
        (fp16 bits), g_idx (or None) and the unpacked q / zero for inspection.
        """
        q, zero, scales = self.quantize_rtn(W, bits, group, g_idx, sym)
        stored = self.store_zeros(zero, bits, fmt)
        return {
            "qweight": self.pack_k(q, bits),
            "qzeros": self.pack_n(stored, bits),
            "scales": scales,
            "g_idx": None if g_idx is None else np.ascontiguousarray(g_idx, np.int32),
            "q": q,
            "zero": zero,
            "bits": bits,
            "group": group,
            "fmt": fmt,
        }


_default = None


def default():
    """The oracle built from gptq_oracle.c in this directory."""
    global _default
    if _default is None:
        _default = Oracle(_load())
    return _default


def __getattr__(name):
    # module-level access (oracle.gemm, oracle.dequant, ...) goes to the default build
    if name.startswith("_"):
        raise AttributeError(name)
    return getattr(default(), name)
