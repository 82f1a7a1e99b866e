"""GB300 (sm_103a) GPTQ mixed-precision GEMM -- Python binding of the C ABI (include/gptq.h).

Argument marshalling only: every step of the computation runs in the CUDA library
``_lib/libgptq_gb300.so`` (built in-tree by ``build.py``).  PyTorch supplies device memory
and streams.  There is no fallback: if the library is missing or the device is not a GB300
(sm_103), calls raise ``GPTQError``.

Operations (page "增强 vLLM 对 GPTQv2 格式的支持：分析与实现", sections "LLM 的权重量化",
"从 GPTQv1 到 GPTQv2", "调整细节：根据格式选择处理方式"):

  gemm(A, qweight, qzeros, scales, g_idx, bits, group, fmt)  -> C = A @ dequant(W)
  dequant(qweight, qzeros, scales, g_idx, K, bits, group, fmt, dtype) -> W [K, N]
  quantize_rtn(W, bits, group, g_idx, sym, fmt)              -> (qweight, qzeros, scales)
  repack_zeros_v1_to_v2(qzeros_v1, N, bits)                  (host memory)
  prepack_act_order(qweight, g_idx, K, N, bits, group)      (host memory) -> (qweight', perm)
  prepack_act_order_device(qweight, g_idx, K, N, bits, group) (device memory) -> (qweight', perm)
  gemm_perm(A, perm, qweight', qzeros, scales, bits, group) -> A[:, perm] @ dequant(W'), M <= 32
  prepack_interleave(qweight, K, N, bits)                    (host memory) -> qweight in the decode
                                                             kernel's interleaved layout
  gemm_interleaved(A, qweight_il, qzeros, scales, perm, N, bits, group) -> the decode GEMM on it
  gemm_grouped(A, offsets, qweight[E], qzeros[E], scales[E], bits, group, max_m)
                                                             -> rows of expert e times W_e
  device_status(stream)                                      -> GPTQ_DEV_* bits
"""
import ctypes
import os
import re

import numpy as np

HERE = os.path.dirname(os.path.abspath(__file__))
LIB_PATH = os.path.join(HERE, "_lib", "libgptq_gb300.so")
HEADER = os.path.join(os.path.dirname(HERE), "include", "gptq.h")

F16, BF16 = 0, 1
V1, V2 = 1, 2
DEV_TIMEOUT, DEV_GIDX_RANGE, DEV_SCALE_OVERFLOW, DEV_EXPERT_ROWS, DEV_GIDX_GROUPS = 0x1, 0x2, 0x4, 0x8, 0x10
DECODE_MAX_M = 32

_STATUS = {0: "GPTQ_OK", -1: "GPTQ_ERR_ARG", -2: "GPTQ_ERR_SHAPE", -3: "GPTQ_ERR_ALIGN",
           -4: "GPTQ_ERR_WORKSPACE", -5: "GPTQ_ERR_ZERO_OVERFLOW", -6: "GPTQ_ERR_CUDA",
           -7: "GPTQ_ERR_UNSUPPORTED", -8: "GPTQ_ERR_DEVICE"}


class GPTQError(RuntimeError):
    def __init__(self, code, what=""):
        self.code = code
        msg = "%s (%d)" % (_STATUS.get(code, "unknown"), code)
        try:
            msg = lib().gptq_strerror(code).decode()
        except Exception:
            pass
        super().__init__("%s%s" % (what + ": " if what else "", msg))


_lib = None

_P, _I, _SZ = ctypes.c_void_p, ctypes.c_int, ctypes.c_size_t
_SIGNATURES = {
    "gptq_dequant": (_I, [_P, _P, _P, _P, _I, _I, _I, _I, _I, _I, _P, _P]),
    "gptq_gemm": (_I, [_P, _I, _I, _I, _P, _P, _P, _P, _I, _I, _I, _I, _P, _P, _SZ, _P]),
    "gptq_gemm_host": (_I, [_P, _P, _I, _I, _I, _P, _P, _P, _P, _I, _I, _I, _I, _P, _P, _P, _SZ, _P]),
    "gptq_host_plan_create": (_I, [ctypes.POINTER(ctypes.c_void_p), _P, _P, _I, _I, _I, _P, _P, _P, _P, _I, _I, _I,
                                   _I, _P, _P, _P, _SZ, _P]),
    "gptq_host_plan_run": (_I, [_P]),
    "gptq_host_plan_destroy": (_I, [_P]),
    "gptq_gemm_workspace_size": (_SZ, [_I, _I, _I, _I, _I]),
    "gptq_gemm_act_order_workspace_size": (_SZ, [_I, _I, _I, _I, _I]),
    "gptq_repack_zeros_v1_to_v2": (_I, [_P, _P, _I, _I, _I]),
    "gptq_quantize_rtn": (_I, [_P, _I, _I, _I, _I, _P, _I, _I, _P, _P, _P, _P]),
    "gptq_get_device_status": (_I, [_P, ctypes.POINTER(ctypes.c_uint)]),
    "gptq_strerror": (ctypes.c_char_p, [_I]),
    "gptq_selftest_wait_timeout": (_I, [ctypes.c_ulonglong, _P, _P]),
    "gptq_prepack_act_order": (_I, [_P, _P, _I, _I, _I, _I, _P, _P]),
    "gptq_prepack_act_order_device": (_I, [_P, _P, _I, _I, _I, _I, _P, _P, _P, _SZ, _P]),
    "gptq_prepack_act_order_device_workspace_size": (_SZ, [_I, _I, _I]),
    "gptq_gemm_perm": (_I, [_P, _I, _I, _I, _P, _P, _P, _P, _I, _I, _I, _I, _P, _P, _SZ, _P]),
    "gptq_gemm_perm_workspace_size": (_SZ, [_I, _I]),
    "gptq_gemm_perm_noalloc": (_I, [_P, _I, _I, _I, _P, _P, _P, _P, _I, _I, _I, _I, _P, _P]),
    "gptq_gemm_grouped": (_I, [_P, _I, _I, _I, _P, _I, _I, _P, _P, _P, _I, _I, _I, _I, _P, _P]),
    "gptq_prepack_interleave": (_I, [_P, _I, _I, _I, _P]),
    "gptq_gemm_interleaved": (_I, [_P, _I, _I, _I, _P, _P, _P, _P, _I, _I, _I, _I, _P, _P, _SZ, _P]),
}


def lib():
    """The loaded C library (ctypes).  Raises if it has not been built."""
    global _lib
    if _lib is None:
        if not os.path.exists(LIB_PATH):
            raise RuntimeError("GPTQ CUDA library not built (%s): run "
                               "`python -c 'import __graft_entry__ as g; g.build()'`" % LIB_PATH)
        handle = ctypes.CDLL(LIB_PATH)
        for name, (res, args) in _SIGNATURES.items():
            fn = getattr(handle, name)
            fn.restype = res
            fn.argtypes = args
        _lib = handle
    return _lib


def header_functions():
    """Names of the functions include/gptq.h declares."""
    with open(HEADER) as f:
        text = f.read()
    return sorted(set(re.findall(r"^\s*(?:int|size_t|const char\s*\*)\s+(gptq_\w+)\s*\(", text, re.M)))


def selftest_wait_timeout(limit_ns=50_000_000, stream=None):
    """Run the bounded-wait self-test; returns (waited_out, status bits)."""
    torch = _torch()
    flag = torch.zeros(1, dtype=torch.int32, device="cuda")
    _check(lib().gptq_selftest_wait_timeout(int(limit_ns), _ptr(flag), _stream(stream)),
           "gptq_selftest_wait_timeout")
    status = device_status(stream)
    return int(flag.item()), status


def _check(rc, what):
    if rc != 0:
        raise GPTQError(rc, what)


def _torch():
    import torch
    return torch


def _dtype_code(t):
    torch = _torch()
    if t.dtype == torch.float16:
        return F16
    if t.dtype == torch.bfloat16:
        return BF16
    raise TypeError("activations must be float16 or bfloat16, got %s" % t.dtype)


def _ptr(t, dtype=None, name="tensor"):
    if t is None:
        return None
    if not t.is_cuda:
        raise ValueError("%s must be a CUDA tensor" % name)
    if not t.is_contiguous():
        raise ValueError("%s must be contiguous" % name)
    if dtype is not None and t.dtype != dtype:
        raise TypeError("%s must be %s, got %s" % (name, dtype, t.dtype))
    return ctypes.c_void_p(t.data_ptr())


def _stream(stream):
    torch = _torch()
    s = torch.cuda.current_stream() if stream is None else stream
    return ctypes.c_void_p(s.cuda_stream)


def gemm(A, qweight, qzeros, scales, g_idx=None, *, bits, group, fmt=V2, out=None, workspace=None,
         sort_rows=True, stream=None):
    """C[M, N] = A[M, K] @ dequant(qweight, qzeros, scales, g_idx) on the current stream.  When no
    workspace is given one is allocated here: act-order (g_idx) with sort_rows, where the shape
    qualifies, takes act_order_workspace_size(...) bytes (rows sorted by group on the device);
    otherwise bf16 activations take workspace_size(...) bytes."""
    torch = _torch()
    M, K = A.shape
    N = qweight.shape[1]
    if out is None:
        out = torch.empty((M, N), dtype=A.dtype, device=A.device)
    if workspace is None and M > 0:
        size = act_order_workspace_size(M, K, N, bits, group) if (g_idx is not None and sort_rows) else 0
        if size == 0 and A.dtype == torch.bfloat16:
            size = workspace_size(M, K, N, bits, group)
        if size:
            workspace = torch.empty(size, dtype=torch.uint8, device=A.device)
    ws_ptr = _ptr(workspace, name="workspace") if workspace is not None else None
    ws_len = workspace.numel() * workspace.element_size() if workspace is not None else 0
    rc = lib().gptq_gemm(_ptr(A, name="A"), M, K, _dtype_code(A),
                         _ptr(qweight, torch.int32, "qweight"), _ptr(qzeros, torch.int32, "qzeros"),
                         _ptr(scales, torch.float16, "scales"), _ptr(g_idx, torch.int32, "g_idx"),
                         N, bits, group, fmt, _ptr(out, A.dtype, "out"), ws_ptr, ws_len, _stream(stream))
    _check(rc, "gptq_gemm")
    return out


class HostGemm:
    """gptq_gemm_host prepared once, for a loop that reruns one problem on the same host and device
    buffers (only the contents of A_host change between calls): calling the object takes A_host
    [M, K] (a CPU tensor, page-locked for the direct path) into A_dev, computes C = A @ dequant(W)
    and returns C_host (a CPU tensor) once it holds the result.  On a named stream the call is
    captured into a CUDA graph (gptq_host_plan_create, which runs it once) and each call replays
    the graph; on the default stream each call is one gptq_gemm_host call with the arguments
    marshalled here.  The staging buffers and the workspace belong to the caller and must outlive
    the object (as for gemm, a bf16 prefill needs workspace_size(...) bytes)."""

    def __init__(self, A_host, A_dev, qweight, qzeros, scales, g_idx=None, *, bits, group, C_dev, C_host,
                 fmt=V2, workspace=None, stream=None):
        torch = _torch()
        M, K = A_host.shape
        N = qweight.shape[1]
        for t, name in ((A_host, "A_host"), (C_host, "C_host")):
            if t.is_cuda or not t.is_contiguous():
                raise ValueError("%s must be a contiguous CPU tensor" % name)
        if A_dev.dtype != A_host.dtype or C_dev.dtype != A_host.dtype or C_host.dtype != A_host.dtype:
            raise TypeError("A_host, A_dev, C_dev and C_host must share A's dtype")
        if A_dev.numel() < M * K or C_dev.numel() < M * N or C_host.numel() < M * N:
            raise ValueError("staging buffers smaller than the problem")
        ws_ptr = _ptr(workspace, name="workspace") if workspace is not None else None
        ws_len = workspace.numel() * workspace.element_size() if workspace is not None else 0
        # the tensors stay referenced for as long as the object can be called
        self._keep = (A_host, A_dev, qweight, qzeros, scales, g_idx, C_dev, C_host, workspace)
        self._args = (ctypes.c_void_p(A_host.data_ptr()), _ptr(A_dev, name="A_dev"), M, K, _dtype_code(A_host),
                      _ptr(qweight, torch.int32, "qweight"), _ptr(qzeros, torch.int32, "qzeros"),
                      _ptr(scales, torch.float16, "scales"), _ptr(g_idx, torch.int32, "g_idx"), N, bits, group,
                      fmt, _ptr(C_dev, name="C_dev"), ctypes.c_void_p(C_host.data_ptr()), ws_ptr, ws_len,
                      _stream(stream))
        self.C_host = C_host
        self._plan = None
        if self._args[-1].value:
            # a named stream: the call is captured once (gptq_host_plan_create, which also runs it
            # once) and each call replays the capture
            h = ctypes.c_void_p()
            _check(lib().gptq_host_plan_create(ctypes.byref(h), *self._args), "gptq_host_plan_create")
            self._plan = h
            self._run = lib().gptq_host_plan_run
        else:
            self._fn = lib().gptq_gemm_host

    def __call__(self):
        if self._plan is not None:
            _check(self._run(self._plan), "gptq_host_plan_run")
        else:
            _check(self._fn(*self._args), "gptq_gemm_host")
        return self.C_host

    def close(self):
        """Release the captured plan (also done when the object is collected)."""
        if getattr(self, "_plan", None) is not None and _lib is not None:
            lib().gptq_host_plan_destroy(self._plan)
        self._plan = None

    def __del__(self):
        try:
            self.close()
        except Exception:
            pass


def gemm_host(A_host, A_dev, qweight, qzeros, scales, g_idx=None, *, bits, group, C_dev, C_host, fmt=V2,
              workspace=None, stream=None):
    """One gptq_gemm_host call: returns C_host holding C = A @ dequant(W) (HostGemm prepares the
    call for a loop over the same buffers)."""
    torch = _torch()
    M, K = A_host.shape
    N = qweight.shape[1]
    for t, name in ((A_host, "A_host"), (C_host, "C_host")):
        if t.is_cuda or not t.is_contiguous():
            raise ValueError("%s must be a contiguous CPU tensor" % name)
    if A_dev.dtype != A_host.dtype or C_dev.dtype != A_host.dtype or C_host.dtype != A_host.dtype:
        raise TypeError("A_host, A_dev, C_dev and C_host must share A's dtype")
    if A_dev.numel() < M * K or C_dev.numel() < M * N or C_host.numel() < M * N:
        raise ValueError("staging buffers smaller than the problem")
    ws_ptr = _ptr(workspace, name="workspace") if workspace is not None else None
    ws_len = workspace.numel() * workspace.element_size() if workspace is not None else 0
    rc = lib().gptq_gemm_host(ctypes.c_void_p(A_host.data_ptr()), _ptr(A_dev, name="A_dev"), M, K,
                              _dtype_code(A_host), _ptr(qweight, torch.int32, "qweight"),
                              _ptr(qzeros, torch.int32, "qzeros"), _ptr(scales, torch.float16, "scales"),
                              _ptr(g_idx, torch.int32, "g_idx"), N, bits, group, fmt, _ptr(C_dev, name="C_dev"),
                              ctypes.c_void_p(C_host.data_ptr()), ws_ptr, ws_len, _stream(stream))
    _check(rc, "gptq_gemm_host")
    return C_host


def dequant(qweight, qzeros, scales, g_idx=None, *, K, bits, group, fmt=V2, dtype=None, out=None,
            stream=None):
    """W[K, N] = RN((q - zero) * scale) in `dtype` (float16 default)."""
    torch = _torch()
    dtype = torch.float16 if dtype is None else dtype
    N = qweight.shape[1]
    if out is None:
        out = torch.empty((K, N), dtype=dtype, device=qweight.device)
    code = F16 if dtype == torch.float16 else BF16
    rc = lib().gptq_dequant(_ptr(qweight, torch.int32, "qweight"), _ptr(qzeros, torch.int32, "qzeros"),
                            _ptr(scales, torch.float16, "scales"), _ptr(g_idx, torch.int32, "g_idx"),
                            K, N, bits, group, fmt, code, _ptr(out, dtype, "out"), _stream(stream))
    _check(rc, "gptq_dequant")
    return out


def quantize_rtn(W, *, bits, group, g_idx=None, sym=False, fmt=V2, out=None, stream=None):
    """Round-to-nearest checkpoint of fp32 weights W [K, N]: (qweight, qzeros, scales), written
    into `out` = (qweight, qzeros, scales) when given."""
    torch = _torch()
    K, N = W.shape
    G = 1 if group == -1 else K // group
    if out is not None:
        qweight, qzeros, scales = out
    else:
        qweight = torch.empty((K * bits // 32, N), dtype=torch.int32, device=W.device)
        qzeros = torch.empty((G, N * bits // 32), dtype=torch.int32, device=W.device)
        scales = torch.empty((G, N), dtype=torch.float16, device=W.device)
    if (tuple(qweight.shape) != (K * bits // 32, N) or tuple(qzeros.shape) != (G, N * bits // 32)
            or tuple(scales.shape) != (G, N)):
        raise ValueError("quantize_rtn: output buffers of the wrong shape")
    rc = lib().gptq_quantize_rtn(_ptr(W, torch.float32, "W"), K, N, bits, group,
                                 _ptr(g_idx, torch.int32, "g_idx"), int(bool(sym)), fmt,
                                 _ptr(qweight), _ptr(qzeros), _ptr(scales), _stream(stream))
    _check(rc, "gptq_quantize_rtn")
    return qweight, qzeros, scales


def repack_zeros_v1_to_v2(qzeros_v1, N, bits):
    """Host repack of v1 qzeros (numpy int32 [G, N*bits/32]) into a new v2 array."""
    src = np.ascontiguousarray(qzeros_v1, dtype=np.int32)
    out = np.empty_like(src)
    G = src.shape[0]
    rc = lib().gptq_repack_zeros_v1_to_v2(src.ctypes.data_as(_P), out.ctypes.data_as(_P), G, N, bits)
    _check(rc, "gptq_repack_zeros_v1_to_v2")
    return out


def prepack_act_order(qweight, g_idx, *, K, N, bits, group):
    """Host: sort an act-order checkpoint's rows by group.  qweight (numpy int32 [K*bits/32, N])
    and g_idx (numpy int32 [K]) -> (qweight_out, perm), with A @ W == A[:, perm] @ W_out."""
    qw = np.ascontiguousarray(qweight, dtype=np.int32)
    gi = np.ascontiguousarray(g_idx, dtype=np.int32)
    out = np.empty_like(qw)
    perm = np.empty(K, dtype=np.int32)
    rc = lib().gptq_prepack_act_order(qw.ctypes.data_as(_P), gi.ctypes.data_as(_P), K, N, bits, group,
                                      out.ctypes.data_as(_P), perm.ctypes.data_as(_P))
    _check(rc, "gptq_prepack_act_order")
    return out, perm


def prepack_act_order_device_workspace_size(K, bits, group):
    return int(lib().gptq_prepack_act_order_device_workspace_size(K, bits, group))


def prepack_act_order_device(qweight, g_idx, *, K, N, bits, group, workspace=None, stream=None):
    """Device: sort an act-order checkpoint's rows by group on `stream` (asynchronous).  qweight
    (int32 [K*bits/32, N]) and g_idx (int32 [K]) on the device -> (qweight_out, perm) on the
    device, bit-identical to prepack_act_order.  A g_idx whose groups are not all of `group` rows
    leaves both unwritten and sets DEV_GIDX_GROUPS in the device status word."""
    torch = _torch()
    ws_bytes = prepack_act_order_device_workspace_size(K, bits, group)
    if ws_bytes == 0:
        raise GPTQError(-2, "gptq_prepack_act_order_device")
    if workspace is None:
        workspace = torch.empty(ws_bytes, dtype=torch.uint8, device=qweight.device)
    out = torch.empty_like(qweight)
    perm = torch.empty(K, dtype=torch.int32, device=qweight.device)
    rc = lib().gptq_prepack_act_order_device(_ptr(qweight, torch.int32, "qweight"), _ptr(g_idx, torch.int32, "g_idx"),
                                             K, N, bits, group, _ptr(out, torch.int32, "qweight_out"),
                                             _ptr(perm, torch.int32, "perm"), _ptr(workspace, name="workspace"),
                                             workspace.numel() * workspace.element_size(), _stream(stream))
    _check(rc, "gptq_prepack_act_order_device")
    return out, perm


def gemm_perm_workspace_size(M, K):
    return int(lib().gptq_gemm_perm_workspace_size(M, K))


def gemm_perm(A, perm, qweight, qzeros, scales, *, bits, group, fmt=V2, out=None, workspace=None,
              stream=None):
    """C[M, N] = A[:, perm] @ dequant(prepacked qweight), M <= 32.  For M > 1 a workspace of
    gemm_perm_workspace_size(M, K) bytes is used (allocated here when not given)."""
    torch = _torch()
    M, K = A.shape
    N = qweight.shape[1]
    if out is None:
        out = torch.empty((M, N), dtype=A.dtype, device=A.device)
    ws_bytes = gemm_perm_workspace_size(M, K)
    if ws_bytes and workspace is None:
        workspace = torch.empty(ws_bytes, dtype=torch.uint8, device=A.device)
    ws_ptr = _ptr(workspace, name="workspace") if ws_bytes else None
    ws_len = workspace.numel() * workspace.element_size() if ws_bytes else 0
    rc = lib().gptq_gemm_perm(_ptr(A, name="A"), M, K, _dtype_code(A), _ptr(perm, torch.int32, "perm"),
                              _ptr(qweight, torch.int32, "qweight"), _ptr(qzeros, torch.int32, "qzeros"),
                              _ptr(scales, torch.float16, "scales"), N, bits, group, fmt,
                              _ptr(out, A.dtype, "out"), ws_ptr, ws_len, _stream(stream))
    _check(rc, "gptq_gemm_perm")
    return out


def prepack_interleave(qweight, *, K, N, bits):
    """Host: qweight (numpy int32 [K*bits/32, N]) in the decode kernel's interleaved layout."""
    qw = np.ascontiguousarray(qweight, dtype=np.int32)
    out = np.empty(qw.size, dtype=np.int32)
    rc = lib().gptq_prepack_interleave(qw.ctypes.data_as(_P), K, N, bits, out.ctypes.data_as(_P))
    _check(rc, "gptq_prepack_interleave")
    return out


def gemm_interleaved(A, qweight_il, qzeros, scales, perm=None, *, N, bits, group, fmt=V2, out=None,
                     workspace=None, stream=None):
    """C[M, N] = A @ dequant(W) (A[:, perm] @ ... with perm) for an interleaved qweight, M <= 32."""
    torch = _torch()
    M, K = A.shape
    if out is None:
        out = torch.empty((M, N), dtype=A.dtype, device=A.device)
    ws_bytes = gemm_perm_workspace_size(M, K) if perm is not None else 0
    if ws_bytes and workspace is None:
        workspace = torch.empty(ws_bytes, dtype=torch.uint8, device=A.device)
    ws_ptr = _ptr(workspace, name="workspace") if ws_bytes else None
    ws_len = workspace.numel() * workspace.element_size() if ws_bytes else 0
    rc = lib().gptq_gemm_interleaved(_ptr(A, name="A"), M, K, _dtype_code(A), _ptr(perm, torch.int32, "perm"),
                                     _ptr(qweight_il, torch.int32, "qweight_il"), _ptr(qzeros, torch.int32, "qzeros"),
                                     _ptr(scales, torch.float16, "scales"), N, bits, group, fmt,
                                     _ptr(out, A.dtype, "out"), ws_ptr, ws_len, _stream(stream))
    _check(rc, "gptq_gemm_interleaved")
    return out


def gemm_grouped(A, offsets, qweight, qzeros, scales, *, bits, group, max_m, fmt=V2, out=None,
                 stream=None):
    """Mixture-of-experts GEMM: rows [offsets[e], offsets[e+1]) of A [rows, K] times expert e's
    weight, into the same rows of C [rows, N].  qweight [E, K*bits/32, N], qzeros
    [E, G, N*bits/32], scales [E, G, N] fp16; offsets [E+1] int32 on the device; every expert
    has at most max_m (<= 32) rows."""
    torch = _torch()
    rows, K = A.shape
    E, _, N = qweight.shape
    if out is None:
        out = torch.empty((rows, N), dtype=A.dtype, device=A.device)
    rc = lib().gptq_gemm_grouped(_ptr(A, name="A"), rows, K, _dtype_code(A),
                                 _ptr(offsets, torch.int32, "offsets"), E, max_m,
                                 _ptr(qweight, torch.int32, "qweight"), _ptr(qzeros, torch.int32, "qzeros"),
                                 _ptr(scales, torch.float16, "scales"), N, bits, group, fmt,
                                 _ptr(out, A.dtype, "out"), _stream(stream))
    _check(rc, "gptq_gemm_grouped")
    return out


def workspace_size(M, K, N, bits, group):
    return int(lib().gptq_gemm_workspace_size(M, K, N, bits, group))


def act_order_workspace_size(M, K, N, bits, group):
    return int(lib().gptq_gemm_act_order_workspace_size(M, K, N, bits, group))


def device_status(stream=None):
    """Synchronize `stream`, read and clear the device status word (GPTQ_DEV_* bits)."""
    v = ctypes.c_uint(0)
    _check(lib().gptq_get_device_status(_stream(stream), ctypes.byref(v)), "gptq_get_device_status")
    return int(v.value)


def strerror(code):
    return lib().gptq_strerror(code).decode()
