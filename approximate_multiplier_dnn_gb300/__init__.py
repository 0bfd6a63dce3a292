"""Python binding of libamsim (LUT-simulated approximate multipliers on GB300).

Argument marshalling only: every function forwards to the C ABI declared in
``include/amsim.h`` with the same name.  Device buffers are torch CUDA tensors
(or raw integer device pointers); the stream defaults to torch's current
stream.  All arithmetic runs in the library's CUDA kernels; there is no CPU
fallback -- importing works without a GPU, but calls fail loudly when the
library is not built or no GPU is present.
"""
from __future__ import annotations

import ctypes
import os
import re

HERE = os.path.dirname(os.path.abspath(__file__))
ROOT = os.path.dirname(HERE)
HEADER = os.path.join(ROOT, "include", "amsim.h")
LIB_PATH = os.path.join(HERE, "_build", "libamsim.so")

AMSIM_EXACT = 0
AMSIM_MITCHELL = 1
KINDS = {"exact": AMSIM_EXACT, "mitchell": AMSIM_MITCHELL}

AMSIM_OK = 0
AMSIM_EINVAL = 1
AMSIM_EUNSUPPORTED = 2
AMSIM_ENOMEM = 3
AMSIM_ECUDA = 4
AMSIM_ETIMEOUT = 5
AMSIM_WAIT_COPY = 1
AMSIM_WAIT_PARTIAL = 2
AMSIM_WAIT_PHASE = 4

_lib = None


class AmsimError(RuntimeError):
    def __init__(self, fn: str, status: int):
        self.status = status
        super().__init__(f"{fn} failed: {status} ({status_string(status)})")


class ConvDesc(ctypes.Structure):
    _fields_ = [(n, ctypes.c_int) for n in
                ("N", "H", "W", "C", "K", "R", "S", "stride_h", "stride_w", "pad_h", "pad_w", "dil_h", "dil_w")]

    @classmethod
    def make(cls, N, H, W, C, K, R, S, stride=(1, 1), pad=(0, 0), dil=(1, 1)):
        return cls(N, H, W, C, K, R, S, stride[0], stride[1], pad[0], pad[1], dil[0], dil[1])


APPROX_MUL_FN = ctypes.CFUNCTYPE(ctypes.c_float, ctypes.c_float, ctypes.c_float)


class GemmProblem(ctypes.Structure):
    """amsim_gemm_problem: one GEMM of a grouped launch."""
    _fields_ = [("A", ctypes.c_void_p), ("B", ctypes.c_void_p), ("C", ctypes.c_void_p),
                ("strideA", ctypes.c_int64), ("strideB", ctypes.c_int64), ("strideC", ctypes.c_int64),
                ("m", ctypes.c_int), ("n", ctypes.c_int), ("k", ctypes.c_int), ("lda", ctypes.c_int),
                ("ldb", ctypes.c_int), ("ldc", ctypes.c_int), ("batch", ctypes.c_int),
                ("alpha", ctypes.c_float), ("beta", ctypes.c_float),
                ("transA", ctypes.c_char), ("transB", ctypes.c_char)]

    @classmethod
    def make(cls, transA, transB, m, n, k, alpha, A, lda, B, ldb, beta, C, ldc, strideA=0, strideB=0, strideC=0,
             batch=1):
        return cls(_ptr(A), _ptr(B), _ptr(C), strideA, strideB, strideC, m, n, k, lda, ldb, ldc, batch,
                   float(alpha), float(beta), transA.encode(), transB.encode())


def build():
    from . import build_ext
    return build_ext.build()


def lib():
    """Load libamsim.so (raises if it has not been built)."""
    global _lib
    if _lib is not None:
        return _lib
    if not os.path.exists(LIB_PATH):
        raise ImportError(f"libamsim.so is not built ({LIB_PATH}); run __graft_entry__.build()")
    L = ctypes.CDLL(LIB_PATH)
    vp, i32, i64, f32, sz, ch = (ctypes.c_void_p, ctypes.c_int, ctypes.c_int64, ctypes.c_float,
                                 ctypes.c_size_t, ctypes.c_char)
    sig = {
        "amsim_status_string": ([i32], ctypes.c_char_p),
        "amsim_kernel_launches": ([], ctypes.c_ulonglong),
        "amsim_last_path": ([], i32),
        "amsim_device_errors": ([ctypes.POINTER(ctypes.c_uint), i32], i32),
        "amsim_set_flag_wait_limit": ([ctypes.c_longlong], i32),
        "amsim_set_cooperative_launches": ([i32], i32),
        "amsim_lut_generate": ([i32, i32, vp], i32),
        "amsim_lut_generate_from_fn": ([APPROX_MUL_FN, i32, vp], i32),
        "amsim_lut_build": ([i32, i32, ctypes.POINTER(vp)], i32),
        "amsim_lut_build_from_entries": ([vp, i32, ctypes.POINTER(vp)], i32),
        "amsim_lut_build_from_fn": ([APPROX_MUL_FN, i32, ctypes.POINTER(vp)], i32),
        "amsim_lut_entries": ([vp, vp], i32),
        "amsim_lut_info": ([vp, ctypes.POINTER(i32), ctypes.POINTER(i32), ctypes.POINTER(i32)], i32),
        "amsim_lut_set_closed_form": ([vp, i32], i32),
        "amsim_lut_set_exponent_bits": ([vp, i32], i32),
        "amsim_lut_destroy": ([vp], None),
        "amsim_mul": ([vp, vp, vp, i64, vp, vp], i32),
        "amsim_gemm": ([ch, ch, i32, i32, i32, f32, vp, i32, vp, i32, f32, vp, i32, vp, vp, sz, vp], i32),
        "amsim_gemm_strided_batched": ([ch, ch, i32, i32, i32, f32, vp, i32, i64, vp, i32, i64, f32, vp, i32,
                                        i64, i32, vp, vp, sz, vp], i32),
        "amsim_gemm_workspace_size": ([ch, ch, i32, i32, i32, i32, vp], sz),
        "amsim_gemm_grouped": ([i32, ctypes.POINTER(GemmProblem), vp, vp, sz, vp], i32),
        "amsim_gemm_noalloc": ([ch, ch, i32, i32, i32, f32, vp, i32, vp, i32, f32, vp, i32, vp, vp], i32),
        "amsim_gemm_grouped_workspace_size": ([i32, ctypes.POINTER(GemmProblem), vp], sz),
        "amsim_gemm_phased": ([i32, ctypes.POINTER(GemmProblem), i32, ctypes.POINTER(i32), ctypes.POINTER(i32), vp,
                               vp, sz, vp], i32),
        "amsim_gemm_phased_workspace_size": ([i32, ctypes.POINTER(GemmProblem), i32, ctypes.POINTER(i32),
                                              ctypes.POINTER(i32), vp], sz),
        "amsim_conv2d_out_hw": ([ctypes.POINTER(ConvDesc), ctypes.POINTER(i32), ctypes.POINTER(i32)], i32),
        "amsim_conv2d_fwd": ([ctypes.POINTER(ConvDesc), vp, vp, vp, vp, vp, sz, vp], i32),
        "amsim_conv2d_bwd_data": ([ctypes.POINTER(ConvDesc), vp, vp, vp, vp, vp, sz, vp], i32),
        "amsim_conv2d_bwd_filter": ([ctypes.POINTER(ConvDesc), vp, vp, vp, vp, vp, sz, vp], i32),
        "amsim_conv2d_workspace_size": ([ctypes.POINTER(ConvDesc), i32, vp], sz),
        "amsim_dwconv2d_fwd": ([ctypes.POINTER(ConvDesc), vp, vp, vp, vp, vp, sz, vp], i32),
        "amsim_dwconv2d_bwd_data": ([ctypes.POINTER(ConvDesc), vp, vp, vp, vp, vp, sz, vp], i32),
        "amsim_dwconv2d_bwd_filter": ([ctypes.POINTER(ConvDesc), vp, vp, vp, vp, vp, sz, vp], i32),
        "amsim_dwconv2d_workspace_size": ([ctypes.POINTER(ConvDesc), i32, vp], sz),
        "amsim_softmax_rows": ([vp, vp, i64, i32, vp], i32),
        "amsim_softmax_rows_backward": ([vp, vp, vp, i64, i32, vp], i32),
    }
    for name, (args, res) in sig.items():
        fn = getattr(L, name)
        fn.argtypes = args
        fn.restype = res
    _lib = L
    return _lib


def header_functions() -> list[str]:
    """Names of the functions that include/amsim.h declares."""
    with open(HEADER) as f:
        text = f.read()
    text = re.sub(r"/\*.*?\*/", "", text, flags=re.S)
    names = re.findall(r"\b(amsim_[a-z0-9_]+)\s*\(", text)
    return sorted(set(names))


AMSIM_PATH_PLANES = 1
AMSIM_PATH_INKERNEL_DECODE = 4
AMSIM_PATH_SINGLE_ROLE = 8
AMSIM_PATH_STREAMK = 16
AMSIM_PATH_FIXUP = 32
AMSIM_PATH_CONV_BOXES = 64
AMSIM_PATH_RAW_TILES = 128
AMSIM_PATH_PHASED = 256
AMSIM_PATH_CLOSED_FORM = 512
AMSIM_PATH_DW_TILES = 1024
AMSIM_PATH_DW_DIRECT = 2048
AMSIM_PATH_WIDE_TILES = 4096


def amsim_last_path() -> int:
    """Kernel-path bits (AMSIM_PATH_*) of this thread's most recent GEMM or convolution call."""
    return int(lib().amsim_last_path())


def amsim_kernel_launches() -> int:
    """Kernels the library has enqueued so far in this process."""
    return int(lib().amsim_kernel_launches())


def amsim_device_errors(clear: bool = True) -> tuple[int, int]:
    """(status, AMSIM_WAIT_* bits) of the device-side waits that gave up on the
    current device since the last clear (synchronises the device)."""
    bits = ctypes.c_uint(0)
    rc = lib().amsim_device_errors(ctypes.byref(bits), 1 if clear else 0)
    if rc not in (AMSIM_OK, AMSIM_ETIMEOUT):
        raise AmsimError("amsim_device_errors", rc)
    return rc, int(bits.value)


def amsim_set_flag_wait_limit(ns: int) -> None:
    _check("amsim_set_flag_wait_limit", lib().amsim_set_flag_wait_limit(int(ns)))


def amsim_set_cooperative_launches(on: bool) -> None:
    _check("amsim_set_cooperative_launches", lib().amsim_set_cooperative_launches(1 if on else 0))


def status_string(status: int) -> str:
    return lib().amsim_status_string(int(status)).decode()


def _check(fn: str, rc: int):
    if rc != AMSIM_OK:
        raise AmsimError(fn, rc)


def _ptr(t) -> int | None:
    if t is None:
        return None
    if isinstance(t, int):
        return t
    if hasattr(t, "data_ptr"):
        return t.data_ptr()
    if hasattr(t, "ctypes"):
        return t.ctypes.data
    raise TypeError(f"cannot take a pointer of {type(t)}")


def _stream(stream) -> int | None:
    if stream is None:
        import torch
        return torch.cuda.current_stream().cuda_stream
    if isinstance(stream, int):
        return stream
    return stream.cuda_stream


def _nbytes(t) -> int:
    if t is None:
        return 0
    return t.numel() * t.element_size()


def _kind(kind) -> int:
    return KINDS[kind] if isinstance(kind, str) else int(kind)


# ------------------------------------------------------------------ LUT
class Lut:
    """Owner of an amsim_lut_t handle (device LUT on the current device)."""

    def __init__(self, handle: int, M: int):
        self.handle = handle
        self.M = M

    @classmethod
    def build(cls, kind, M: int) -> "Lut":
        return cls(amsim_lut_build(kind, M), M)

    @classmethod
    def from_entries(cls, entries, M: int) -> "Lut":
        return cls(amsim_lut_build_from_entries(entries, M), M)

    @classmethod
    def from_fn(cls, approx_mul, M: int) -> "Lut":
        return cls(amsim_lut_build_from_fn(approx_mul, M), M)

    def info(self):
        return amsim_lut_info(self.handle)

    def entries(self):
        return amsim_lut_entries(self.handle, self.M)

    def set_closed_form(self, on: bool = True) -> "Lut":
        amsim_lut_set_closed_form(self.handle, on)
        return self

    def set_exponent_bits(self, E: int) -> "Lut":
        amsim_lut_set_exponent_bits(self.handle, E)
        return self

    def close(self):
        if self.handle:
            lib().amsim_lut_destroy(self.handle)
            self.handle = None

    def __del__(self):
        try:
            self.close()
        except Exception:
            pass


def _h(lut) -> int:
    return lut.handle if isinstance(lut, Lut) else lut


def amsim_lut_generate(kind, M: int):
    import numpy as np
    out = np.zeros(1 << (2 * M) if 1 <= M <= 11 else 1, dtype=np.uint32)
    _check("amsim_lut_generate", lib().amsim_lut_generate(_kind(kind), M, out.ctypes.data))
    return out


def amsim_lut_generate_from_fn(approx_mul, M: int):
    import numpy as np
    out = np.zeros(1 << (2 * M) if 1 <= M <= 11 else 1, dtype=np.uint32)
    cb = APPROX_MUL_FN(approx_mul)
    _check("amsim_lut_generate_from_fn", lib().amsim_lut_generate_from_fn(cb, M, out.ctypes.data))
    return out


def amsim_lut_build(kind, M: int) -> int:
    h = ctypes.c_void_p(0)
    _check("amsim_lut_build", lib().amsim_lut_build(_kind(kind), M, ctypes.byref(h)))
    return h.value


def amsim_lut_build_from_entries(entries, M: int) -> int:
    import numpy as np
    e = np.ascontiguousarray(entries, dtype=np.uint32)
    h = ctypes.c_void_p(0)
    _check("amsim_lut_build_from_entries", lib().amsim_lut_build_from_entries(e.ctypes.data, M, ctypes.byref(h)))
    return h.value


def amsim_lut_build_from_fn(approx_mul, M: int) -> int:
    """approx_mul: a Python callable (float, float) -> float, called through a C
    function pointer during the call."""
    cb = APPROX_MUL_FN(approx_mul)
    h = ctypes.c_void_p(0)
    _check("amsim_lut_build_from_fn", lib().amsim_lut_build_from_fn(cb, M, ctypes.byref(h)))
    return h.value


def amsim_lut_entries(lut, M: int):
    import numpy as np
    out = np.zeros(1 << (2 * M), dtype=np.uint32)
    _check("amsim_lut_entries", lib().amsim_lut_entries(_h(lut), out.ctypes.data))
    return out


def amsim_lut_set_closed_form(lut, on: bool = True) -> None:
    _check("amsim_lut_set_closed_form", lib().amsim_lut_set_closed_form(_h(lut), 1 if on else 0))


def amsim_lut_set_exponent_bits(lut, E: int) -> None:
    """Exponent width E (1..8) of the simulated (1, E, M) multiplier."""
    _check("amsim_lut_set_exponent_bits", lib().amsim_lut_set_exponent_bits(_h(lut), int(E)))


def amsim_lut_info(lut):
    M, w, s = ctypes.c_int(0), ctypes.c_int(0), ctypes.c_int(0)
    _check("amsim_lut_info", lib().amsim_lut_info(_h(lut), ctypes.byref(M), ctypes.byref(w), ctypes.byref(s)))
    return {"M": M.value, "width_bits": w.value, "shift": s.value}


def amsim_lut_destroy(lut):
    if isinstance(lut, Lut):
        lut.close()
    else:
        lib().amsim_lut_destroy(lut)


# ------------------------------------------------------------------ compute calls
def amsim_mul(a, b, c, n: int, lut, stream=None):
    _check("amsim_mul", lib().amsim_mul(_ptr(a), _ptr(b), _ptr(c), int(n), _h(lut), _stream(stream)))


def amsim_gemm(transA, transB, m, n, k, alpha, A, lda, B, ldb, beta, C, ldc, lut, ws=None, ws_bytes=None,
               stream=None):
    ws_bytes = _nbytes(ws) if ws_bytes is None else ws_bytes
    _check("amsim_gemm", lib().amsim_gemm(transA.encode(), transB.encode(), m, n, k, float(alpha), _ptr(A), lda,
                                          _ptr(B), ldb, float(beta), _ptr(C), ldc, _h(lut), _ptr(ws), ws_bytes,
                                          _stream(stream)))


def amsim_gemm_strided_batched(transA, transB, m, n, k, alpha, A, lda, strideA, B, ldb, strideB, beta, C, ldc,
                               strideC, batch, lut, ws=None, ws_bytes=None, stream=None):
    ws_bytes = _nbytes(ws) if ws_bytes is None else ws_bytes
    _check("amsim_gemm_strided_batched",
           lib().amsim_gemm_strided_batched(transA.encode(), transB.encode(), m, n, k, float(alpha), _ptr(A), lda,
                                            strideA, _ptr(B), ldb, strideB, float(beta), _ptr(C), ldc, strideC,
                                            batch, _h(lut), _ptr(ws), ws_bytes, _stream(stream)))


def amsim_gemm_noalloc(transA, transB, m, n, k, alpha, A, lda, B, ldb, beta, C, ldc, lut, stream=None):
    """amsim_gemm with its scratch inside the library (no workspace, no allocation)."""
    _check("amsim_gemm_noalloc", lib().amsim_gemm_noalloc(transA.encode(), transB.encode(), m, n, k, float(alpha),
                                                          _ptr(A), lda, _ptr(B), ldb, float(beta), _ptr(C), ldc,
                                                          _h(lut), _stream(stream)))


def amsim_gemm_workspace_size(transA, transB, m, n, k, batch, lut) -> int:
    return int(lib().amsim_gemm_workspace_size(transA.encode(), transB.encode(), m, n, k, batch, _h(lut)))


def _problem_array(problems):
    if isinstance(problems, ctypes.Array):
        return problems
    arr = (GemmProblem * len(problems))()
    for i, p in enumerate(problems):
        arr[i] = p
    return arr


def amsim_gemm_grouped(problems, lut, ws=None, ws_bytes=None, stream=None):
    """problems: a sequence of GemmProblem (or a ctypes array of them)."""
    arr = _problem_array(problems)
    ws_bytes = _nbytes(ws) if ws_bytes is None else ws_bytes
    _check("amsim_gemm_grouped", lib().amsim_gemm_grouped(len(arr), arr, _h(lut), _ptr(ws), ws_bytes,
                                                          _stream(stream)))


def _phase_arrays(phase_first, phase_after):
    n = len(phase_first)
    if len(phase_after) != n:
        raise ValueError("phase_first and phase_after differ in length")
    return n, (ctypes.c_int32 * n)(*phase_first), (ctypes.c_int32 * n)(*phase_after)


def amsim_gemm_phased(problems, phase_first, phase_after, lut, ws=None, ws_bytes=None, stream=None):
    """Ordered phases of GEMMs (sequences of GemmProblem): phase ph is
    problems[phase_first[ph]:phase_first[ph + 1]] and reads outputs of phases
    before phase_after[ph] only."""
    arr = _problem_array(problems)
    nph, first, after = _phase_arrays(phase_first, phase_after)
    ws_bytes = _nbytes(ws) if ws_bytes is None else ws_bytes
    _check("amsim_gemm_phased", lib().amsim_gemm_phased(len(arr), arr, nph, first, after, _h(lut), _ptr(ws),
                                                        ws_bytes, _stream(stream)))


def amsim_gemm_phased_workspace_size(problems, phase_first, phase_after, lut) -> int:
    arr = _problem_array(problems)
    nph, first, after = _phase_arrays(phase_first, phase_after)
    return int(lib().amsim_gemm_phased_workspace_size(len(arr), arr, nph, first, after, _h(lut)))


def amsim_gemm_grouped_workspace_size(problems, lut) -> int:
    arr = _problem_array(problems)
    return int(lib().amsim_gemm_grouped_workspace_size(len(arr), arr, _h(lut)))


def amsim_conv2d_out_hw(desc: ConvDesc):
    P, Q = ctypes.c_int(0), ctypes.c_int(0)
    _check("amsim_conv2d_out_hw", lib().amsim_conv2d_out_hw(ctypes.byref(desc), ctypes.byref(P), ctypes.byref(Q)))
    return P.value, Q.value


def _conv(name, desc, t0, t1, out, lut, ws, ws_bytes, stream):
    ws_bytes = _nbytes(ws) if ws_bytes is None else ws_bytes
    _check(name, getattr(lib(), name)(ctypes.byref(desc), _ptr(t0), _ptr(t1), _ptr(out), _h(lut), _ptr(ws),
                                      ws_bytes, _stream(stream)))


def amsim_conv2d_fwd(desc, x, w, y, lut, ws=None, ws_bytes=None, stream=None):
    _conv("amsim_conv2d_fwd", desc, x, w, y, lut, ws, ws_bytes, stream)


def amsim_conv2d_bwd_data(desc, dy, w, dx, lut, ws=None, ws_bytes=None, stream=None):
    _conv("amsim_conv2d_bwd_data", desc, dy, w, dx, lut, ws, ws_bytes, stream)


def amsim_conv2d_bwd_filter(desc, x, dy, dw, lut, ws=None, ws_bytes=None, stream=None):
    _conv("amsim_conv2d_bwd_filter", desc, x, dy, dw, lut, ws, ws_bytes, stream)


def amsim_conv2d_workspace_size(desc, which: int, lut) -> int:
    return int(lib().amsim_conv2d_workspace_size(ctypes.byref(desc), int(which), _h(lut)))


def amsim_dwconv2d_fwd(desc, x, w, y, lut, ws=None, ws_bytes=None, stream=None):
    """Depthwise forward; desc.K = C * D, w is R x S x C x D."""
    _conv("amsim_dwconv2d_fwd", desc, x, w, y, lut, ws, ws_bytes, stream)


def amsim_dwconv2d_bwd_data(desc, dy, w, dx, lut, ws=None, ws_bytes=None, stream=None):
    _conv("amsim_dwconv2d_bwd_data", desc, dy, w, dx, lut, ws, ws_bytes, stream)


def amsim_dwconv2d_bwd_filter(desc, x, dy, dw, lut, ws=None, ws_bytes=None, stream=None):
    _conv("amsim_dwconv2d_bwd_filter", desc, x, dy, dw, lut, ws, ws_bytes, stream)


def amsim_dwconv2d_workspace_size(desc, which: int, lut) -> int:
    return int(lib().amsim_dwconv2d_workspace_size(ctypes.byref(desc), int(which), _h(lut)))


def amsim_softmax_rows_backward(P, dP, dS, rows, cols, stream=None):
    _check("amsim_softmax_rows_backward",
           lib().amsim_softmax_rows_backward(_ptr(P), _ptr(dP), _ptr(dS), int(rows), int(cols), _stream(stream)))


def amsim_softmax_rows(S, P, rows, cols, stream=None):
    _check("amsim_softmax_rows", lib().amsim_softmax_rows(_ptr(S), _ptr(P), int(rows), int(cols),
                                                          _stream(stream)))


# ------------------------------------------------------------------ conveniences (still marshalling only)
def workspace(nbytes: int, device=None):
    """A caller-owned scratch buffer (uint8 torch tensor, 256-byte aligned by the caching allocator)."""
    import torch
    return torch.empty(max(int(nbytes), 1), dtype=torch.uint8, device=device or "cuda")


def gemm(A, B, lut, *, transA=False, transB=False, alpha=1.0, beta=0.0, C=None, ws=None, stream=None):
    """C = alpha op(A) op(B) + beta C for contiguous row-major fp32 CUDA tensors."""
    import torch
    m = A.shape[1] if transA else A.shape[0]
    k = A.shape[0] if transA else A.shape[1]
    n = B.shape[0] if transB else B.shape[1]
    if C is None:
        C = torch.empty((m, n), dtype=torch.float32, device=A.device)
    if ws is None:
        ws = workspace(amsim_gemm_workspace_size("T" if transA else "N", "T" if transB else "N", m, n, k, 1, lut),
                       A.device)
    amsim_gemm("T" if transA else "N", "T" if transB else "N", m, n, k, alpha, A, max(1, A.shape[1]), B,
               max(1, B.shape[1]), beta, C, max(1, n), lut, ws=ws, stream=stream)
    return C
