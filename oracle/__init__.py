"""CPU oracle for LUT-simulated approximate multiplication (test infrastructure).

Only the tests, ``__graft_entry__.smoke()`` and the benchmark's CPU-baseline leg
may import this package.  The product library never does; the two share no
code.  The arithmetic lives in ``amsim_oracle.c`` (plain C, products summed in
double); this module compiles it with gcc, loads it with ctypes and adds the
attention reference (scaled QK^T, softmax in double, PV).

Page followed: "ApproxTrain: Fast Simulation of Approximate Multipliers for
DNN Training and Inference", Sec. V-A (Algorithm 1), Sec. V-B (Algorithm 2),
Sec. VI-B (Algorithms 3 and 4, Fig. 8); depthwise convolution from Sec. III's
Table I, written as the grouped case of those sums.

A multiplier is named by ``kind`` -- "exact", "mitchell", or a numpy array of
2^(2M) uint32 table entries (carry << 23 | mantissa, first operand's mantissa
in the high index bits), e.g. from ``lut_from_fn`` over a user's approx_mul --
plus ``M`` and the exponent width ``ebits`` (1..8, default 8 = fp32's) of the
simulated (1, e, M) format (Sec. V-B, last paragraph).

Parity unpinned: nothing.  Every function here has a pin in
``tests/test_oracle_*.py`` (see the module docstrings there).
"""
from __future__ import annotations

import ctypes
import os
import subprocess
import threading

import numpy as np

EXACT = 0
MITCHELL = 1
TABLE = 2
KINDS = {"exact": EXACT, "mitchell": MITCHELL}

_HERE = os.path.dirname(os.path.abspath(__file__))
_SRC = os.path.join(_HERE, "amsim_oracle.c")
_BUILD_DIR = os.path.join(_HERE, "_build")
_LIB_PATH = os.path.join(_BUILD_DIR, "libamsim_oracle.so")
_lock = threading.Lock()
_lib = None

USER_FN = ctypes.CFUNCTYPE(ctypes.c_float, ctypes.c_float, ctypes.c_float)


class _Mult(ctypes.Structure):
    """orc_mult: kind, M, exponent bits, table pointer."""
    _fields_ = [("kind", ctypes.c_int), ("M", ctypes.c_int), ("E", ctypes.c_int), ("table", ctypes.c_void_p)]


def build(force: bool = False) -> str:
    """Compile the oracle with gcc (no fast-math, no FMA contraction)."""
    os.makedirs(_BUILD_DIR, exist_ok=True)
    if (not force and os.path.exists(_LIB_PATH)
            and os.path.getmtime(_LIB_PATH) >= os.path.getmtime(_SRC)):
        return _LIB_PATH
    tmp = _LIB_PATH + f".tmp{os.getpid()}"
    cmd = ["gcc", "-O2", "-std=c11", "-fPIC", "-shared", "-pthread",
           "-ffp-contract=off", "-fno-fast-math", _SRC, "-o", tmp, "-lm"]
    subprocess.run(cmd, check=True)
    os.replace(tmp, _LIB_PATH)
    return _LIB_PATH


def lib():
    global _lib
    with _lock:
        if _lib is None:
            path = build()
            L = ctypes.CDLL(path)
            u32, i32, i64, f32, f64 = (ctypes.c_uint32, ctypes.c_int, ctypes.c_int64,
                                       ctypes.c_float, ctypes.c_double)
            vp = ctypes.c_void_p
            L.orc_approx_mul.argtypes = [i32, i32, f32, f32]
            L.orc_approx_mul.restype = f32
            L.orc_lut_entry.argtypes = [i32, i32, u32, u32, ctypes.POINTER(u32)]
            L.orc_lut_entry.restype = i32
            L.orc_lut.argtypes = [i32, i32, vp]
            L.orc_lut.restype = i32
            L.orc_amsim_bits.argtypes = [i32, i32, u32, u32]
            L.orc_amsim_bits.restype = u32
            L.orc_lut_from_fn.argtypes = [USER_FN, i32, vp]
            L.orc_lut_from_fn.restype = i32
            mp = ctypes.POINTER(_Mult)
            L.orc_amsim_mult_bits.argtypes = [mp, u32, u32]
            L.orc_amsim_mult_bits.restype = u32
            L.orc_mul.argtypes = [mp, vp, vp, vp, i64]
            L.orc_mul.restype = i32
            L.orc_gemm_rows.argtypes = [mp, i32, i32, i32, i32, i32, f64, vp, i64, vp, i64,
                                        f64, vp, i64, vp, i32, vp, vp, i32]
            L.orc_gemm_rows.restype = i32
            for name in ("orc_conv2d_fwd_points", "orc_conv2d_bwd_data_points",
                         "orc_conv2d_bwd_filter_points", "orc_dwconv2d_fwd_points",
                         "orc_dwconv2d_bwd_data_points", "orc_dwconv2d_bwd_filter_points"):
                fn = getattr(L, name)
                fn.argtypes = [mp, vp, vp, vp, vp, i64, vp, vp, i32]
                fn.restype = i32
            L.orc_conv2d_out_hw.argtypes = [vp, ctypes.POINTER(i32), ctypes.POINTER(i32)]
            L.orc_conv2d_out_hw.restype = i32
            _lib = L
    return _lib


def _kind(kind) -> int:
    return KINDS[kind] if isinstance(kind, str) else int(kind)


def mult(kind, M: int, ebits: int = 8):
    """The orc_mult for a closed-form kind or a table of entries (kept alive by
    the returned struct)."""
    if isinstance(kind, np.ndarray):
        table = np.ascontiguousarray(kind, dtype=np.uint32)
        if table.size != 1 << (2 * M):
            raise ValueError(f"a table for M={M} has {1 << (2 * M)} entries, not {table.size}")
        mu = _Mult(TABLE, M, ebits, table.ctypes.data)
        mu._table = table
        return mu
    return _Mult(_kind(kind), M, ebits, None)


def _f32(a) -> np.ndarray:
    return np.ascontiguousarray(a, dtype=np.float32)


def _ptr(a: np.ndarray):
    return ctypes.c_void_p(a.ctypes.data)


def default_threads() -> int:
    return os.cpu_count() or 1


# ---------------------------------------------------------------- scalar level
def approx_mul(kind, M: int, a: float, b: float) -> float:
    """The multiplier model approx_mul (normal operands, normal product)."""
    return float(lib().orc_approx_mul(_kind(kind), M, float(a), float(b)))


def lut_entry(kind, M: int, p: int, q: int) -> int:
    """Algorithm 1 for one mantissa pair: carry << 23 | mantissa."""
    out = ctypes.c_uint32(0)
    rc = lib().orc_lut_entry(_kind(kind), M, p, q, ctypes.byref(out))
    if rc:
        raise ValueError(f"orc_lut_entry rc={rc}")
    return int(out.value)


def lut(kind, M: int) -> np.ndarray:
    """All 2^(2M) u32 entries, first operand's mantissa in the high index bits."""
    out = np.zeros(1 << (2 * M), dtype=np.uint32)
    rc = lib().orc_lut(_kind(kind), M, _ptr(out))
    if rc:
        raise ValueError(f"orc_lut rc={rc}")
    return out


def lut_from_fn(approx_mul, M: int) -> np.ndarray:
    """Algorithm 1 over a user's approx_mul(A, B) -> C (a Python callable on
    fp32 values, called through a C function pointer): 2^(2M) u32 entries."""
    out = np.zeros(1 << (2 * M) if 1 <= M <= 11 else 1, dtype=np.uint32)
    cb = USER_FN(approx_mul)
    rc = lib().orc_lut_from_fn(cb, M, _ptr(out))
    if rc:
        raise ValueError(f"orc_lut_from_fn rc={rc}")
    return out


def amsim_bits(kind, M: int, a_bits: int, b_bits: int, ebits: int = 8) -> int:
    return int(lib().orc_amsim_mult_bits(ctypes.byref(mult(kind, M, ebits)), a_bits & 0xFFFFFFFF,
                                         b_bits & 0xFFFFFFFF))


def mul(kind, M: int, a, b, ebits: int = 8) -> np.ndarray:
    """Elementwise AMSim products (bit patterns exactly as Algorithm 2 gives)."""
    a = _f32(a)
    b = _f32(b)
    assert a.shape == b.shape
    c = np.empty_like(a)
    mu = mult(kind, M, ebits)
    if lib().orc_mul(ctypes.byref(mu), _ptr(a), _ptr(b), _ptr(c), a.size):
        raise ValueError("orc_mul: invalid multiplier")
    return c


# ---------------------------------------------------------------- contractions
def gemm(kind, M: int, A, B, *, transA=False, transB=False, alpha=1.0, beta=0.0, C0=None,
         rows=None, nthreads=None, ebits: int = 8):
    """Row-major C = alpha*op(A)op(B) + beta*C0 for the listed rows.

    Returns (out[nrows, n] float32, sumabs[nrows, n] float64) where sumabs is
    sum_k |product| (the scale the contraction tolerance is stated against).
    """
    A = _f32(A)
    B = _f32(B)
    m = A.shape[1] if transA else A.shape[0]
    k = A.shape[0] if transA else A.shape[1]
    n = B.shape[0] if transB else B.shape[1]
    kb = B.shape[1] if transB else B.shape[0]
    assert k == kb, (A.shape, B.shape, transA, transB)
    rows = np.arange(m, dtype=np.int32) if rows is None else np.ascontiguousarray(rows, dtype=np.int32)
    out = np.empty((rows.size, n), dtype=np.float32)
    sa = np.empty((rows.size, n), dtype=np.float64)
    if C0 is not None:
        C0 = _f32(C0)
        ldc = C0.shape[1]
        c0p = _ptr(C0)
    else:
        ldc, c0p = 0, None
        assert beta == 0.0
    mu = mult(kind, M, ebits)
    rc = lib().orc_gemm_rows(ctypes.byref(mu), int(transA), int(transB), m, n, k, float(alpha),
                             _ptr(A), A.shape[1], _ptr(B), B.shape[1], float(beta), c0p, ldc,
                             _ptr(rows), rows.size, _ptr(out), _ptr(sa),
                             nthreads or default_threads())
    if rc:
        raise ValueError(f"orc_gemm_rows rc={rc}")
    return out, sa


def conv_desc(N, H, W, C, K, R, S, stride=(1, 1), pad=(0, 0), dil=(1, 1)) -> np.ndarray:
    return np.array([N, H, W, C, K, R, S, stride[0], stride[1], pad[0], pad[1], dil[0], dil[1]],
                    dtype=np.int32)


def conv_out_hw(desc) -> tuple[int, int]:
    desc = np.ascontiguousarray(desc, dtype=np.int32)
    P = ctypes.c_int(0)
    Q = ctypes.c_int(0)
    if lib().orc_conv2d_out_hw(_ptr(desc), ctypes.byref(P), ctypes.byref(Q)):
        raise ValueError("bad conv descriptor")
    return P.value, Q.value


def _conv(fn_name, kind, M, desc, t0, t1, pts, nthreads, ebits=8):
    desc = np.ascontiguousarray(desc, dtype=np.int32)
    t0 = _f32(t0)
    t1 = _f32(t1)
    pts = np.ascontiguousarray(pts, dtype=np.int64)
    out = np.empty(pts.size, dtype=np.float32)
    sa = np.empty(pts.size, dtype=np.float64)
    mu = mult(kind, M, ebits)
    rc = getattr(lib(), fn_name)(ctypes.byref(mu), _ptr(desc), _ptr(t0), _ptr(t1), _ptr(pts), pts.size,
                                 _ptr(out), _ptr(sa), nthreads or default_threads())
    if rc:
        raise ValueError(f"{fn_name} rc={rc}")
    return out, sa


def conv2d_fwd(kind, M, desc, x, w, pts, nthreads=None, ebits=8):
    """Y (NPQK) at flat indices pts: sum over (r,s,c) of AMSim(x, w)."""
    return _conv("orc_conv2d_fwd_points", kind, M, desc, x, w, pts, nthreads, ebits)


def conv2d_bwd_data(kind, M, desc, dy, w, pts, nthreads=None, ebits=8):
    """dX (NHWC) at flat indices pts: sum over (r,s,k) of AMSim(dy, w)."""
    return _conv("orc_conv2d_bwd_data_points", kind, M, desc, dy, w, pts, nthreads, ebits)


def conv2d_bwd_filter(kind, M, desc, x, dy, pts, nthreads=None, ebits=8):
    """dW (RSCK) at flat indices pts: sum over (n,p,q) of AMSim(x, dy)."""
    return _conv("orc_conv2d_bwd_filter_points", kind, M, desc, x, dy, pts, nthreads, ebits)


def dwconv2d_fwd(kind, M, desc, x, w, pts, nthreads=None, ebits=8):
    """Depthwise Y (NPQK, K = C*D) at flat indices pts: sum over (r,s) of
    AMSim(x[..., c], w[r,s,c,d]) for output channel k = c*D + d; w is RSCD."""
    return _conv("orc_dwconv2d_fwd_points", kind, M, desc, x, w, pts, nthreads, ebits)


def dwconv2d_bwd_data(kind, M, desc, dy, w, pts, nthreads=None, ebits=8):
    """Depthwise dX (NHWC) at flat indices pts: sum over (r,s,d) of AMSim(dy, w)."""
    return _conv("orc_dwconv2d_bwd_data_points", kind, M, desc, dy, w, pts, nthreads, ebits)


def dwconv2d_bwd_filter(kind, M, desc, x, dy, pts, nthreads=None, ebits=8):
    """Depthwise dW (RSCD) at flat indices pts: sum over (n,p,q) of AMSim(x, dy)."""
    return _conv("orc_dwconv2d_bwd_filter_points", kind, M, desc, x, dy, pts, nthreads, ebits)


# ---------------------------------------------------------------- attention
def softmax_rows(S) -> np.ndarray:
    """Row softmax computed in double (exact reference), returned in double."""
    S = np.asarray(S, dtype=np.float64)
    z = S - S.max(axis=-1, keepdims=True)
    e = np.exp(z)
    return e / e.sum(axis=-1, keepdims=True)


def softmax_rows_backward(P, dP) -> np.ndarray:
    """Gradient of the row softmax: dS = P * (dP - sum_c P dP) per row (the
    softmax Jacobian diag(P) - P P^T applied to dP), in double."""
    P = np.asarray(P, dtype=np.float64)
    dP = np.asarray(dP, dtype=np.float64)
    return P * (dP - (P * dP).sum(axis=-1, keepdims=True))


def attention_scores(kind, M, Q, K, scale, rows=None, nthreads=None, ebits=8):
    """S = scale * Q K^T for one (batch, head) slice, AMSim products (q, k)."""
    return gemm(kind, M, Q, K, transB=True, alpha=scale, rows=rows, nthreads=nthreads, ebits=ebits)


def attention_output(kind, M, P, V, rows=None, nthreads=None, ebits=8):
    """O = P V for one (batch, head) slice, AMSim products (p, v)."""
    return gemm(kind, M, P, V, rows=rows, nthreads=nthreads, ebits=ebits)
