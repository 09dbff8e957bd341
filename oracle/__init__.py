"""Python access to the CPU oracle (``oracle/bsgemv_oracle.c``) for the block-scaled GEMV.

TEST INFRASTRUCTURE ONLY.  The oracle is the plain binary64 definition of

    y[M, N] = A[M, K] . deq(W)[N, K]^T

that the CUDA library is checked against.  Only the test suite, ``__graft_entry__.smoke()`` and
``bench.py``'s CPU-baseline / reference arm may import this module.  It shares nothing with the
CUDA library: it is plain C compiled with gcc into ``oracle/_build/liboracle.so`` and loaded with
ctypes.  It never imports ``block_scaled_bit_gb300``.

Formats are named by strings ("int4", "int8", "fp8", "nvfp4"); activations by "f16" / "bf16".
A "case" is any object with the attributes ``fmt, act, block_size, has_zp, N, K, M, A, W,
scales, zp, gscale`` holding numpy arrays (the seeded generators produce such objects), and
optionally ``bias`` (uint16 [N] activation-dtype bits, or None).
"""
from __future__ import annotations

import ctypes
import hashlib
import os
import subprocess
import threading

import numpy as np

_HERE = os.path.dirname(os.path.abspath(__file__))
_SRC = os.path.join(_HERE, "bsgemv_oracle.c")
_BUILD_DIR = os.path.join(_HERE, "_build")
_LOCK = threading.Lock()
_LIB = None

FORMAT_IDS = {"int4": 1, "int8": 2, "fp8": 3, "nvfp4": 4}

# minifloat parameters: (exponent bits, mantissa bits, bias, special-value convention)
SPECIAL_NONE, SPECIAL_FN, SPECIAL_IEEE = 0, 1, 2
F16 = (5, 10, 15, SPECIAL_IEEE)
BF16 = (8, 7, 127, SPECIAL_IEEE)
E4M3 = (4, 3, 7, SPECIAL_FN)
E2M1 = (2, 1, 1, SPECIAL_NONE)


def _lib_path() -> str:
    with open(_SRC, "rb") as f:
        digest = hashlib.sha1(f.read()).hexdigest()[:12]
    return os.path.join(_BUILD_DIR, f"liboracle_{digest}.so")


def build(verbose: bool = False) -> str:
    """Compile the oracle with gcc (OpenMP if available).  Returns the shared-library path."""
    path = _lib_path()
    if os.path.exists(path):
        return path
    os.makedirs(_BUILD_DIR, exist_ok=True)
    tmp = path + f".tmp{os.getpid()}"
    base = ["gcc", "-O2", "-std=c11", "-shared", "-fPIC", _SRC, "-o", tmp, "-lm"]
    try:
        subprocess.run(base[:1] + ["-fopenmp"] + base[1:], check=True, capture_output=not verbose)
    except subprocess.CalledProcessError:
        subprocess.run(base, check=True, capture_output=not verbose)  # no OpenMP on this host
    os.replace(tmp, path)
    return path


def lib() -> ctypes.CDLL:
    global _LIB
    with _LOCK:
        if _LIB is None:
            L = ctypes.CDLL(build())
            c_dbl_p = ctypes.POINTER(ctypes.c_double)
            L.orc_minifloat_value.restype = ctypes.c_double
            L.orc_minifloat_value.argtypes = [ctypes.c_uint32] + [ctypes.c_int] * 4
            L.orc_round_minifloat.restype = ctypes.c_uint32
            L.orc_round_minifloat.argtypes = [ctypes.c_double] + [ctypes.c_int] * 4
            L.orc_decode_array.restype = None
            L.orc_decode_array.argtypes = [ctypes.c_void_p, c_dbl_p, ctypes.c_long] + [ctypes.c_int] * 4
            L.orc_round_array.restype = None
            L.orc_round_array.argtypes = [c_dbl_p, ctypes.c_void_p, ctypes.c_long] + [ctypes.c_int] * 4
            L.orc_dequant_rows.restype = ctypes.c_int
            L.orc_dequant_rows.argtypes = [
                ctypes.c_int, ctypes.c_int, ctypes.c_int, ctypes.c_long, ctypes.c_long,
                ctypes.c_void_p, ctypes.c_void_p, ctypes.c_void_p, ctypes.c_void_p,
                ctypes.c_long, ctypes.c_long, c_dbl_p]
            L.orc_gemv.restype = ctypes.c_int
            L.orc_gemv.argtypes = [
                ctypes.c_int, ctypes.c_int, ctypes.c_int, ctypes.c_int, ctypes.c_long,
                ctypes.c_long, ctypes.c_int, ctypes.c_void_p, ctypes.c_void_p, ctypes.c_void_p,
                ctypes.c_void_p, ctypes.c_void_p, ctypes.c_void_p, ctypes.c_void_p,
                ctypes.c_long, ctypes.c_void_p, ctypes.c_void_p, ctypes.c_void_p]
            L.orc_dense_gemv.restype = ctypes.c_int
            L.orc_dense_gemv.argtypes = [ctypes.c_int, ctypes.c_long, ctypes.c_long, ctypes.c_int,
                                         ctypes.c_void_p, ctypes.c_void_p, ctypes.c_void_p,
                                         ctypes.c_void_p, ctypes.c_void_p]
            L.orc_max_threads.restype = ctypes.c_int
            L.orc_set_threads.restype = None
            L.orc_set_threads.argtypes = [ctypes.c_int]
            _LIB = L
    return _LIB


def _ptr(a):
    return None if a is None else a.ctypes.data_as(ctypes.c_void_p)


# ---------------------------------------------------------------------------- code <-> value
def minifloat_values(codes, params) -> np.ndarray:
    """Exact binary64 values of minifloat codes (any integer array)."""
    c = np.ascontiguousarray(np.asarray(codes, dtype=np.uint32).ravel())
    out = np.empty(c.size, dtype=np.float64)
    lib().orc_decode_array(_ptr(c), out.ctypes.data_as(ctypes.POINTER(ctypes.c_double)), c.size, *params)
    return out.reshape(np.shape(codes))


def round_minifloat(x, params) -> np.ndarray:
    """Round binary64 values to minifloat codes, round-to-nearest-even."""
    xs = np.ascontiguousarray(np.asarray(x, dtype=np.float64).ravel())
    out = np.empty(xs.size, dtype=np.uint32)
    lib().orc_round_array(xs.ctypes.data_as(ctypes.POINTER(ctypes.c_double)), _ptr(out), xs.size, *params)
    return out.reshape(np.shape(x))


def e4m3_table() -> np.ndarray:
    return minifloat_values(np.arange(256), E4M3)


def e2m1_table() -> np.ndarray:
    return minifloat_values(np.arange(16), E2M1)


def act_values(bits, act: str) -> np.ndarray:
    return minifloat_values(bits, F16 if act == "f16" else BF16)


def round_act(x, act: str) -> np.ndarray:
    return round_minifloat(x, F16 if act == "f16" else BF16).astype(np.uint16)


# ---------------------------------------------------------------------------- the method
def _gscale_arr(case):
    g = getattr(case, "gscale", None)
    return None if g is None else np.ascontiguousarray(np.asarray(g, dtype=np.float32).reshape(1))


def dequant(case, n0: int = 0, count: int | None = None) -> np.ndarray:
    """Exact dequantised weight rows [n0, n0+count) as float64 [count, K]."""
    count = case.N - n0 if count is None else count
    out = np.empty((count, case.K), dtype=np.float64)
    rc = lib().orc_dequant_rows(
        FORMAT_IDS[case.fmt], case.block_size, int(case.has_zp), case.N, case.K,
        _ptr(case.W), _ptr(case.scales), _ptr(case.zp), _ptr(_gscale_arr(case)), n0, count,
        out.ctypes.data_as(ctypes.POINTER(ctypes.c_double)))
    if rc != 0:
        raise ValueError(f"orc_dequant_rows failed ({rc})")
    return out


def _bias_arr(case):
    b = getattr(case, "bias", None)
    return None if b is None else np.ascontiguousarray(np.asarray(b, dtype=np.uint16).reshape(-1))


def gemv(case, rows=None, M: int | None = None):
    """Oracle GEMV.  Returns (ybits uint16 [M, R], exact float64 [M, R], absdot float64 [M, R])
    for the output columns ``rows`` (all N if None); R = len(rows) or N.  A case with a ``bias``
    gets it added to every row before the rounding (and |bias| in absdot)."""
    M = case.M if M is None else M
    r = None if rows is None else np.ascontiguousarray(np.asarray(rows, dtype=np.int64))
    count = case.N if r is None else r.size
    ybits = np.empty((M, count), dtype=np.uint16)
    exact = np.empty((M, count), dtype=np.float64)
    absdot = np.empty((M, count), dtype=np.float64)
    A = np.ascontiguousarray(case.A[:M])
    rc = lib().orc_gemv(
        FORMAT_IDS[case.fmt], 1 if case.act == "bf16" else 0, case.block_size, int(case.has_zp),
        case.N, case.K, M, _ptr(A), _ptr(case.W), _ptr(case.scales), _ptr(case.zp),
        _ptr(_gscale_arr(case)), _ptr(_bias_arr(case)), _ptr(r), 0 if r is None else r.size,
        _ptr(ybits), _ptr(exact), _ptr(absdot))
    if rc != 0:
        raise ValueError(f"orc_gemv failed ({rc})")
    return ybits, exact, absdot


def dense_gemv(A_bits, B_bits, act: str):
    """Dense oracle GEMV y[M, N] = A[M, K] . B[K, N] (fp16 / bf16 bit patterns, B row-major).
    Returns (ybits uint16 [M, N], exact float64 [M, N], absdot float64 [M, N])."""
    A = np.ascontiguousarray(A_bits, dtype=np.uint16)
    B = np.ascontiguousarray(B_bits, dtype=np.uint16)
    M, K = A.shape
    K2, N = B.shape
    if K2 != K:
        raise ValueError("A is [M, K] and B is [K, N]")
    ybits = np.empty((M, N), dtype=np.uint16)
    exact = np.empty((M, N), dtype=np.float64)
    absdot = np.empty((M, N), dtype=np.float64)
    rc = lib().orc_dense_gemv(1 if act == "bf16" else 0, N, K, M, _ptr(A), _ptr(B), _ptr(ybits),
                              _ptr(exact), _ptr(absdot))
    if rc != 0:
        raise ValueError(f"orc_dense_gemv failed ({rc})")
    return ybits, exact, absdot


def dense_tolerance_violations(A_bits, B_bits, act: str, ybits_gpu, rel: float = 1e-3):
    """The parity bar of tolerance_violations for the dense GEMV."""
    ref_bits, _, absdot = dense_gemv(A_bits, B_bits, act)
    y = act_values(np.asarray(ybits_gpu), act)
    r = act_values(ref_bits, act)
    bound = ulp(r, act) + rel * absdot
    finite = np.isfinite(r)
    with np.errstate(invalid="ignore"):
        err = np.abs(y - r)
    bad = np.where(finite, ~(err <= bound), ~((y == r) | (np.isnan(y) & np.isnan(r))))
    with np.errstate(invalid="ignore", divide="ignore"):  # inf / inf where the oracle overflows
        worst = float(np.max(np.where(finite, err / bound, 0.0))) if r.size else 0.0
    return int(bad.sum()), worst, ref_bits


def max_threads() -> int:
    return int(lib().orc_max_threads())


def set_threads(n: int) -> None:
    lib().orc_set_threads(int(n))


# ---------------------------------------------------------------------------- the parity bar
def ulp(values: np.ndarray, act: str) -> np.ndarray:
    """Spacing of the activation dtype at |values| (fp16: 10, bf16: 7 stored mantissa bits),
    never below the smallest subnormal spacing."""
    v = np.abs(np.asarray(values, dtype=np.float64))
    mbits, qmin = (10, -24) if act == "f16" else (7, -133)
    with np.errstate(divide="ignore"):
        e = np.floor(np.log2(np.where(v > 0, v, 1.0)))
    q = np.exp2(np.maximum(e - mbits, qmin))
    return np.where(v > 0, q, np.exp2(qmin))


def tolerance_violations(case, ybits_gpu: np.ndarray, rows=None, M: int | None = None,
                         rel: float = 1e-3):
    """Compare GPU output bits [M, R] with the oracle on the same inputs.  The bar:
        |y - y_ref| <= 1 ulp(|y_ref|) + rel * (sum_k |a_k * w_k| [+ |bias|])
    with y_ref the oracle's correctly rounded result; infinities must match exactly.
    Returns (number of violations, max |y - y_ref| / bound, oracle bits)."""
    ref_bits, _, absdot = gemv(case, rows=rows, M=M)
    y = act_values(np.asarray(ybits_gpu), case.act)
    r = act_values(ref_bits, case.act)
    bound = ulp(r, case.act) + rel * absdot
    finite = np.isfinite(r)
    with np.errstate(invalid="ignore"):
        err = np.abs(y - r)
    bad = np.where(finite, ~(err <= bound), ~((y == r) | (np.isnan(y) & np.isnan(r))))
    with np.errstate(invalid="ignore", divide="ignore"):  # inf / inf where the oracle overflows
        worst = float(np.max(np.where(finite, err / bound, 0.0))) if r.size else 0.0
    return int(bad.sum()), worst, ref_bits
