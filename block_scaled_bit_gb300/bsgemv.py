"""ctypes binding to ``libbsgemv.so`` (the C ABI of include/bsgemv.h).

Argument marshalling only: every step of the GEMV runs in the library's CUDA kernels.  Tensors
are torch tensors (device memory and streams are torch's); their data pointers are passed as
plain addresses.  Importing this module loads the library and raises if it has not been built
(``python -c "import __graft_entry__ as g; g.build()"``) -- there is no fallback.
"""
from __future__ import annotations

import ctypes
import os

from . import _build

FORMATS = {"int4": 1, "int8": 2, "fp8": 3, "nvfp4": 4}
ACT_BF16 = 0x100
VARIANTS = {"auto": 0, "mma": 1, "cuda_core": 2}
SPLITS = {"auto": 0, "stream_k": 1, "cluster": 2}

OK = 0
ERR_INVALID_ARG = -1
ERR_UNSUPPORTED = -2
ERR_MISALIGNED = -3
ERR_M_TOO_LARGE = -4
ERR_CUDA = -5
ERR_WRONG_DEVICE = -6
ERR_DEVICE_TIMEOUT = -7
ERR_SCRATCH_LIMIT = -8

# Every extern "C" entry point of include/bsgemv.h.
EXPORTS = ("bsgemv_plan", "bsgemv_run", "bsgemv_run_bias", "bsgemv_run_host",
           "bsgemv_run_host_async", "bsgemv_destroy",
           "bsgemv_status_string", "bsgemv_debug_dequant", "bsgemv_plan_set_override",
           "bsgemv_plan_describe", "bsgemv_geometry_for", "bsgemv_device_status",
           "bsgemv_run_noalloc", "bsgemv_plan_set_split", "bsgemv_plan_autotune",
           "bsgemv_plan_set_test_fault",
           "bsgemv_dense_plan", "bsgemv_dense_run", "bsgemv_dense_describe",
           "bsgemv_dense_geometry_for", "bsgemv_dense_device_status", "bsgemv_dense_destroy",
           "bsgemv_version")


class Geometry(ctypes.Structure):
    _fields_ = [("variant", ctypes.c_int), ("rows_per_tile", ctypes.c_int),
                ("k_per_stage", ctypes.c_int), ("stages", ctypes.c_int),
                ("consumer_warps", ctypes.c_int), ("ctas", ctypes.c_int),
                ("ctas_per_sm", ctypes.c_int), ("sm_count", ctypes.c_int),
                ("tiles", ctypes.c_int64), ("stages_per_tile", ctypes.c_int64),
                ("total_stages", ctypes.c_int64), ("smem_bytes", ctypes.c_int),
                ("workspace_bytes", ctypes.c_int64), ("cluster", ctypes.c_int)]

    def as_dict(self) -> dict:
        return {name: getattr(self, name) for name, _ in self._fields_}


class BsgemvError(RuntimeError):
    def __init__(self, status: int, what: str):
        self.status = status
        super().__init__(f"{what}: {status_string(status)} ({status})")


_LIB = None


def lib_path() -> str:
    return _build.LIB_PATH


def lib() -> ctypes.CDLL:
    global _LIB
    if _LIB is None:
        path = lib_path()
        if not os.path.exists(path):
            raise RuntimeError(f"{path} is missing: build the CUDA library first "
                               "(python -c 'import __graft_entry__ as g; g.build()')")
        L = ctypes.CDLL(path)
        vp, i64, ci = ctypes.c_void_p, ctypes.c_int64, ctypes.c_int
        L.bsgemv_plan.argtypes = [ctypes.POINTER(vp), ci, ci, ci, i64, i64, ci]
        L.bsgemv_run.argtypes = [vp, vp, vp, vp, vp, vp, ci, vp]
        L.bsgemv_run_bias.argtypes = [vp, vp, vp, vp, vp, vp, vp, ci, vp]
        L.bsgemv_run_host.argtypes = [vp, vp, vp, vp, vp, vp, ci, vp]
        L.bsgemv_run_host_async.argtypes = [vp, vp, vp, vp, vp, vp, ci, vp]
        L.bsgemv_destroy.argtypes = [vp]
        L.bsgemv_status_string.argtypes = [ci]
        L.bsgemv_status_string.restype = ctypes.c_char_p
        L.bsgemv_debug_dequant.argtypes = [vp, vp, vp, vp, vp, vp]
        L.bsgemv_plan_set_override.argtypes = [vp, ci, ci, ci, ci]
        L.bsgemv_plan_set_split.argtypes = [vp, ci, ci]
        L.bsgemv_plan_autotune.argtypes = [vp, vp, vp, vp, vp, vp, ci, ci, vp]
        L.bsgemv_dense_plan.argtypes = [ctypes.POINTER(vp), ci, i64, i64, ci]
        L.bsgemv_dense_run.argtypes = [vp, vp, vp, vp, ci, vp]
        L.bsgemv_dense_describe.argtypes = [vp, ctypes.POINTER(Geometry)]
        L.bsgemv_dense_geometry_for.argtypes = [ci, i64, i64, ci, ci, ctypes.POINTER(Geometry)]
        L.bsgemv_dense_device_status.argtypes = [vp, vp]
        L.bsgemv_dense_destroy.argtypes = [vp]
        L.bsgemv_plan_describe.argtypes = [vp, ctypes.POINTER(Geometry)]
        L.bsgemv_geometry_for.argtypes = [ci, ci, ci, i64, i64, ci, ci, ctypes.POINTER(Geometry)]
        L.bsgemv_device_status.argtypes = [vp, vp]
        L.bsgemv_run_noalloc.argtypes = [ci, ci, ci, i64, i64, vp, vp, vp, vp, vp, ci, vp]
        L.bsgemv_plan_set_test_fault.argtypes = [vp, ci, i64]
        for name in EXPORTS:
            if name != "bsgemv_status_string":
                getattr(L, name).restype = ci
        _LIB = L
    return _LIB


def status_string(status: int) -> str:
    return lib().bsgemv_status_string(int(status)).decode()


def _check(status: int, what: str) -> None:
    if status != OK:
        raise BsgemvError(status, what)


def format_code(fmt: str, act: str) -> int:
    return FORMATS[fmt] | (ACT_BF16 if act == "bf16" else 0)


def geometry_for(fmt: str, act: str, block_size: int, has_zp: bool, N: int, K: int, max_M: int,
                 sm_count: int) -> dict:
    """The launch geometry a plan would take on a device with `sm_count` SMs (no GPU needed)."""
    g = Geometry()
    _check(lib().bsgemv_geometry_for(format_code(fmt, act), block_size, int(has_zp), N, K,
                                     max_M, sm_count, ctypes.byref(g)), "bsgemv_geometry_for")
    return g.as_dict()


def run_noalloc_status(fmt: str, act: str, block_size: int, has_zp: bool, N: int, K: int, A, W,
                       scales, zp, y, M: int | None = None, stream=None) -> int:
    """One GEMV through bsgemv_run_noalloc (no plan, no allocation); returns the status."""
    M = A.shape[0] if M is None else M
    return lib().bsgemv_run_noalloc(format_code(fmt, act), block_size, int(has_zp), N, K, _ptr(A),
                                    _ptr(W), _ptr(scales), _ptr(zp), _ptr(y), int(M),
                                    _stream(stream))


def noalloc_device_status(stream=None) -> int:
    """Read and clear bsgemv_run_noalloc's error word on the current device (after a stream
    synchronisation): bsgemv_device_status(NULL, stream)."""
    return lib().bsgemv_device_status(None, _stream(stream))


def _ptr(t) -> int | None:
    if t is None:
        return None
    if isinstance(t, int):
        return t
    return t.data_ptr()


def _stream(stream) -> int | None:
    if stream is None:
        import torch
        return torch.cuda.current_stream().cuda_stream
    return getattr(stream, "cuda_stream", stream)


class Plan:
    """A plan for one weight shape: y[M, N] = A[M, K] . deq(W)[N, K]^T for M <= max_M."""

    def __init__(self, fmt: str, act: str, block_size: int, has_zp: bool, N: int, K: int,
                 max_M: int = 16):
        self.fmt, self.act, self.block_size, self.has_zp = fmt, act, block_size, bool(has_zp)
        self.N, self.K, self.max_M = N, K, max_M
        h = ctypes.c_void_p()
        _check(lib().bsgemv_plan(ctypes.byref(h), format_code(fmt, act), block_size,
                                 int(has_zp), N, K, max_M), "bsgemv_plan")
        self._h = h

    def close(self) -> None:
        if getattr(self, "_h", None) is not None and self._h.value:
            lib().bsgemv_destroy(self._h)
            self._h = None

    def __del__(self):
        try:
            self.close()
        except Exception:
            pass

    def __enter__(self):
        return self

    def __exit__(self, *exc):
        self.close()

    @property
    def handle(self) -> int:
        return self._h.value

    def run_status(self, A, W, scales, zp, y, M: int | None = None, stream=None,
                   bias=None) -> int:
        """Enqueue the GEMV (plus `bias` [N] if given); returns the library status instead of
        raising."""
        M = A.shape[0] if M is None and hasattr(A, "shape") else M
        if bias is not None:
            return lib().bsgemv_run_bias(self._h, _ptr(A), _ptr(W), _ptr(scales), _ptr(zp),
                                         _ptr(bias), _ptr(y), int(M), _stream(stream))
        return lib().bsgemv_run(self._h, _ptr(A), _ptr(W), _ptr(scales), _ptr(zp), _ptr(y),
                                int(M), _stream(stream))

    def run(self, A, W, scales, zp, y, M: int | None = None, stream=None, bias=None) -> None:
        _check(self.run_status(A, W, scales, zp, y, M, stream, bias),
               "bsgemv_run" if bias is None else "bsgemv_run_bias")

    def run_host(self, A_host, W, scales, zp, y_host, M: int | None = None, stream=None) -> None:
        """A and y in host memory (pinned for asynchronous copies); returns when y is ready."""
        M = A_host.shape[0] if M is None else M
        _check(lib().bsgemv_run_host(self._h, _ptr(A_host), _ptr(W), _ptr(scales), _ptr(zp),
                                     _ptr(y_host), int(M), _stream(stream)), "bsgemv_run_host")

    def run_host_async(self, A_host, W, scales, zp, y_host, M: int | None = None,
                       stream=None) -> None:
        """As run_host, but only enqueued: y_host is ready after the stream is synchronised."""
        M = A_host.shape[0] if M is None else M
        _check(lib().bsgemv_run_host_async(self._h, _ptr(A_host), _ptr(W), _ptr(scales), _ptr(zp),
                                           _ptr(y_host), int(M), _stream(stream)),
               "bsgemv_run_host_async")

    def debug_dequant(self, W, scales, zp, out, stream=None) -> None:
        _check(lib().bsgemv_debug_dequant(self._h, _ptr(W), _ptr(scales), _ptr(zp), _ptr(out),
                                          _stream(stream)), "bsgemv_debug_dequant")

    def set_override(self, variant: int = 0, ctas: int = 0, stages: int = 0,
                     rows_per_tile: int = 0) -> int:
        return lib().bsgemv_plan_set_override(self._h, variant, ctas, rows_per_tile, stages)

    def set_split(self, split: str = "auto", cluster: int = 0) -> int:
        """K split of the tiles: "auto", "stream_k" or "cluster" (cluster = CTAs per tile)."""
        return lib().bsgemv_plan_set_split(self._h, SPLITS[split], cluster)

    def autotune_status(self, A, W, scales, zp, y, M: int | None = None, reps: int = 4,
                        stream=None) -> int:
        """Time the plan's candidate geometries on the device (back-to-back calls over weight
        copies that keep L2 cold) and keep the fastest; returns the library status."""
        M = A.shape[0] if M is None and hasattr(A, "shape") else M
        return lib().bsgemv_plan_autotune(self._h, _ptr(A), _ptr(W), _ptr(scales), _ptr(zp),
                                          _ptr(y), int(M), int(reps), _stream(stream))

    def autotune(self, A, W, scales, zp, y, M: int | None = None, reps: int = 4,
                 stream=None) -> dict:
        _check(self.autotune_status(A, W, scales, zp, y, M, reps, stream), "bsgemv_plan_autotune")
        return self.describe()

    def describe(self) -> dict:
        g = Geometry()
        _check(lib().bsgemv_plan_describe(self._h, ctypes.byref(g)), "bsgemv_plan_describe")
        return g.as_dict()

    def device_status(self, stream=None) -> int:
        return lib().bsgemv_device_status(self._h, _stream(stream))

    def set_test_fault(self, skip_stage: int = -1, wait_ns: int = 0) -> int:
        """Test hook of the bounded waits (bsgemv_plan_set_test_fault): CTA 0's copy warp leaves
        out stage `skip_stage` of its range, the waits give up after `wait_ns`; (-1, 0) undoes it."""
        return lib().bsgemv_plan_set_test_fault(self._h, int(skip_stage), int(wait_ns))


def dense_geometry_for(act: str, N: int, K: int, max_M: int, sm_count: int) -> dict:
    """The geometry a dense plan would take on a device with `sm_count` SMs (no GPU needed)."""
    g = Geometry()
    _check(lib().bsgemv_dense_geometry_for(1 if act == "bf16" else 0, N, K, max_M, sm_count,
                                           ctypes.byref(g)), "bsgemv_dense_geometry_for")
    return g.as_dict()


class DensePlan:
    """The dense small-N GEMV y[M, N] = A[M, K] . B[K, N] (B row-major) for M <= max_M <= 8."""

    def __init__(self, act: str, N: int, K: int, max_M: int = 8):
        self.act, self.N, self.K, self.max_M = act, N, K, max_M
        h = ctypes.c_void_p()
        _check(lib().bsgemv_dense_plan(ctypes.byref(h), 1 if act == "bf16" else 0, N, K, max_M),
               "bsgemv_dense_plan")
        self._h = h

    def close(self) -> None:
        if getattr(self, "_h", None) is not None and self._h.value:
            lib().bsgemv_dense_destroy(self._h)
            self._h = None

    def __del__(self):
        try:
            self.close()
        except Exception:
            pass

    def __enter__(self):
        return self

    def __exit__(self, *exc):
        self.close()

    def run_status(self, A, B, y, M: int | None = None, stream=None) -> int:
        M = A.shape[0] if M is None and hasattr(A, "shape") else M
        return lib().bsgemv_dense_run(self._h, _ptr(A), _ptr(B), _ptr(y), int(M), _stream(stream))

    def run(self, A, B, y, M: int | None = None, stream=None) -> None:
        _check(self.run_status(A, B, y, M, stream), "bsgemv_dense_run")

    def describe(self) -> dict:
        g = Geometry()
        _check(lib().bsgemv_dense_describe(self._h, ctypes.byref(g)), "bsgemv_dense_describe")
        return g.as_dict()

    def device_status(self, stream=None) -> int:
        return lib().bsgemv_dense_device_status(self._h, _stream(stream))


def upload(case, device="cuda"):
    """Copy a host case (numpy arrays in the storage layouts) to device tensors and allocate y.
    Returns an object with A, W, scales, zp (the NVFP4 global scale for nvfp4), bias (None
    without one) and y."""
    import types

    import numpy as np
    import torch

    def t(a):
        if a is None:
            return None
        a = np.ascontiguousarray(a)
        if a.dtype == np.uint16:
            a = a.view(np.int16)
        return torch.from_numpy(a).to(device)

    zp = t(case.gscale) if case.fmt == "nvfp4" else t(case.zp)
    y = torch.empty((case.M, case.N), dtype=torch.int16, device=device)
    return types.SimpleNamespace(A=t(case.A), W=t(case.W), scales=t(case.scales), zp=zp,
                                 bias=t(getattr(case, "bias", None)), y=y)


def y_bits(y) -> "np.ndarray":
    """Device output tensor (int16 storage) -> numpy uint16 bit patterns."""
    return y.cpu().numpy().view("uint16")
