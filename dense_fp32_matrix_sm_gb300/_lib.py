"""ctypes binding for libsgemm_gb300.so (the C ABI in include/sgemm.h).

Argument marshalling only: every step of the product runs in the library's
CUDA kernels.  PyTorch is used for device memory and streams.  If the
library has not been built this module raises on first use; there is no
fallback of any kind.
"""
from __future__ import annotations

import ctypes
import os
import threading
from typing import Optional

_PKG = os.path.dirname(os.path.abspath(__file__))
# SGEMM_GB300_LIBRARY=checked loads the checked build (build.py: device-side
# bounds checks that report SGEMM_ERR_BOUNDS instead of touching memory out
# of range); the default is the normal build.
LIB_PATH = os.path.join(_PKG, "libsgemm_gb300_checked.so" if os.environ.get("SGEMM_GB300_LIBRARY") == "checked"
                        else "libsgemm_gb300.so")

SGEMM_OK = 0
SGEMM_ERR_INVALID_ARG = -1
SGEMM_ERR_UNSUPPORTED = -2
SGEMM_ERR_CUDA = -3
SGEMM_ERR_TIMEOUT = -4
SGEMM_ERR_NOMEM = -5
SGEMM_ERR_BOUNDS = -6
SGEMM_TUNE_TENSOR_CORES = 1

# Every function include/sgemm.h declares, with (restype, argtypes).
_i64 = ctypes.c_int64
_vp = ctypes.c_void_p
_int = ctypes.c_int
_f32 = ctypes.c_float
SIGNATURES = {
    "sgemm_plan": (_int, [_i64, _i64, _i64, _i64, _i64, _i64, ctypes.POINTER(_vp)]),
    "sgemm_plan_with_config": (_int, [_i64, _i64, _i64, _i64, _i64, _i64, _int, ctypes.POINTER(_vp)]),
    "sgemm_run": (_int, [_vp, _f32, _vp, _vp, _f32, _vp, _vp]),
    "sgemm_run_host": (_int, [_vp, _f32, _vp, _vp, _f32, _vp, _vp, _vp, _vp, _vp]),
    "sgemm_plan_destroy": (_int, [_vp]),
    "sgemm_plan_describe": (_int, [_vp, ctypes.c_char_p, ctypes.c_size_t]),
    "sgemm_plan_launches": (_int, [_vp, ctypes.POINTER(_int)]),
    "sgemm_plan_config_id": (_int, [_vp, ctypes.POINTER(_int)]),
    "sgemm_num_configs": (_int, []),
    "sgemm_config_name": (ctypes.c_char_p, [_int]),
    "sgemm_status_string": (ctypes.c_char_p, [_int]),
    "sgemm_device_status": (_int, [_int]),
    "sgemm_set_wait_timeout_ns": (_int, [ctypes.c_uint64]),
    "sgemm_wait_limit_ns": (_int, [_i64, _i64, _i64, _i64, _int, ctypes.POINTER(ctypes.c_uint64)]),
    "sgemm_selftest_wait_timeout": (_int, [ctypes.c_uint64, _vp]),
    "sgemm_table_choice": (_int, [_i64, _i64, _i64, _i64, _i64, _i64, _i64, _i64, _int, _int, ctypes.c_char_p,
                                  ctypes.c_size_t, ctypes.POINTER(_int), ctypes.POINTER(_int)]),
    "sgemm_streamk_schedule": (_int, [_i64, _i64, _int, _int, ctypes.POINTER(_i64), ctypes.POINTER(_int),
                                      ctypes.POINTER(_i64)]),
    "sgemm_run_static_scratch": (_int, [_i64, _i64, _i64, _i64, _i64, _i64, _f32, _vp, _vp, _f32, _vp, _vp]),
    "sgemm_plan_ex": (_int, [_int, _int, _int, _i64, _i64, _i64, _i64, _i64, _i64, _int, ctypes.POINTER(_vp)]),
    "sgemm_plan_ex_batched": (_int, [_int, _int, _int, _i64, _i64, _i64, _i64, _i64, _i64, _i64, _i64, _i64, _i64,
                                     _int, ctypes.POINTER(_vp)]),
    "sgemm_run_host_pipelined": (_int, [_vp, _int, _f32, ctypes.POINTER(_vp), ctypes.POINTER(_vp), _f32,
                                        ctypes.POINTER(_vp), ctypes.POINTER(_vp), ctypes.POINTER(_vp),
                                        ctypes.POINTER(_vp), _vp]),
    "sgemm_probe_ffma": (_int, [_int, ctypes.POINTER(ctypes.c_double), ctypes.POINTER(ctypes.c_double)]),
    "sgemm_plan_autotune": (_int, [_i64, _i64, _i64, _i64, _i64, _i64, _vp, _vp, _vp, _int, _vp,
                                   ctypes.POINTER(ctypes.c_double), ctypes.POINTER(_vp)]),
    "sgemm_plan_batched": (_int, [_i64, _i64, _i64, _i64, _i64, _i64, _i64, _i64, _i64, _i64, _int,
                                  ctypes.POINTER(_vp)]),
}

_lib = None
_lock = threading.Lock()


class SgemmError(RuntimeError):
    def __init__(self, status: int, where: str):
        self.status = status
        super().__init__(f"{where}: {status_string(status)} ({status})")


def lib() -> ctypes.CDLL:
    """Load libsgemm_gb300.so (once).  Raises if it has not been built."""
    global _lib
    if _lib is not None:
        return _lib
    with _lock:
        if _lib is None:
            if not os.path.exists(LIB_PATH):
                raise ImportError(
                    f"{LIB_PATH} is missing: build the CUDA library first "
                    "(python -c 'import __graft_entry__ as g; g.build()' or "
                    "python dense_fp32_matrix_sm_gb300/build.py). There is no fallback path.")
            l = ctypes.CDLL(LIB_PATH)
            for name, (res, args) in SIGNATURES.items():
                f = getattr(l, name)
                f.restype = res
                f.argtypes = args
            _lib = l
    return _lib


def status_string(status: int) -> str:
    s = lib().sgemm_status_string(int(status))
    return s.decode() if s else f"status {status}"


def _check(status: int, where: str):
    if status != SGEMM_OK:
        raise SgemmError(status, where)


def num_configs() -> int:
    return int(lib().sgemm_num_configs())


def config_name(config_id: int) -> Optional[str]:
    s = lib().sgemm_config_name(int(config_id))
    return s.decode() if s else None


def config_names():
    return [config_name(i) for i in range(num_configs())]


def config_id(name: str) -> int:
    names = config_names()
    if name not in names:
        raise KeyError(f"unknown variant {name!r}; have {names}")
    return names.index(name)


def device_status(reset: bool = True) -> int:
    """Read (and clear) the current device's kernel status word: SGEMM_OK or SGEMM_ERR_TIMEOUT."""
    return int(lib().sgemm_device_status(1 if reset else 0))


def set_wait_timeout_ns(ns: int) -> None:
    _check(lib().sgemm_set_wait_timeout_ns(int(ns)), "sgemm_set_wait_timeout_ns")


def wait_limit_ns(M: int, N: int, K: int, batch: int = 1, num_sms: int = 152) -> int:
    """The in-kernel wait limit a launch of this product gets (the setting, or its work-based floor)."""
    out = ctypes.c_uint64()
    _check(lib().sgemm_wait_limit_ns(int(M), int(N), int(K), int(batch), int(num_sms), ctypes.byref(out)),
           "sgemm_wait_limit_ns")
    return int(out.value)


def table_choice(M: int, N: int, K: int, lda: Optional[int] = None, ldb: Optional[int] = None, batch: int = 1,
                 stride_a: int = 0, stride_b: int = 0, b_trans: bool = False, num_sms: int = 152):
    """The shape table's variant for a row-major product on a device with num_sms SMs, and whether the
    plan would first copy A / B into padded rows: (name, repack_a, repack_b).  No CUDA call."""
    buf = ctypes.create_string_buffer(128)
    ra, rb = _int(), _int()
    _check(lib().sgemm_table_choice(int(M), int(N), int(K), int(K if lda is None else lda),
                                    int(N if ldb is None else ldb), int(batch), int(stride_a), int(stride_b),
                                    1 if b_trans else 0, int(num_sms), buf, len(buf), ctypes.byref(ra),
                                    ctypes.byref(rb)), "sgemm_table_choice")
    return buf.value.decode(), bool(ra.value), bool(rb.value)


def streamk_schedule(tiles: int, k_slices: int, num_sms: int = 152, ctas_per_sm: int = 1):
    """The persistent grid of a transposed-A plan: (grid, dp_waves, sk_iters).  No CUDA call."""
    g, d, i = _i64(), _int(), _i64()
    _check(lib().sgemm_streamk_schedule(int(tiles), int(k_slices), int(num_sms), int(ctas_per_sm), ctypes.byref(g),
                                        ctypes.byref(d), ctypes.byref(i)), "sgemm_streamk_schedule")
    return int(g.value), int(d.value), int(i.value)


def selftest_wait_timeout(ns: int, stream=None) -> int:
    return int(lib().sgemm_selftest_wait_timeout(int(ns), _stream_handle(stream)))


def _stream_handle(stream) -> Optional[int]:
    if stream is None:
        try:
            import torch

            if torch.cuda.is_available():
                return torch.cuda.current_stream().cuda_stream or None
        except Exception:
            pass
        return None
    if isinstance(stream, int):
        return stream or None
    return getattr(stream, "cuda_stream", None) or None


def _ptr(x) -> Optional[int]:
    if x is None:
        return None
    if isinstance(x, int):
        return x or None
    return x.data_ptr() or None


def _dev_ptr(x, name: str) -> Optional[int]:
    """A device address for sgemm_run: raw integers pass through; a tensor must
    be float32 and on a CUDA device (a host or half-precision buffer handed to
    the kernels would be read as device float32)."""
    if x is not None and not isinstance(x, int):
        if getattr(x, "is_cuda", False) is not True or str(getattr(x, "dtype", "")) != "torch.float32":
            raise TypeError(f"{name} must be a float32 CUDA tensor or a device address")
    return _ptr(x)


class Plan:
    """A plan for one (M, N, K, lda, ldb, ldc) on the current CUDA device.

    config: None for the library's per-shape table, or a variant name / id.
    """

    def __init__(self, M: int, N: int, K: int, lda: Optional[int] = None, ldb: Optional[int] = None,
                 ldc: Optional[int] = None, config=None, order: str = "row", transa: bool = False,
                 transb: bool = False, batch: Optional[int] = None, stride_a: int = 0, stride_b: int = 0,
                 stride_c: int = 0):
        l = lib()
        self.M, self.N, self.K = int(M), int(N), int(K)
        row = order == "row"
        if order not in ("row", "col"):
            raise ValueError("order must be 'row' or 'col'")
        # default leading dimensions: dense stored matrices in the given order
        a_rows, a_cols = (self.K, self.M) if transa else (self.M, self.K)
        b_rows, b_cols = (self.N, self.K) if transb else (self.K, self.N)
        self.lda = int(lda) if lda is not None else max(1, a_cols if row else a_rows)
        self.ldb = int(ldb) if ldb is not None else max(1, b_cols if row else b_rows)
        self.ldc = int(ldc) if ldc is not None else max(1, self.N if row else self.M)
        h = ctypes.c_void_p()
        if batch is not None:
            cid = -1 if config is None else (config if isinstance(config, int) else config_id(config))
            if not row or transa or transb:
                st = l.sgemm_plan_ex_batched(0 if row else 1, 1 if transa else 0, 1 if transb else 0, self.M, self.N,
                                             self.K, self.lda, self.ldb, self.ldc, int(batch), int(stride_a),
                                             int(stride_b), int(stride_c), cid, ctypes.byref(h))
            else:
                st = l.sgemm_plan_batched(self.M, self.N, self.K, self.lda, self.ldb, self.ldc, int(batch),
                                          int(stride_a), int(stride_b), int(stride_c), cid, ctypes.byref(h))
        elif not row or transa or transb:
            cid = -1 if config is None else (config if isinstance(config, int) else config_id(config))
            st = l.sgemm_plan_ex(0 if row else 1, 1 if transa else 0, 1 if transb else 0, self.M, self.N, self.K,
                                 self.lda, self.ldb, self.ldc, cid, ctypes.byref(h))
        elif config is None:
            st = l.sgemm_plan(self.M, self.N, self.K, self.lda, self.ldb, self.ldc, ctypes.byref(h))
        else:
            cid = config if isinstance(config, int) else config_id(config)
            st = l.sgemm_plan_with_config(self.M, self.N, self.K, self.lda, self.ldb, self.ldc, cid,
                                          ctypes.byref(h))
        _check(st, "sgemm_plan")
        self._h = h

    @property
    def handle(self):
        return self._h

    def run(self, alpha: float, A, B, beta: float, C, stream=None) -> None:
        """Enqueue C = alpha*A*B + beta*C.  A, B, C: CUDA tensors (or raw device addresses)."""
        _check(lib().sgemm_run(self._h, float(alpha), _dev_ptr(A, "A"), _dev_ptr(B, "B"), float(beta),
                               _dev_ptr(C, "C"), _stream_handle(stream)), "sgemm_run")

    def run_host(self, alpha: float, hA, hB, beta: float, hC, dA, dB, dC, stream=None) -> None:
        """Host buffers in, host result out: H2D copies, the kernel, D2H copy, all on `stream`."""
        _check(lib().sgemm_run_host(self._h, float(alpha), _ptr(hA), _ptr(hB), float(beta), _ptr(hC),
                                    _ptr(dA), _ptr(dB), _ptr(dC), _stream_handle(stream)), "sgemm_run_host")

    def run_host_pipelined(self, alpha: float, hA, hB, beta: float, hC, dA2, dB2, dC2, stream=None) -> None:
        """len(hC) products from host buffers through two device buffer sets (dA2, dB2, dC2: pairs),
        copies overlapped with the kernels; all results are in host memory once `stream` gets there."""
        n = len(hC)
        arr = lambda xs: (ctypes.c_void_p * len(xs))(*[_ptr(x) for x in xs])
        _check(lib().sgemm_run_host_pipelined(self._h, n, float(alpha), arr(hA), arr(hB), float(beta), arr(hC),
                                              arr(dA2), arr(dB2), arr(dC2), _stream_handle(stream)),
               "sgemm_run_host_pipelined")

    def describe(self) -> str:
        buf = ctypes.create_string_buffer(512)
        _check(lib().sgemm_plan_describe(self._h, buf, 512), "sgemm_plan_describe")
        return buf.value.decode()

    def info(self) -> dict:
        out = {}
        for tok in self.describe().split():
            k, _, v = tok.partition("=")
            out[k] = int(v) if v.lstrip("-").isdigit() else v
        return out

    @property
    def launches(self) -> int:
        n = ctypes.c_int()
        _check(lib().sgemm_plan_launches(self._h, ctypes.byref(n)), "sgemm_plan_launches")
        return n.value

    @property
    def config_id(self) -> int:
        n = ctypes.c_int()
        _check(lib().sgemm_plan_config_id(self._h, ctypes.byref(n)), "sgemm_plan_config_id")
        return n.value

    @property
    def config_name(self) -> str:
        return config_name(self.config_id)

    def close(self) -> None:
        if getattr(self, "_h", None):
            lib().sgemm_plan_destroy(self._h)
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


def _ld(t) -> int:
    if t.dim() != 2:
        raise ValueError("expected a 2-D tensor")
    if t.shape[0] > 0 and t.shape[1] > 0 and t.stride(1) != 1:
        raise ValueError("rows must be contiguous (stride(1) == 1); row-major layout only")
    return max(1, t.stride(0), t.shape[1]) if t.shape[0] > 1 else max(1, t.shape[1])


# Plans made by sgemm(), kept for reuse: (device, M, N, K, lda, ldb, ldc,
# config, stream handle) -> Plan, least recently used first.  A plan's
# stream-K workspace must not be shared by runs that overlap in time, so a
# plan serves one stream only: runs on one stream are ordered.
_PLAN_CACHE_MAX = 64
_plan_cache = {}
_plan_cache_lock = threading.Lock()


def _cached_plan(key, make):
    with _plan_cache_lock:
        plan = _plan_cache.pop(key, None)
        if plan is None:
            plan = make()
        _plan_cache[key] = plan  # most recently used last
        evicted = []
        while len(_plan_cache) > _PLAN_CACHE_MAX:
            evicted.append(_plan_cache.pop(next(iter(_plan_cache))))
    for p in evicted:
        p.close()
    return plan


def clear_plan_cache() -> None:
    """Destroy every plan sgemm() keeps (frees their device workspaces; the
    frees synchronise the device)."""
    with _plan_cache_lock:
        plans = list(_plan_cache.values())
        _plan_cache.clear()
    for p in plans:
        p.close()


def plan_cache_size() -> int:
    with _plan_cache_lock:
        return len(_plan_cache)


def sgemm(A, B, C=None, alpha: float = 1.0, beta: float = 0.0, stream=None, config=None):
    """C = alpha*A*B + beta*C for row-major float32 CUDA tensors; returns C.

    C is allocated (and beta must be 0) when not given.  Runs on the current
    stream unless `stream` is given.

    Plans are cached per (device, shape, leading dimensions, config, stream):
    the first call for a key makes a plan, which may allocate its device
    workspace (cudaMalloc); later calls reuse it and allocate nothing of the
    library's, so they only enqueue work and do not synchronise.  At most 64
    plans are kept; the least recently used one is destroyed beyond that,
    and destroying a plan with a workspace frees it (cudaFree synchronises
    the device).  clear_plan_cache() drops them all.
    """
    import torch

    for name, t in (("A", A), ("B", B)):
        if t.dtype != torch.float32 or not t.is_cuda:
            raise TypeError(f"{name} must be a float32 CUDA tensor")
    M, K = A.shape
    K2, N = B.shape
    if K != K2:
        raise ValueError(f"inner dimensions differ: {tuple(A.shape)} x {tuple(B.shape)}")
    if C is None:
        if beta != 0.0:
            raise ValueError("beta != 0 needs C")
        C = torch.empty((M, N), dtype=torch.float32, device=A.device)
    if C.dtype != torch.float32 or not C.is_cuda or tuple(C.shape) != (M, N):
        raise TypeError("C must be an M x N float32 CUDA tensor")
    lda, ldb, ldc = _ld(A) if K > 0 else 1, _ld(B), _ld(C)
    key = (A.device.index if A.device.index is not None else torch.cuda.current_device(), M, N, K, lda, ldb, ldc,
           config, _stream_handle(stream))
    with torch.cuda.device(A.device):
        plan = _cached_plan(key, lambda: Plan(M, N, K, lda, ldb, ldc, config=config))
        plan.run(alpha, A, B, beta, C, stream)
    return C


def run_static_scratch(M: int, N: int, K: int, alpha: float, A, B, beta: float, C, lda: Optional[int] = None,
                       ldb: Optional[int] = None, ldc: Optional[int] = None, stream=None) -> None:
    """Enqueue C = alpha*A*B + beta*C through sgemm_run_static_scratch: no plan and no allocation.
    The scratch is shared per device, so calls must not overlap in time.
    A, B, C: CUDA tensors or raw device addresses; ld* default to dense rows."""
    M, N, K = int(M), int(N), int(K)
    lda = int(lda) if lda is not None else max(1, K)
    ldb = int(ldb) if ldb is not None else max(1, N)
    ldc = int(ldc) if ldc is not None else max(1, N)
    _check(lib().sgemm_run_static_scratch(M, N, K, lda, ldb, ldc, float(alpha), _ptr(A), _ptr(B), float(beta),
                                          _ptr(C), _stream_handle(stream)), "sgemm_run_static_scratch")


def probe_ffma(paired: bool = True):
    """(TFLOP/s, SM MHz measured inside the kernel) of an FMA-only kernel on the current device."""
    t = ctypes.c_double()
    f = ctypes.c_double()
    _check(lib().sgemm_probe_ffma(1 if paired else 0, ctypes.byref(t), ctypes.byref(f)), "sgemm_probe_ffma")
    return t.value, f.value


def autotune(M: int, N: int, K: int, A, B, C, lda: Optional[int] = None, ldb: Optional[int] = None,
             ldc: Optional[int] = None, tensor_cores: bool = False, stream=None, with_times: bool = False):
    """Time every variant that takes this shape on the scratch buffers A, B, C (C is overwritten) and
    return a Plan for the fastest; with_times also returns {variant name: ms per run}."""
    M, N, K = int(M), int(N), int(K)
    lda = int(lda) if lda is not None else max(1, K)
    ldb = int(ldb) if ldb is not None else max(1, N)
    ldc = int(ldc) if ldc is not None else max(1, N)
    n = num_configs()
    times = (ctypes.c_double * n)() if with_times else None
    h = ctypes.c_void_p()
    _check(lib().sgemm_plan_autotune(M, N, K, lda, ldb, ldc, _ptr(A), _ptr(B), _ptr(C),
                                     SGEMM_TUNE_TENSOR_CORES if tensor_cores else 0, _stream_handle(stream),
                                     times, ctypes.byref(h)), "sgemm_plan_autotune")
    plan = Plan.__new__(Plan)
    plan.M, plan.N, plan.K, plan.lda, plan.ldb, plan.ldc = M, N, K, lda, ldb, ldc
    plan._h = h
    if not with_times:
        return plan
    return plan, {config_name(i): times[i] for i in range(n) if times[i] >= 0}
