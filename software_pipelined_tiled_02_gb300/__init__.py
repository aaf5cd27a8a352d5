"""Software-pipelined tiled GEMM for GB300: Python binding of ``libtgemm.so``.

``C[M,N] = A[M,K] . B[N,K]^T`` with fp16/bf16 operands and fp32 accumulation,
computed by the hand-written sm_103a kernel behind the C ABI declared in
``include/tgemm.h``.  This module only marshals arguments: it passes torch
tensors' device pointers and CUDA streams to the library and maps status
codes to exceptions.  There is no fallback: if ``libtgemm.so`` is missing or
fails to load, every call raises.

The same names as the C ABI are exported (``tgemm_plan`` ... ``tgemm_strerror``)
plus a ``Plan`` wrapper and ``gemm()``.
"""

from __future__ import annotations

import collections
import ctypes
import os
import threading

HERE = os.path.dirname(os.path.abspath(__file__))
LIB_PATH = os.path.join(HERE, "libtgemm.so")

F16, BF16, F32 = 0, 1, 2
OK, ERR_INVALID_ARG, ERR_UNSUPPORTED_DTYPE, ERR_ALIGNMENT, ERR_SMEM_BUDGET, ERR_NO_KERNEL, ERR_ARCH, ERR_CUDA, \
    ERR_TIMEOUT, ERR_CHECK = range(10)
_DT_NAMES = {"f16": F16, "bf16": BF16, "f32": F32}

SYMBOLS = ("tgemm_smem_bound", "tgemm_smem_bytes", "tgemm_smem_limit", "tgemm_validate", "tgemm_plan",
           "tgemm_run", "tgemm_run_host", "tgemm_status", "tgemm_set_watchdog_ns", "tgemm_debug_stall",
           "tgemm_get_plan_info", "tgemm_destroy", "tgemm_strerror", "tgemm_run_noalloc", "tgemm_plan_ex",
           "tgemm_validate_ex")


class TgemmError(RuntimeError):
    def __init__(self, code: int, what: str = ""):
        self.code = code
        super().__init__(f"{what}: {strerror(code)} (code {code})" if what else strerror(code))


class PlanInfo(ctypes.Structure):
    _fields_ = [("M", ctypes.c_int64), ("N", ctypes.c_int64), ("K", ctypes.c_int64),
                ("dtype", ctypes.c_int), ("out_dtype", ctypes.c_int), ("block_M", ctypes.c_int),
                ("block_N", ctypes.c_int), ("block_K", ctypes.c_int), ("num_stages", ctypes.c_int),
                ("tiles_m", ctypes.c_int), ("tiles_n", ctypes.c_int), ("num_tiles", ctypes.c_int),
                ("grid", ctypes.c_int), ("threads", ctypes.c_int), ("num_k_blocks", ctypes.c_int),
                ("acc_stages", ctypes.c_int), ("tmem_columns", ctypes.c_int), ("smem_bytes", ctypes.c_int64),
                ("smem_bound", ctypes.c_int64), ("smem_limit", ctypes.c_int), ("num_sms", ctypes.c_int),
                ("cta_pair", ctypes.c_int), ("split_k", ctypes.c_int), ("num_units", ctypes.c_int),
                ("prefetch", ctypes.c_int), ("cluster_k", ctypes.c_int), ("stream_operands", ctypes.c_int),
                ("grid_reduce", ctypes.c_int), ("stream_k_tiles", ctypes.c_int), ("multicast_b", ctypes.c_int)]

    def as_dict(self):
        return {name: getattr(self, name) for name, _ in self._fields_}


class PlanOpts(ctypes.Structure):
    _fields_ = [("cta_pair", ctypes.c_int), ("group_m", ctypes.c_int), ("split_k", ctypes.c_int),
                ("prefetch", ctypes.c_int), ("cluster_k", ctypes.c_int), ("stream_operands", ctypes.c_int),
                ("grid_reduce", ctypes.c_int), ("stream_k", ctypes.c_int), ("multicast_b", ctypes.c_int)]


_lock = threading.Lock()
_lib = None


def load(path: str | None = None):
    """Load ``libtgemm.so`` (raises if it is absent: there is no fallback).
    The environment variable ``TGEMM_LIB`` names another build of the same
    library, such as the debug-check build ``libtgemm_debug.so``."""
    global _lib
    with _lock:
        if _lib is not None:
            return _lib
        path = path or os.environ.get("TGEMM_LIB") or LIB_PATH
        if not os.path.exists(path):
            raise RuntimeError(f"libtgemm.so not built at {path}; run software_pipelined_tiled_02_gb300/build.py "
                               "or __graft_entry__.build()")
        L = ctypes.CDLL(path)
        i64, i32, vp = ctypes.c_int64, ctypes.c_int, ctypes.c_void_p
        L.tgemm_smem_bound.argtypes = [i32] * 5
        L.tgemm_smem_bound.restype = i64
        L.tgemm_smem_bytes.argtypes = [i32] * 6
        L.tgemm_smem_bytes.restype = i64
        L.tgemm_smem_limit.argtypes = []
        L.tgemm_smem_limit.restype = i32
        L.tgemm_validate.argtypes = [i64, i64, i64, i32, i32, i32, i32, i32, i32, i64]
        L.tgemm_validate.restype = i32
        L.tgemm_plan.argtypes = [ctypes.POINTER(vp), i64, i64, i64, i32, i32, i32, i32, i32, i32]
        L.tgemm_plan.restype = i32
        L.tgemm_run.argtypes = [vp, vp, vp, vp, vp]
        L.tgemm_run.restype = i32
        L.tgemm_run_host.argtypes = [vp] * 8
        L.tgemm_run_host.restype = i32
        L.tgemm_status.argtypes = [vp, ctypes.POINTER(ctypes.c_int)]
        L.tgemm_status.restype = i32
        L.tgemm_set_watchdog_ns.argtypes = [vp, ctypes.c_uint64]
        L.tgemm_set_watchdog_ns.restype = i32
        L.tgemm_debug_stall.argtypes = [vp, i32]
        L.tgemm_debug_stall.restype = i32
        L.tgemm_get_plan_info.argtypes = [vp, ctypes.POINTER(PlanInfo)]
        L.tgemm_get_plan_info.restype = i32
        L.tgemm_destroy.argtypes = [vp]
        L.tgemm_destroy.restype = i32
        L.tgemm_run_noalloc.argtypes = [i64, i64, i64, i32, i32, i32, i32, i32, i32, vp, vp, vp, vp,
                                        ctypes.POINTER(ctypes.c_int)]
        L.tgemm_run_noalloc.restype = i32
        L.tgemm_plan_ex.argtypes = [ctypes.POINTER(vp), i64, i64, i64, i32, i32, i32, i32, i32, i32,
                                    ctypes.POINTER(PlanOpts)]
        L.tgemm_plan_ex.restype = i32
        L.tgemm_validate_ex.argtypes = [i64, i64, i64, i32, i32, i32, i32, i32, i32, i64, ctypes.POINTER(PlanOpts)]
        L.tgemm_validate_ex.restype = i32
        L.tgemm_strerror.argtypes = [i32]
        L.tgemm_strerror.restype = ctypes.c_char_p
        _lib = L
        return L


def _dt(x) -> int:
    if isinstance(x, int):
        return x
    if isinstance(x, str):
        return _DT_NAMES[x]
    import torch

    return {torch.float16: F16, torch.bfloat16: BF16, torch.float32: F32}[x]


def _torch_dtype(code: int):
    import torch

    return {F16: torch.float16, BF16: torch.bfloat16, F32: torch.float32}[code]


# ------------------------------------------------------------- C ABI names

def tgemm_smem_bound(dtype, block_M, block_N, block_K, num_stages) -> int:
    return int(load().tgemm_smem_bound(_dt(dtype), block_M, block_N, block_K, num_stages))


def tgemm_smem_bytes(dtype, out_dtype, block_M, block_N, block_K, num_stages) -> int:
    return int(load().tgemm_smem_bytes(_dt(dtype), _dt(out_dtype), block_M, block_N, block_K, num_stages))


def tgemm_smem_limit() -> int:
    return int(load().tgemm_smem_limit())


def tgemm_validate(M, N, K, dtype, out_dtype, block_M, block_N, block_K, num_stages, smem_limit) -> int:
    return int(load().tgemm_validate(M, N, K, _dt(dtype), _dt(out_dtype), block_M, block_N, block_K, num_stages,
                                     smem_limit))


def tgemm_plan(M, N, K, dtype, out_dtype, block_M, block_N, block_K, num_stages):
    """Returns ``(status, handle)``; handle is None on failure."""
    h = ctypes.c_void_p()
    rc = load().tgemm_plan(ctypes.byref(h), M, N, K, _dt(dtype), _dt(out_dtype), block_M, block_N, block_K,
                           num_stages)
    return int(rc), (h if rc == OK else None)


def tgemm_plan_ex(M, N, K, dtype, out_dtype, block_M, block_N, block_K, num_stages, cta_pair=0, group_m=0,
                  split_k=0, prefetch=0, cluster_k=0, stream_operands=0, grid_reduce=0, stream_k=0, multicast_b=0):
    """Returns ``(status, handle)``; handle is None on failure."""
    h = ctypes.c_void_p()
    opts = PlanOpts(int(cta_pair), int(group_m), int(split_k), int(prefetch), int(cluster_k), int(stream_operands),
                    int(grid_reduce), int(stream_k), int(multicast_b))
    rc = load().tgemm_plan_ex(ctypes.byref(h), M, N, K, _dt(dtype), _dt(out_dtype), block_M, block_N, block_K,
                              num_stages, ctypes.byref(opts))
    return int(rc), (h if rc == OK else None)


def tgemm_validate_ex(M, N, K, dtype, out_dtype, block_M, block_N, block_K, num_stages, smem_limit, cta_pair=0,
                      group_m=0, split_k=0, prefetch=0, cluster_k=0, stream_operands=0, grid_reduce=0,
                      stream_k=0, multicast_b=0) -> int:
    opts = PlanOpts(int(cta_pair), int(group_m), int(split_k), int(prefetch), int(cluster_k), int(stream_operands),
                    int(grid_reduce), int(stream_k), int(multicast_b))
    return int(load().tgemm_validate_ex(M, N, K, _dt(dtype), _dt(out_dtype), block_M, block_N, block_K,
                                        num_stages, smem_limit, ctypes.byref(opts)))


def tgemm_run(plan, A_ptr: int, B_ptr: int, C_ptr: int, stream: int = 0) -> int:
    return int(load().tgemm_run(plan, A_ptr, B_ptr, C_ptr, stream))


def tgemm_run_host(plan, hA: int, hB: int, hC: int, dA: int, dB: int, dC: int, stream: int = 0) -> int:
    return int(load().tgemm_run_host(plan, hA, hB, hC, dA, dB, dC, stream))


def tgemm_status(plan):
    d = (ctypes.c_int * 4)()
    rc = load().tgemm_status(plan, d)
    return int(rc), list(d)


def tgemm_set_watchdog_ns(plan, ns: int) -> int:
    return int(load().tgemm_set_watchdog_ns(plan, ns))


def tgemm_debug_stall(plan, on: bool) -> int:
    return int(load().tgemm_debug_stall(plan, 1 if on else 0))


def tgemm_get_plan_info(plan) -> dict:
    info = PlanInfo()
    rc = load().tgemm_get_plan_info(plan, ctypes.byref(info))
    if rc != OK:
        raise TgemmError(rc, "tgemm_get_plan_info")
    return info.as_dict()


def tgemm_destroy(plan) -> int:
    return int(load().tgemm_destroy(plan))


def tgemm_run_noalloc(M, N, K, dtype, out_dtype, block_M, block_N, block_K, num_stages, A_ptr: int, B_ptr: int,
                      C_ptr: int, stream: int = 0, want_status: bool = True):
    """The allocation-free entry point: returns (return code, kernel status or None)."""
    st = ctypes.c_int(-1)
    rc = load().tgemm_run_noalloc(M, N, K, _dt(dtype), _dt(out_dtype), block_M, block_N, block_K, num_stages,
                                  A_ptr, B_ptr, C_ptr, stream, ctypes.byref(st) if want_status else None)
    return int(rc), (int(st.value) if want_status else None)


def strerror(code: int) -> str:
    try:
        return load().tgemm_strerror(int(code)).decode()
    except RuntimeError:
        return f"status {code}"


tgemm_strerror = strerror


# ------------------------------------------------------------- conveniences

class Plan:
    """A validated GEMM configuration on the current CUDA device."""

    def __init__(self, M, N, K, dtype="f16", out_dtype=None, block=(128, 256, 64), num_stages=4, pair=False,
                 split_k=1, prefetch=0, group_m=0, cluster_k=0, stream_operands=False, grid_reduce=False,
                 stream_k=False, multicast_b=False):
        dtype = _dt(dtype)
        out_dtype = dtype if out_dtype is None else _dt(out_dtype)
        bm, bn, bk = block
        if (pair or split_k > 1 or prefetch or group_m or cluster_k > 1 or stream_operands or grid_reduce or stream_k
                or multicast_b):
            rc, h = tgemm_plan_ex(M, N, K, dtype, out_dtype, bm, bn, bk, num_stages, cta_pair=int(bool(pair)),
                                  split_k=int(split_k), prefetch=int(prefetch), group_m=int(group_m),
                                  cluster_k=int(cluster_k), stream_operands=int(bool(stream_operands)),
                                  grid_reduce=int(bool(grid_reduce)), stream_k=int(bool(stream_k)),
                                  multicast_b=int(bool(multicast_b)))
        else:
            rc, h = tgemm_plan(M, N, K, dtype, out_dtype, bm, bn, bk, num_stages)
        if rc != OK:
            raise TgemmError(rc, f"tgemm_plan(M={M}, N={N}, K={K}, block={block}, num_stages={num_stages}, "
                                 f"pair={pair}, split_k={split_k}, cluster_k={cluster_k}, "
                                 f"stream_operands={stream_operands}, multicast_b={multicast_b})")
        self.pair = bool(pair)
        self.split_k = int(split_k)
        self.cluster_k = int(cluster_k)
        self.handle = h
        self.lock = threading.Lock()  # a plan serves one host thread at a time
        self.M, self.N, self.K = M, N, K
        self.dtype, self.out_dtype = dtype, out_dtype
        self.block, self.num_stages = tuple(block), num_stages

    @property
    def info(self) -> dict:
        return tgemm_get_plan_info(self.handle)

    def _check(self, A, B, C):
        import torch

        for name, t, shape, dt in (("A", A, (self.M, self.K), self.dtype), ("B", B, (self.N, self.K), self.dtype),
                                   ("C", C, (self.M, self.N), self.out_dtype)):
            if t.dtype != _torch_dtype(dt):
                raise TypeError(f"{name} must be {_torch_dtype(dt)}, got {t.dtype}")
            if tuple(t.shape) != shape:
                raise ValueError(f"{name} must have shape {shape}, got {tuple(t.shape)}")
            if not t.is_contiguous():
                raise ValueError(f"{name} must be contiguous (row-major)")
        if not (A.is_cuda and B.is_cuda and C.is_cuda):
            raise ValueError("A, B and C must be CUDA tensors")
        if not (A.device == B.device == C.device == torch.device("cuda", torch.cuda.current_device())):
            raise ValueError("A, B, C must be on the current CUDA device")

    def run(self, A, B, C=None, stream=None):
        """Enqueue ``C = A . B^T`` on ``stream`` (default: torch's current stream); returns C."""
        import torch

        if C is None:
            C = torch.empty((self.M, self.N), dtype=_torch_dtype(self.out_dtype), device=A.device)
        self._check(A, B, C)
        s = (stream if stream is not None else torch.cuda.current_stream()).cuda_stream
        rc = tgemm_run(self.handle, A.data_ptr(), B.data_ptr(), C.data_ptr(), s)
        if rc != OK:
            raise TgemmError(rc, "tgemm_run")
        return C

    def run_host(self, hA, hB, hC, dA, dB, dC, stream=None):
        """Host operands in, host result out (copies enqueued by the library).

        hA, hB, hC are CPU tensors (pinned for asynchronous copies), dA, dB, dC
        the device buffers the library copies through; all contiguous, with
        the plan's shapes and dtypes."""
        import torch

        self._check(dA, dB, dC)
        for name, h, d in (("hA", hA, dA), ("hB", hB, dB), ("hC", hC, dC)):
            if h.is_cuda:
                raise ValueError(f"{name} must be a host (CPU) tensor")
            if h.dtype != d.dtype or tuple(h.shape) != tuple(d.shape):
                raise ValueError(f"{name} must match its device buffer: {d.dtype} {tuple(d.shape)}, "
                                 f"got {h.dtype} {tuple(h.shape)}")
            if not h.is_contiguous():
                raise ValueError(f"{name} must be contiguous (row-major)")
        s = (stream if stream is not None else torch.cuda.current_stream()).cuda_stream
        rc = tgemm_run_host(self.handle, hA.data_ptr(), hB.data_ptr(), hC.data_ptr(), dA.data_ptr(),
                            dB.data_ptr(), dC.data_ptr(), s)
        if rc != OK:
            raise TgemmError(rc, "tgemm_run_host")
        return hC

    def status(self):
        """Read and clear the device status word; (code, detail)."""
        return tgemm_status(self.handle)

    def set_watchdog_ns(self, ns: int):
        tgemm_set_watchdog_ns(self.handle, ns)

    def debug_stall(self, on: bool):
        tgemm_debug_stall(self.handle, on)

    def close(self):
        if self.handle is not None:
            tgemm_destroy(self.handle)
            self.handle = None

    def __del__(self):
        try:
            self.close()
        except Exception:
            pass


# gemm()'s plans, least recently used first.  Bounded, because every plan holds
# device memory (its status word, and a workspace when K is split).
_plans: "collections.OrderedDict" = collections.OrderedDict()
_plans_lock = threading.Lock()
_PLANS_MAX = 64


def default_config(M, N, K, dtype="f16", out_dtype=None) -> dict:
    """The tuned default {block, num_stages, cta_pair, split_k, group_m, cluster_k, stream_operands,
    grid_reduce, stream_k, multicast_b} for a shape."""
    from . import defaults

    return defaults.choose(M, N, K, _dt(dtype), _dt(dtype) if out_dtype is None else _dt(out_dtype))


def gemm(A, B, out_dtype=None, block=None, num_stages=None, out=None, stream=None, pair=None, split_k=None,
         group_m=None, cluster_k=None, stream_operands=None, grid_reduce=None, stream_k=None, multicast_b=None):
    """``A[M,K] . B[N,K]^T`` on the GPU through ``libtgemm.so``.

    ``out_dtype`` defaults to the operand dtype; ``torch.float32`` returns the
    raw fp32 accumulator.  ``block``/``num_stages`` default to the tuned table,
    and so does every launch option left as None.
    """
    M, K = A.shape
    N, K2 = B.shape
    if K != K2:
        raise ValueError("A and B must agree on K")
    dt = _dt(A.dtype)
    odt = dt if out_dtype is None else _dt(out_dtype)
    if block is None or num_stages is None:
        cfg = default_config(M, N, K, dt, odt)
        block = block or cfg["block"]
        num_stages = num_stages or cfg["num_stages"]
    else:
        from . import defaults

        cfg = defaults.DEFAULT_OPTS
    pair = bool(cfg["cta_pair"] if pair is None else pair)
    split_k = int((cfg["split_k"] if split_k is None else split_k) or 1)
    group_m = int((cfg["group_m"] if group_m is None else group_m) or 0)
    cluster_k = int((cfg["cluster_k"] if cluster_k is None else cluster_k) or 0)
    stream_operands = bool(cfg["stream_operands"] if stream_operands is None else stream_operands)
    grid_reduce = bool(cfg["grid_reduce"] if grid_reduce is None else grid_reduce)
    stream_k = bool(cfg["stream_k"] if stream_k is None else stream_k)
    multicast_b = bool(cfg["multicast_b"] if multicast_b is None else multicast_b)
    key = (M, N, K, dt, odt, tuple(block), num_stages, pair, split_k, group_m, cluster_k, stream_operands,
           grid_reduce, stream_k, multicast_b, A.device.index)
    # The cache lock covers the lookup only; the enqueue holds the plan's own
    # lock (a plan caches tensor maps per pointer triple, so one host thread
    # at a time), so threads running different plans do not serialise.
    while True:
        with _plans_lock:
            plan = _plans.get(key)
            if plan is None:
                plan = _plans[key] = Plan(M, N, K, dt, odt, block, num_stages, pair=pair, split_k=split_k,
                                          group_m=group_m, cluster_k=cluster_k, stream_operands=stream_operands,
                                          grid_reduce=grid_reduce, stream_k=stream_k, multicast_b=multicast_b)
                while len(_plans) > _PLANS_MAX:
                    victim = _plans.popitem(last=False)[1]
                    with victim.lock:  # waits for an enqueue in progress on it
                        victim.close()
            else:
                _plans.move_to_end(key)
        with plan.lock:
            if plan.handle is None:  # evicted between the lookup and here: look up again
                continue
            return plan.run(A, B, out, stream)
