"""Fused N-way partial reduce + residual add + RMSNorm (+ per-token FP8 E4M3) on GB300.

A thin ctypes binding over ``libar.so`` (see ``include/ar.h``).  The functions named like
the C ABI (``ar_init``, ``ar_reduce_sum``, ``ar_fused_reduce_rmsnorm``,
``ar_fused_reduce_rmsnorm_batch``, ``ar_fused_reduce_rmsnorm_host``,
``ar_fused_reduce_rmsnorm_noalloc``, ``ar_destroy`` ...) take raw pointers and sizes exactly
as the C functions do; the ``Context`` methods (``reduce_sum``, ``fused_reduce_rmsnorm``,
``fused_reduce_rmsnorm_batch``, ``fused_reduce_rmsnorm_host``) marshal torch tensors into
those calls.  Every step of the computation runs in the library's CUDA kernels: there is no
Python or PyTorch compute path, and using the package without a built ``libar.so`` raises.
"""
from __future__ import annotations

import ctypes
import os
from typing import Optional, Sequence

PKG = os.path.dirname(os.path.abspath(__file__))
LIB_PATH = os.path.join(PKG, "libar.so")

# ---- mirrors of include/ar.h ----------------------------------------------
AR_OK = 0
AR_ERR_INVALID_ARG = 1
AR_ERR_UNSUPPORTED = 2
AR_ERR_ALIGNMENT = 3
AR_ERR_CUDA = 4
AR_ERR_NOT_INITIALIZED = 5
AR_ERR_OVERLAP = 6

AR_DTYPE_F32 = 0
AR_DTYPE_F16 = 1
AR_DTYPE_BF16 = 2
AR_MAX_PARTIALS = 8
AR_MAX_BATCH = 16
AR_QUANT_NONE = 0
AR_QUANT_FP8_E4M3_PER_TOKEN = 1
AR_QUANT_FP8_E4M3_PER_GROUP = 2

AR_OPT_FORCE_VARIANT = 0
AR_OPT_CLUSTER_SIZE = 1
AR_OPT_PACKS_PER_THREAD = 2
AR_OPT_REDUCE_UNROLL = 3
AR_OPT_STAGES = 4
AR_OPT_PDL = 5
AR_OPT_WAIT_CYCLES = 6
AR_OPT_TEST_STALL = 7
AR_OPT_L2_PREFETCH = 8
VARIANT_AUTO, VARIANT_ROW, VARIANT_CLUSTER, VARIANT_STAGED, VARIANT_SCALAR = 0, 1, 2, 3, 4

AR_INFO_SM_COUNT = 0
AR_INFO_L2_BYTES = 1
AR_INFO_REDUCE_TILE_PACKS = 2
AR_INFO_DEVICE = 3


class ArFusedArgs(ctypes.Structure):
    _fields_ = [
        ("n", ctypes.c_int),
        ("partials", ctypes.c_void_p * AR_MAX_PARTIALS),
        ("residual_in", ctypes.c_void_p),
        ("residual_out", ctypes.c_void_p),
        ("weight", ctypes.c_void_p),
        ("out", ctypes.c_void_p),
        ("eps", ctypes.c_float),
        ("gemma", ctypes.c_int),
        ("quant", ctypes.c_int),
        ("q_out", ctypes.c_void_p),
        ("scale_out", ctypes.c_void_p),
        ("m", ctypes.c_int64),
        ("h", ctypes.c_int64),
        ("dtype", ctypes.c_int),
        ("skip_norm", ctypes.c_int),
        ("out_fp32", ctypes.c_int),
        ("group_size", ctypes.c_int),
        ("ld_in", ctypes.c_int64),
        ("ld_out", ctypes.c_int64),
    ]


class ArError(RuntimeError):
    def __init__(self, status: int, where: str, detail: str = ""):
        self.status = status
        msg = f"{where}: {status_string(status)} ({status})"
        if detail:
            msg += f": {detail}"
        super().__init__(msg)


_lib: Optional[ctypes.CDLL] = None


def load_library(path: str = LIB_PATH) -> ctypes.CDLL:
    """Load libar.so once.  Raises if it has not been built (no fallback exists)."""
    global _lib
    if _lib is not None:
        return _lib
    if not os.path.exists(path):
        raise RuntimeError(f"{path} is missing: build it first (python -c 'import __graft_entry__ as g; g.build()')")
    lib = ctypes.CDLL(path)
    vp, i64, c_int = ctypes.c_void_p, ctypes.c_int64, ctypes.c_int
    lib.ar_init.argtypes = [ctypes.POINTER(vp), c_int, ctypes.c_uint]
    lib.ar_destroy.argtypes = [vp]
    lib.ar_reduce_sum.argtypes = [vp, vp, ctypes.POINTER(vp), c_int, i64, c_int, vp]
    lib.ar_fused_reduce_rmsnorm.argtypes = [vp, ctypes.POINTER(ArFusedArgs), vp]
    lib.ar_fused_reduce_rmsnorm_host.argtypes = [vp, ctypes.POINTER(ArFusedArgs), vp]
    lib.ar_fused_reduce_rmsnorm_noalloc.argtypes = [ctypes.POINTER(ArFusedArgs), vp]
    lib.ar_status_string.argtypes = [c_int]
    lib.ar_status_string.restype = ctypes.c_char_p
    lib.ar_last_error.argtypes = [vp]
    lib.ar_last_error.restype = ctypes.c_char_p
    lib.ar_last_variant.argtypes = [vp]
    lib.ar_last_variant.restype = ctypes.c_char_p
    lib.ar_set_option.argtypes = [vp, c_int, i64]
    lib.ar_get_info.argtypes = [vp, c_int, ctypes.POINTER(i64)]
    lib.ar_device_status.argtypes = [vp, ctypes.POINTER(c_int)]
    lib.ar_fused_reduce_rmsnorm_batch.argtypes = [vp, ctypes.POINTER(ArFusedArgs), c_int, vp]
    for f in ("ar_init", "ar_destroy", "ar_reduce_sum", "ar_fused_reduce_rmsnorm", "ar_set_option",
              "ar_get_info", "ar_device_status", "ar_fused_reduce_rmsnorm_batch", "ar_fused_reduce_rmsnorm_host",
              "ar_fused_reduce_rmsnorm_noalloc"):
        getattr(lib, f).restype = c_int
    _lib = lib
    return lib


def ar_status_string(status: int) -> str:
    return load_library().ar_status_string(int(status)).decode()


status_string = ar_status_string


# ---- the C ABI, one Python function per entry point -------------------------

def ar_init(device: int = 0, flags: int = 0) -> int:
    """Create a context; returns its opaque handle (an int)."""
    lib = load_library()
    h = ctypes.c_void_p()
    st = lib.ar_init(ctypes.byref(h), int(device), int(flags))
    if st != AR_OK:
        raise ArError(st, "ar_init")
    return h.value


def ar_destroy(ctx: Optional[int]) -> None:
    st = load_library().ar_destroy(ctx)
    if st != AR_OK:
        raise ArError(st, "ar_destroy")


def ar_last_variant(ctx: int) -> str:
    return load_library().ar_last_variant(ctx).decode()


def ar_last_error(ctx: int) -> str:
    return load_library().ar_last_error(ctx).decode()


def ar_set_option(ctx: int, opt: int, value: int) -> None:
    st = load_library().ar_set_option(ctx, int(opt), int(value))
    if st != AR_OK:
        raise ArError(st, "ar_set_option")


def ar_get_info(ctx: int, key: int) -> int:
    v = ctypes.c_int64()
    st = load_library().ar_get_info(ctx, int(key), ctypes.byref(v))
    if st != AR_OK:
        raise ArError(st, "ar_get_info")
    return v.value


def ar_device_status(ctx: int) -> int:
    """Read and clear the context's device status word (0: no bounded wait ran out)."""
    v = ctypes.c_int()
    st = load_library().ar_device_status(ctx, ctypes.byref(v))
    if st != AR_OK:
        raise ArError(st, "ar_device_status")
    return v.value


def _check(ctx, st, where):
    if st != AR_OK:
        raise ArError(st, where, ar_last_error(ctx) if (ctx and st == AR_ERR_CUDA) else "")


def ar_reduce_sum(ctx: int, out: int, partials: Sequence[int], numel: int, dtype: int,
                  stream: Optional[int] = None, raise_on_error: bool = True) -> int:
    """out[i] = round_T(sum_r partials[r][i]).  Pointers are device addresses (ints)."""
    n = len(partials)
    arr = (ctypes.c_void_p * max(n, 1))(*partials)
    st = load_library().ar_reduce_sum(ctx, out, arr, n, int(numel), int(dtype), stream)
    if raise_on_error:
        _check(ctx, st, "ar_reduce_sum")
    return st


def ar_fused_reduce_rmsnorm(ctx: int, args: ArFusedArgs, stream: Optional[int] = None,
                            raise_on_error: bool = True) -> int:
    st = load_library().ar_fused_reduce_rmsnorm(ctx, ctypes.byref(args), stream)
    if raise_on_error:
        _check(ctx, st, "ar_fused_reduce_rmsnorm")
    return st


def ar_fused_reduce_rmsnorm_host(ctx: int, args: ArFusedArgs, stream: Optional[int] = None,
                                 raise_on_error: bool = True) -> int:
    st = load_library().ar_fused_reduce_rmsnorm_host(ctx, ctypes.byref(args), stream)
    if raise_on_error:
        _check(ctx, st, "ar_fused_reduce_rmsnorm_host")
    return st


def ar_fused_reduce_rmsnorm_noalloc(args: ArFusedArgs, stream: Optional[int] = None,
                                    raise_on_error: bool = True) -> int:
    """The allocation-free form (no context; the calling thread's current device)."""
    st = load_library().ar_fused_reduce_rmsnorm_noalloc(ctypes.byref(args), stream)
    if raise_on_error:
        _check(None, st, "ar_fused_reduce_rmsnorm_noalloc")
    return st


def ar_fused_reduce_rmsnorm_batch(ctx: int, calls: Sequence[ArFusedArgs], stream: Optional[int] = None,
                                  raise_on_error: bool = True) -> int:
    arr = (ArFusedArgs * max(len(calls), 1))(*calls)
    st = load_library().ar_fused_reduce_rmsnorm_batch(ctx, arr, len(calls), stream)
    if raise_on_error:
        _check(ctx, st, "ar_fused_reduce_rmsnorm_batch")
    return st


def make_fused_args(partials: Sequence[int], residual_in: Optional[int], residual_out: Optional[int],
                    weight: Optional[int], out: Optional[int], eps: float, gemma: bool, quant: bool,
                    q_out: Optional[int], scale_out: Optional[int], m: int, h: int, dtype: int,
                    skip_norm: bool = False, out_fp32: bool = False, group_size: int = 0,
                    ld_in: int = 0, ld_out: int = 0) -> ArFusedArgs:
    a = ArFusedArgs()
    a.n = len(partials)
    for i, p in enumerate(partials):
        a.partials[i] = p
    a.residual_in = residual_in
    a.residual_out = residual_out
    a.weight = weight
    a.out = out
    a.eps = eps
    a.gemma = int(bool(gemma))
    a.quant = (AR_QUANT_FP8_E4M3_PER_GROUP if group_size else AR_QUANT_FP8_E4M3_PER_TOKEN) if quant else AR_QUANT_NONE
    a.group_size = int(group_size)
    a.ld_in = int(ld_in)
    a.ld_out = int(ld_out)
    a.q_out = q_out
    a.scale_out = scale_out
    a.m = m
    a.h = h
    a.dtype = dtype
    a.skip_norm = int(bool(skip_norm))
    a.out_fp32 = int(bool(out_fp32))
    return a


# ---- torch marshalling -----------------------------------------------------

def _torch_dtype_code(t) -> int:
    import torch
    return {torch.float32: AR_DTYPE_F32, torch.float16: AR_DTYPE_F16, torch.bfloat16: AR_DTYPE_BF16}[t.dtype]


def _ptr(t) -> Optional[int]:
    return None if t is None else t.data_ptr()


def _stream(stream) -> int:
    import torch
    if stream is None:
        stream = torch.cuda.current_stream()
    return stream.cuda_stream


def _row_stride(tensors, m, h, dtype, what, host: bool = False) -> int:
    """The common row stride (in elements) of [m, h] CUDA tensors (with `host`, CUDA or
    pinned host tensors) with unit column stride."""
    ld = None
    for t in tensors:
        if t is None:
            continue
        placed = t.is_cuda or (host and t.is_pinned())
        if t.shape != (m, h) or not placed or (dtype is not None and t.dtype != dtype) or \
                (h > 1 and t.stride(1) != 1) or (m > 1 and t.stride(0) < h):
            kind = "CUDA or pinned host" if host else "CUDA"
            raise ValueError(f"{what} must be [m, h] {kind} tensors with unit column stride")
        s = t.stride(0) if m > 1 else h
        if ld is not None and s != ld:
            raise ValueError(f"{what} must share one row stride")
        ld = s
    return h if ld is None else ld


class Context:
    """Owns one ar_ctx for a device; torch-tensor front end of the C ABI."""

    def __init__(self, device: int = 0):
        self.device = device
        self.handle = ar_init(device)

    def close(self):
        if self.handle:
            ar_destroy(self.handle)
            self.handle = None

    def __enter__(self):
        return self

    def __exit__(self, *exc):
        self.close()

    def __del__(self):
        try:
            self.close()
        except Exception:
            pass

    @property
    def last_variant(self) -> str:
        return ar_last_variant(self.handle)

    def set_option(self, opt: int, value: int):
        ar_set_option(self.handle, opt, value)

    def info(self, key: int) -> int:
        return ar_get_info(self.handle, key)

    def device_status(self) -> int:
        return ar_device_status(self.handle)

    def reduce_sum(self, partials, out=None, stream=None):
        """Sum contiguous same-shaped device tensors in rank order; returns `out`."""
        import torch
        x0 = partials[0]
        for p in partials:
            if p.shape != x0.shape or p.dtype != x0.dtype or not p.is_contiguous() or not p.is_cuda:
                raise ValueError("partials must be contiguous CUDA tensors of one shape and dtype")
        if out is None:
            out = torch.empty_like(x0)
        ar_reduce_sum(self.handle, out.data_ptr(), [p.data_ptr() for p in partials], x0.numel(),
                      _torch_dtype_code(x0), _stream(stream))
        return out

    def fused_reduce_rmsnorm(self, partials, residual, weight, eps: float = 1e-6, gemma: bool = False,
                             quant: bool = False, out=None, residual_out=None, q_out=None, scale_out=None,
                             want_out: bool = True, want_residual_out: bool = True, stream=None,
                             skip_norm: bool = False, out_fp32: bool = False, group_size: int = 0):
        """Returns (out, residual_out, q_out, scale_out); absent outputs are None.  With
        skip_norm there is no RMSNorm (weight may be None); with out_fp32 `out` is float32.
        Inputs (and given outputs) may have padded rows: unit column stride, one row stride
        for the inputs and one for the outputs; allocated outputs are contiguous."""
        return self._fused(False, partials, residual, weight, eps, gemma, quant, out, residual_out, q_out,
                           scale_out, want_out, want_residual_out, stream, skip_norm, out_fp32, group_size)

    def fused_reduce_rmsnorm_host(self, partials, residual, weight, eps: float = 1e-6, gemma: bool = False,
                                  quant: bool = False, out=None, residual_out=None, q_out=None, scale_out=None,
                                  want_out: bool = True, want_residual_out: bool = True, stream=None,
                                  skip_norm: bool = False, out_fp32: bool = False, group_size: int = 0):
        """fused_reduce_rmsnorm where tensors may be pinned host tensors (or CUDA tensors of
        this device): the kernel reads and writes host memory directly.  Outputs it allocates
        are pinned host tensors.  Asynchronous: synchronise `stream` before reading them."""
        return self._fused(True, partials, residual, weight, eps, gemma, quant, out, residual_out, q_out,
                           scale_out, want_out, want_residual_out, stream, skip_norm, out_fp32, group_size)

    def _fused(self, host, partials, residual, weight, eps, gemma, quant, out, residual_out, q_out, scale_out,
               want_out, want_residual_out, stream, skip_norm, out_fp32, group_size):
        import torch
        x0 = partials[0]
        m, h = x0.shape

        def alloc(shape, dtype):
            if host:
                return torch.empty(shape, dtype=dtype, pin_memory=True)
            return torch.empty(shape, dtype=dtype, device=x0.device)

        ld_in = _row_stride([*partials, residual], m, h, x0.dtype, "partials and residual", host)
        given = [t for t in (out, residual_out, q_out) if t is not None]
        ld_out = _row_stride(given, m, h, None, "outputs", host) if given else h
        if ld_out != h and ((out is None and (want_out or not quant)) or (residual_out is None and want_residual_out)
                            or (quant and q_out is None)):
            raise ValueError("with padded outputs every output must be given")
        if out is None and (want_out or not quant):
            out = alloc((m, h), torch.float32 if out_fp32 else x0.dtype)
        if residual_out is None and want_residual_out:
            residual_out = alloc((m, h), x0.dtype)
        if quant:
            if q_out is None:
                q_out = alloc((m, h), torch.uint8)
            if scale_out is None:
                scale_out = alloc((m, h // group_size) if group_size else (m,), torch.float32)
        args = make_fused_args([p.data_ptr() for p in partials], _ptr(residual), _ptr(residual_out),
                               _ptr(weight), _ptr(out), eps, gemma, quant, _ptr(q_out), _ptr(scale_out),
                               m, h, _torch_dtype_code(x0), skip_norm=skip_norm, out_fp32=out_fp32,
                               group_size=group_size, ld_in=ld_in, ld_out=ld_out)
        (ar_fused_reduce_rmsnorm_host if host else ar_fused_reduce_rmsnorm)(self.handle, args, _stream(stream))
        return out, residual_out, q_out, scale_out

    def fused_reduce_rmsnorm_batch(self, calls, stream=None):
        """Several independent fused calls in one launch.  `calls` is a list of dicts with the
        keyword arguments of fused_reduce_rmsnorm (partials, residual, weight, eps, gemma,
        quant, out, residual_out, q_out, scale_out, skip_norm, out_fp32); missing outputs are
        allocated.  Returns a list of (out, residual_out, q_out, scale_out)."""
        import torch
        results, args = [], []
        for c in calls:
            x0 = c["partials"][0]
            m, h = x0.shape
            quant, out_fp32 = c.get("quant", False), c.get("out_fp32", False)
            out = c.get("out")
            if out is None and (c.get("want_out", True) or not quant):
                out = torch.empty((m, h), dtype=torch.float32 if out_fp32 else x0.dtype, device=x0.device)
            ro = c.get("residual_out")
            if ro is None and c.get("want_residual_out", True):
                ro = torch.empty_like(x0)
            q = c.get("q_out")
            sc = c.get("scale_out")
            g = c.get("group_size", 0)
            if quant:
                q = q if q is not None else torch.empty((m, h), dtype=torch.uint8, device=x0.device)
                sc = sc if sc is not None else torch.empty((m, h // g) if g else (m,), dtype=torch.float32,
                                                           device=x0.device)
            ld_in = _row_stride([*c["partials"], c.get("residual")], m, h, x0.dtype, "partials and residual")
            outs = [t for t in (out, ro, q) if t is not None]
            ld_out = _row_stride(outs, m, h, None, "outputs") if outs else h
            args.append(make_fused_args([p.data_ptr() for p in c["partials"]], _ptr(c.get("residual")), _ptr(ro),
                                        _ptr(c.get("weight")), _ptr(out), c.get("eps", 1e-6), c.get("gemma", False),
                                        quant, _ptr(q), _ptr(sc), m, h, _torch_dtype_code(x0),
                                        skip_norm=c.get("skip_norm", False), out_fp32=out_fp32, group_size=g,
                                        ld_in=ld_in, ld_out=ld_out))
            results.append((out, ro, q, sc))
        ar_fused_reduce_rmsnorm_batch(self.handle, args, _stream(stream))
        return results
