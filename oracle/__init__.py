"""CPU oracle for the fused N-way reduce + residual add + RMSNorm (+ per-token FP8) path.

TEST INFRASTRUCTURE ONLY.  The tests, ``__graft_entry__.smoke()`` and the CPU-baseline
leg of ``bench.py`` may import this module; the product package
(``tensor_all_reduce_gb300``) never does, and the two share no code.

The arithmetic lives in ``ar_oracle.c`` (plain serial C, strict IEEE, compiled with
``-ffp-contract=off``); this module only marshals numpy arrays into it.

Array conventions: bf16/fp16 data are ``numpy.uint16`` bit patterns, fp32 data are
``numpy.float32``, FP8 codes are ``numpy.uint8``; everything is C-contiguous.
"""
from __future__ import annotations

import ctypes
import os
import subprocess
from typing import Optional, Sequence

import numpy as np

_HERE = os.path.dirname(os.path.abspath(__file__))
_SRC = os.path.join(_HERE, "ar_oracle.c")
_HDR = os.path.join(_HERE, "ar_oracle.h")
_LIB = os.path.join(_HERE, "liboracle.so")

DTYPES = {"fp32": 0, "fp16": 1, "bf16": 2}
CFLAGS = ["-std=c11", "-O2", "-ffp-contract=off", "-fno-fast-math", "-fPIC", "-shared"]


def build(src: str = _SRC, out: str = _LIB, extra: Sequence[str] = ()) -> str:
    """Compile the oracle C source into a shared library (gcc, a second or so)."""
    cmd = ["gcc", *CFLAGS, *extra, "-I", os.path.dirname(os.path.abspath(src)), "-o", out, src, "-lm"]
    subprocess.run(cmd, check=True)
    return out


def _stale(lib: str) -> bool:
    if not os.path.exists(lib):
        return True
    t = os.path.getmtime(lib)
    return any(os.path.getmtime(p) > t for p in (_SRC, _HDR))


def load(path: Optional[str] = None) -> ctypes.CDLL:
    """Load (building first if missing or stale) an oracle shared library."""
    if path is None:
        path = _LIB
        if _stale(path):
            build()
    lib = ctypes.CDLL(path)
    vp, i64, c_int, c_float = ctypes.c_void_p, ctypes.c_int64, ctypes.c_int, ctypes.c_float
    for name in ("orc_f32_to_bf16_n", "orc_bf16_to_f32_n", "orc_f32_to_f16_n",
                 "orc_f16_to_f32_n", "orc_f32_to_e4m3_n", "orc_e4m3_to_f32_n"):
        getattr(lib, name).argtypes = [vp, vp, i64]
        getattr(lib, name).restype = None
    lib.orc_f64_to_bf16.argtypes = [ctypes.c_double]
    lib.orc_f64_to_bf16.restype = ctypes.c_uint16
    lib.orc_f64_to_f16.argtypes = [ctypes.c_double]
    lib.orc_f64_to_f16.restype = ctypes.c_uint16
    lib.orc_reduce_sum.argtypes = [vp, vp, c_int, i64, c_int]
    lib.orc_reduce_sum.restype = c_int
    lib.orc_add_rmsnorm.argtypes = [vp, vp, vp, vp, vp, i64, i64, c_float, c_int, c_int]
    lib.orc_add_rmsnorm.restype = c_int
    lib.orc_per_token_quant.argtypes = [vp, vp, vp, i64, i64, c_int]
    lib.orc_per_token_quant.restype = c_int
    lib.orc_fused_reduce_rmsnorm.argtypes = [vp, vp, vp, vp, vp, c_int, vp, vp, i64, i64,
                                             c_float, c_int, c_int, c_int]
    lib.orc_fused_reduce_rmsnorm.restype = c_int
    lib.orc_fused_ex.argtypes = [vp, vp, vp, vp, vp, vp, c_int, vp, vp, i64, i64, c_float, c_int, c_int,
                                 c_int, i64, c_int]
    lib.orc_per_group_quant.argtypes = [vp, vp, vp, i64, i64, i64, c_int]
    lib.orc_per_group_quant.restype = c_int
    lib.orc_fused_ex.restype = c_int
    return lib


class Oracle:
    """numpy front end over one loaded oracle library."""

    def __init__(self, path: Optional[str] = None):
        self.lib = load(path)

    # ---- helpers -------------------------------------------------------
    @staticmethod
    def _ptr(a: Optional[np.ndarray]):
        if a is None:
            return None
        assert a.flags["C_CONTIGUOUS"], "oracle arrays must be C-contiguous"
        return a.ctypes.data

    @staticmethod
    def _storage(dtype: str):
        return np.float32 if dtype == "fp32" else np.uint16

    def _check(self, a: np.ndarray, dtype: str, name: str):
        want = self._storage(dtype)
        if a.dtype != want:
            raise TypeError(f"{name}: expected {np.dtype(want)} storage for {dtype}, got {a.dtype}")

    # ---- format conversions -------------------------------------------
    def f32_to_bits(self, x, dtype: str) -> np.ndarray:
        x = np.ascontiguousarray(x, dtype=np.float32)
        out = np.empty(x.shape, np.uint16)
        fn = self.lib.orc_f32_to_bf16_n if dtype == "bf16" else self.lib.orc_f32_to_f16_n
        fn(self._ptr(out), self._ptr(x), x.size)
        return out

    def bits_to_f32(self, h, dtype: str) -> np.ndarray:
        h = np.ascontiguousarray(h, dtype=np.uint16)
        out = np.empty(h.shape, np.float32)
        fn = self.lib.orc_bf16_to_f32_n if dtype == "bf16" else self.lib.orc_f16_to_f32_n
        fn(self._ptr(out), self._ptr(h), h.size)
        return out

    def f64_to_bits(self, x: float, dtype: str) -> int:
        fn = self.lib.orc_f64_to_bf16 if dtype == "bf16" else self.lib.orc_f64_to_f16
        return int(fn(float(x)))

    def f32_to_e4m3(self, x) -> np.ndarray:
        x = np.ascontiguousarray(x, dtype=np.float32)
        out = np.empty(x.shape, np.uint8)
        self.lib.orc_f32_to_e4m3_n(self._ptr(out), self._ptr(x), x.size)
        return out

    def e4m3_to_f32(self, c) -> np.ndarray:
        c = np.ascontiguousarray(c, dtype=np.uint8)
        out = np.empty(c.shape, np.float32)
        self.lib.orc_e4m3_to_f32_n(self._ptr(out), self._ptr(c), c.size)
        return out

    # ---- the method ----------------------------------------------------
    def reduce_sum(self, partials: Sequence[np.ndarray], dtype: str) -> np.ndarray:
        ps = [np.ascontiguousarray(p) for p in partials]
        for k, p in enumerate(ps):
            self._check(p, dtype, f"partials[{k}]")
            if p.shape != ps[0].shape:
                raise ValueError("partials differ in shape")
        out = np.empty(ps[0].shape, self._storage(dtype))
        arr = (ctypes.c_void_p * len(ps))(*[self._ptr(p) for p in ps])
        rc = self.lib.orc_reduce_sum(self._ptr(out), arr, len(ps), out.size, DTYPES[dtype])
        if rc != 0:
            raise ValueError(f"orc_reduce_sum rejected its arguments ({rc})")
        return out

    def add_rmsnorm(self, s, res_in, w, eps: float, gemma: bool, dtype: str):
        """rmsnorm2d_fwd_with_add: returns (y, res_out)."""
        s = np.ascontiguousarray(s)
        m, h = s.shape
        y = np.empty((m, h), np.uint16)
        res_out = np.empty((m, h), np.uint16)
        rc = self.lib.orc_add_rmsnorm(self._ptr(y), self._ptr(res_out), self._ptr(s),
                                      self._ptr(None if res_in is None else np.ascontiguousarray(res_in)),
                                      self._ptr(np.ascontiguousarray(w)), m, h, eps, int(bool(gemma)),
                                      DTYPES[dtype])
        if rc != 0:
            raise ValueError(f"orc_add_rmsnorm rejected its arguments ({rc})")
        return y, res_out

    def per_token_quant(self, y, dtype: str):
        """dynamic per-token FP8 e4m3 quantisation: returns (q, scale)."""
        y = np.ascontiguousarray(y)
        m, h = y.shape
        q = np.empty((m, h), np.uint8)
        scale = np.empty((m,), np.float32)
        rc = self.lib.orc_per_token_quant(self._ptr(q), self._ptr(scale), self._ptr(y), m, h, DTYPES[dtype])
        if rc != 0:
            raise ValueError(f"orc_per_token_quant rejected its arguments ({rc})")
        return q, scale

    def fused(self, partials: Sequence[np.ndarray], res_in, w, eps: float, gemma: bool,
              quant: bool, dtype: str, want_y: bool = True, want_res_out: bool = True) -> dict:
        """The whole path.  Returns a dict with y, res_out, q, scale (None when not produced)."""
        ps = [np.ascontiguousarray(p) for p in partials]
        m, h = ps[0].shape
        y = np.empty((m, h), np.uint16) if (want_y or not quant) else None
        res_out = np.empty((m, h), np.uint16) if want_res_out else None
        q = np.empty((m, h), np.uint8) if quant else None
        scale = np.empty((m,), np.float32) if quant else None
        arr = (ctypes.c_void_p * len(ps))(*[self._ptr(p) for p in ps])
        rc = self.lib.orc_fused_reduce_rmsnorm(
            self._ptr(y), self._ptr(res_out), self._ptr(q), self._ptr(scale), arr, len(ps),
            self._ptr(None if res_in is None else np.ascontiguousarray(res_in)),
            self._ptr(np.ascontiguousarray(w)), m, h, eps, int(bool(gemma)), int(bool(quant)),
            DTYPES[dtype])
        if rc != 0:
            raise ValueError(f"orc_fused_reduce_rmsnorm rejected its arguments ({rc})")
        return {"y": y, "res_out": res_out, "q": q, "scale": scale}

    def per_group_quant(self, y, group: int, dtype: str):
        """dynamic per-group FP8 e4m3 quantisation: returns (q [m, h], scale [m, h // group])."""
        y = np.ascontiguousarray(y)
        m, h = y.shape
        q = np.empty((m, h), np.uint8)
        scale = np.empty((m, h // group), np.float32)
        rc = self.lib.orc_per_group_quant(self._ptr(q), self._ptr(scale), self._ptr(y), m, h, group, DTYPES[dtype])
        if rc != 0:
            raise ValueError(f"orc_per_group_quant rejected its arguments ({rc})")
        return q, scale

    def fused_ex(self, partials: Sequence[np.ndarray], res_in, w, eps: float, gemma: bool, quant: bool,
                 dtype: str, skip_norm: bool = False, out_fp32: bool = False, group: int = 0) -> dict:
        """The whole path with the skip-norm, fp32-output and per-group-FP8 options.  Returns y
        (16-bit bits), y32 (float32, when out_fp32), res_out, q, scale ([m] per token, or
        [m, h // group] per group)."""
        ps = [np.ascontiguousarray(p) for p in partials]
        m, h = ps[0].shape
        y = np.empty((m, h), np.uint16)
        y32 = np.empty((m, h), np.float32) if out_fp32 else None
        res_out = np.empty((m, h), np.uint16)
        q = np.empty((m, h), np.uint8) if quant else None
        scale = (np.empty((m, h // group) if group else (m,), np.float32)) if quant else None
        arr = (ctypes.c_void_p * len(ps))(*[self._ptr(p) for p in ps])
        rc = self.lib.orc_fused_ex(
            self._ptr(y), self._ptr(y32), self._ptr(res_out), self._ptr(q), self._ptr(scale), arr, len(ps),
            self._ptr(None if res_in is None else np.ascontiguousarray(res_in)),
            self._ptr(None if w is None else np.ascontiguousarray(w)), m, h, eps, int(bool(gemma)),
            int(bool(quant)), int(bool(skip_norm)), int(group), DTYPES[dtype])
        if rc != 0:
            raise ValueError(f"orc_fused_ex rejected its arguments ({rc})")
        return {"y": y, "y32": y32, "res_out": res_out, "q": q, "scale": scale}


_default: Optional[Oracle] = None


def get() -> Oracle:
    """The oracle built from this directory's source (loaded once per process)."""
    global _default
    if _default is None:
        _default = Oracle()
    return _default
