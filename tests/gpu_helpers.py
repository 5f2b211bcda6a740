"""Comparison helpers for the GPU parity tests (no method arithmetic: only tolerances).

Bars (the fused path's contract):
  * reduced sum and residual_out: bit-exact with the oracle;
  * normalised output y: |y - y_oracle| <= 1 ulp of the element type at y_oracle;
  * FP8: codes within 1 code (adjacent in value order) and per-row scales within 1e-6
    relative, where the decision is taken on the same y on both sides (the oracle
    quantises the kernel's own rounded y); against the oracle's own y the scales agree
    exactly whenever the row's largest |y| agrees.
"""
from __future__ import annotations

import numpy as np
import torch

from tensor_all_reduce_gb300 import synth

TDT = {"bf16": torch.bfloat16, "fp16": torch.float16}


def decode(bits: np.ndarray, dtype: str) -> np.ndarray:
    return torch.from_numpy(np.ascontiguousarray(bits).view(np.int16)).view(TDT[dtype]).float().numpy()


def ulp(v: np.ndarray, dtype: str) -> np.ndarray:
    """Spacing of the 16-bit format at |v| (subnormal spacing below the normal range)."""
    a = np.abs(v.astype(np.float64))
    if dtype == "bf16":
        e = np.floor(np.log2(np.maximum(a, 2.0 ** -126)))
        return 2.0 ** (e - 7)
    e = np.floor(np.log2(np.maximum(a, 2.0 ** -14)))
    return 2.0 ** (e - 10)


def assert_bits_equal(got: np.ndarray, ref: np.ndarray, what: str):
    if not np.array_equal(got, ref):
        bad = np.argwhere(got != ref)
        i = tuple(bad[0])
        raise AssertionError(f"{what}: {len(bad)} mismatches, first at {i}: {got[i]:#x} vs {ref[i]:#x}")


def assert_y_within_ulp(got_bits: np.ndarray, ref_bits: np.ndarray, dtype: str, what: str = "y"):
    g = decode(got_bits, dtype).astype(np.float64)
    r = decode(ref_bits, dtype).astype(np.float64)
    err = np.abs(g - r)
    tol = ulp(r, dtype)
    if not np.all(err <= tol):
        i = np.unravel_index(np.argmax(err - tol), err.shape)
        raise AssertionError(f"{what}: {int((err > tol).sum())} elements beyond 1 ulp, worst at {i}: "
                             f"{g[i]!r} vs {r[i]!r}")


def code_ordinal(q: np.ndarray) -> np.ndarray:
    """Sign-magnitude E4M3 code -> position in value order (both zeros map to 0)."""
    mag = (q & 0x7F).astype(np.int32)
    return np.where(q & 0x80, -mag, mag)


def assert_fp8(orc, q: np.ndarray, scale: np.ndarray, y_gpu_bits: np.ndarray, dtype: str,
               ref: dict | None = None, what: str = "fp8"):
    # same-precision decision: quantise the kernel's own y with the oracle
    q_ref, s_ref = orc.per_token_quant(y_gpu_bits, dtype)
    rel = np.abs(scale.astype(np.float64) - s_ref) / np.maximum(np.abs(s_ref.astype(np.float64)), 1e-300)
    assert np.all(rel <= 1e-6), f"{what}: scale beyond 1e-6 relative (max {rel.max():.3g})"
    d = np.abs(code_ordinal(q) - code_ordinal(q_ref))
    assert d.max(initial=0) <= 1, f"{what}: codes differ by {d.max()} codes"
    if ref is not None:
        same = ref["scale"] == scale
        # rows whose largest |y| differs by the 1-ulp y tolerance are the only others allowed
        tol = 2.0 ** -7 if dtype == "bf16" else 2.0 ** -10
        r2 = np.abs(scale.astype(np.float64) - ref["scale"]) / np.maximum(ref["scale"].astype(np.float64), 1e-300)
        assert np.all(same | (r2 <= tol * 1.0001)), f"{what}: scale differs from the oracle beyond 1 ulp of amax"
        # every code within one code of the oracle's own (a scale off by one ulp of amax and a
        # y off by one ulp move a quotient by less than half an E4M3 step)
        d2 = np.abs(code_ordinal(q) - code_ordinal(ref["q"]))
        assert d2.max(initial=0) <= 1, f"{what}: codes differ from the oracle by {d2.max()} codes"
    return q_ref, s_ref


class Guarded:
    """A device buffer with sentinel guard regions on both sides, to catch stray writes."""

    GUARD = 512  # elements on each side (keeps 16-byte alignment for 1-, 2- and 4-byte types)

    def __init__(self, shape, dtype, device, offset_elems: int = 0):
        n = int(np.prod(shape)) if len(shape) else 1
        self.n, self.shape, self.off = n, shape, offset_elems
        self.buf = torch.empty(n + 2 * self.GUARD + offset_elems, dtype=dtype, device=device)
        raw = self.buf.view(torch.uint8)
        raw.fill_(0xA5)
        self.sentinel = raw.clone()
        start = self.GUARD + offset_elems
        self.t = self.buf[start:start + n].view(shape)

    def guards_intact(self) -> bool:
        es = self.buf.element_size()
        start = (self.GUARD + self.off) * es
        end = start + self.n * es
        raw = self.buf.view(torch.uint8)
        return bool(torch.equal(raw[:start], self.sentinel[:start]) and torch.equal(raw[end:], self.sentinel[end:]))


def to_dev(ts, dev):
    return [t.to(dev) for t in ts]


def bits_of(t):
    return synth.bits(t.cpu()) if t is not None else None
