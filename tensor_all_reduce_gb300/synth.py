"""Seeded synthetic inputs and the named workloads.

This module draws inputs only; it holds none of the reduce / norm / quant arithmetic, so
both the CUDA path's tests and the CPU oracle can take their inputs from it.

Recipes (the pages' workloads are TP ranks' partial activations of LLM hidden states;
no dataset is involved):
  * partials and residual ~ N(0, 1) drawn in fp32 from a CPU ``torch.Generator`` and cast
    to the element type, partials first in rank order, then the residual, then the weight;
  * weight = 1 + 0.1 * N(0, 1) for plain RMSNorm, 0.1 * N(0, 1) for gemma ((1 + w)
    weighting), cast to the element type;
  * integer-valued partials ((idx * (r + 1) + seed * (r + 3)) mod 31) - 15, whose sums are
    exact in every element type (page "[HIP] [Perf] Specialize partial tiles in two-stage
    custom all-reduce", the bench_allreduce_tail.py listing, input setter).
"""
from __future__ import annotations

from dataclasses import dataclass, field
from typing import Dict, List, Optional

import numpy as np
import torch

TORCH_DTYPES = {"bf16": torch.bfloat16, "fp16": torch.float16, "fp32": torch.float32}
ELEM_SIZE = {"bf16": 2, "fp16": 2, "fp32": 4}
EPS = 1e-6


def _normal(shape, dtype: str, gen: torch.Generator) -> torch.Tensor:
    return torch.randn(shape, generator=gen, dtype=torch.float32).to(TORCH_DTYPES[dtype])


def fused_inputs(n: int, m: int, h: int, dtype: str = "bf16", seed: int = 1234,
                 gemma: bool = False, residual: bool = True) -> Dict[str, object]:
    """N partials [m, h], residual [m, h] (or None) and weight [h] on the CPU."""
    gen = torch.Generator().manual_seed(seed)
    partials = [_normal((m, h), dtype, gen) for _ in range(n)]
    res = _normal((m, h), dtype, gen) if residual else None
    wn = torch.randn((h,), generator=gen, dtype=torch.float32)
    weight = (0.1 * wn if gemma else 1.0 + 0.1 * wn).to(TORCH_DTYPES[dtype])
    return {"partials": partials, "residual": res, "weight": weight}


def fill_fused_inputs_device(partials: List[torch.Tensor], residual: Optional[torch.Tensor], weight: torch.Tensor,
                             seed: int, gemma: bool = False) -> None:
    """The fused_inputs recipe drawn on the tensors' device (a generator of that device,
    seeded) into existing [m, h] partials, residual and [h] weight: for tests that need fresh
    inputs many times over without a host round trip."""
    gen = torch.Generator(device=weight.device).manual_seed(seed)
    for t in list(partials) + ([residual] if residual is not None else []):
        t.copy_(torch.randn(t.shape, generator=gen, dtype=torch.float32, device=t.device))
    wn = torch.randn(weight.shape, generator=gen, dtype=torch.float32, device=weight.device)
    weight.copy_(0.1 * wn if gemma else 1.0 + 0.1 * wn)


def fill_reduce_inputs_device(partials: List[torch.Tensor], seed: int) -> None:
    """N(0, 1) values drawn on the tensors' device into existing flat partials."""
    gen = torch.Generator(device=partials[0].device).manual_seed(seed)
    for t in partials:
        t.copy_(torch.randn(t.shape, generator=gen, dtype=torch.float32, device=t.device))


def reduce_inputs(n: int, numel: int, dtype: str, seed: int = 1234) -> List[torch.Tensor]:
    """N flat ~N(0, 1) partials on the CPU."""
    gen = torch.Generator().manual_seed(seed)
    return [_normal((numel,), dtype, gen) for _ in range(n)]


def integer_partials(n: int, numel: int, dtype: str, seed: int) -> List[torch.Tensor]:
    """Integer-valued partials in [-15, 15]; every partial sum is exact in every dtype."""
    idx = torch.arange(numel, dtype=torch.int64)
    return [(((idx * (r + 1) + seed * (r + 3)) % 31) - 15).to(TORCH_DTYPES[dtype]) for r in range(n)]


def bits(t: Optional[torch.Tensor]) -> Optional[np.ndarray]:
    """numpy view of a CPU tensor in the oracle's storage convention (uint16 bits / float32)."""
    if t is None:
        return None
    t = t.contiguous()
    if t.dtype in (torch.bfloat16, torch.float16):
        return t.view(torch.int16).numpy().view(np.uint16)
    if t.dtype == torch.float32:
        return t.numpy()
    if t.dtype == torch.uint8:
        return t.numpy()
    raise TypeError(f"unsupported dtype {t.dtype}")


@dataclass
class FusedWorkload:
    """One fused reduce + residual + RMSNorm (+ FP8) call shape."""
    name: str
    n: int
    m: int
    h: int
    dtype: str = "bf16"
    gemma: bool = False
    quant: bool = False
    mirror: bool = True          # write the normed output (the bf16 mirror when quant is on)
    residual: bool = True
    seed: int = 1234
    skip_norm: bool = False      # all-reduce (+ residual) + per-token FP8 without RMSNorm
    out_fp32: bool = False       # the normed output stored as fp32
    group: int = 0               # per-group FP8 with this many elements per group (0: per token)
    pad: int = 0                 # rows of inputs and outputs padded by this many elements (row stride h + pad)

    def inputs(self) -> Dict[str, object]:
        return fused_inputs(self.n, self.m, self.h, self.dtype, self.seed, self.gemma, self.residual)

    def algorithmic_bytes(self) -> int:
        """Bytes a call must move at minimum: N partial reads, residual read and res_out
        write, one weight read, the normed output, FP8 codes and per-row scales."""
        b = ELEM_SIZE[self.dtype]
        mh = self.m * self.h
        total = self.n * mh * b + (0 if self.skip_norm else self.h * b)
        if self.residual:
            total += 2 * mh * b
        if self.mirror or not self.quant:
            total += mh * (4 if self.out_fp32 else b)
        if self.quant:
            total += mh + 4 * (self.m * (self.h // self.group) if self.group else self.m)
        return total


@dataclass
class ReduceWorkload:
    name: str
    n: int
    numel: int
    dtype: str
    seed: int = 1234
    shape: tuple = field(default_factory=tuple)

    def algorithmic_bytes(self) -> int:
        return (self.n + 1) * self.numel * ELEM_SIZE[self.dtype]


# The five workload families, named by what they are.
def small_fused() -> List[FusedWorkload]:
    return [FusedWorkload("n4_m16_h6144_bf16_plain", 4, 16, 6144, seed=1234)]


def reduce_only() -> List[ReduceWorkload]:
    out = []
    for dt in ("fp16", "fp32"):
        for m in (1023, 1024, 1025):
            out.append(ReduceWorkload(f"reduce_n4_m{m}_h512_{dt}", 4, m * 512, dt, seed=1235,
                                      shape=(m, 512)))
    return out


def reduce_large() -> List[ReduceWorkload]:
    """Streaming sizes of the plain reduce (well above L2): 4 and 8 partials of 4096 x 6144
    bf16 (48 MiB each), and 4 of the same shape in fp32."""
    return [ReduceWorkload("reduce_n4_m4096_h6144_bf16", 4, 4096 * 6144, "bf16", seed=1238, shape=(4096, 6144)),
            ReduceWorkload("reduce_n8_m4096_h6144_bf16", 8, 4096 * 6144, "bf16", seed=1238, shape=(4096, 6144)),
            ReduceWorkload("reduce_n4_m4096_h6144_fp32", 4, 4096 * 6144, "fp32", seed=1238, shape=(4096, 6144))]


def decode_sweep() -> List[FusedWorkload]:
    return [FusedWorkload(f"n4_m{m}_h6144_bf16_decode", 4, m, 6144, seed=1236) for m in (1, 16, 64, 256)]


def gemma_fp8() -> List[FusedWorkload]:
    return [FusedWorkload(f"n4_m{m}_h{h}_bf16_gemma_fp8", 4, m, h, gemma=True, quant=True, mirror=True,
                          seed=1237) for (m, h) in ((1024, 6144), (2800, 6144), (1024, 7168))]


def large_m() -> List[FusedWorkload]:
    return [FusedWorkload("n8_m4096_h6144_bf16_plain", 8, 4096, 6144, seed=1238)]


def options() -> List[FusedWorkload]:
    """The fused path's further forms: all-reduce + residual + per-token FP8 without the norm,
    the normalised output in fp32, and per-group FP8 (groups of 128)."""
    return [FusedWorkload("n4_m2800_h6144_bf16_nonorm_fp8", 4, 2800, 6144, quant=True, mirror=False,
                          skip_norm=True, seed=1239),
            FusedWorkload("n4_m2800_h6144_bf16_f32out", 4, 2800, 6144, out_fp32=True, seed=1240),
            FusedWorkload("n4_m2800_h6144_bf16_gemma_fp8_group128", 4, 2800, 6144, gemma=True, quant=True,
                          mirror=True, group=128, seed=1241)]


def padded_rows() -> List[FusedWorkload]:
    """The every-step call on padded rows (row stride 6144 + 64 for inputs and outputs): the
    fused path on [m, h] views of wider buffers."""
    return [FusedWorkload("n4_m2800_h6144_bf16_gemma_fp8_pad64", 4, 2800, 6144, gemma=True, quant=True, mirror=True,
                          seed=1245, pad=64)]


def wide_rows() -> List[FusedWorkload]:
    """Rows longer than 8192 elements (hidden sizes of larger models), split over a cluster."""
    return [FusedWorkload("n4_m2048_h12288_bf16_gemma_fp8", 4, 2048, 12288, gemma=True, quant=True, mirror=True,
                          seed=1242),
            FusedWorkload("n4_m1536_h16384_bf16_gemma_fp8", 4, 1536, 16384, gemma=True, quant=True, mirror=True,
                          seed=1243)]


def mid_batch() -> List[FusedWorkload]:
    """512 x 8192 (a shape of the fused-kernel test list on page "[HIP] fix(custom-ar): gfx1250
    fused all-reduce + RMSNorm", Changes): 3-4 rows per SM on GB300, between the decode
    sizes and the long streaming batches."""
    return [FusedWorkload("n4_m512_h8192_bf16_gemma_fp8", 4, 512, 8192, gemma=True, quant=True, mirror=True,
                          seed=1244)]


def all_fused() -> List[FusedWorkload]:
    return small_fused() + decode_sweep() + gemma_fp8() + large_m() + wide_rows() + mid_batch()


def by_name(name: str):
    for w in all_fused() + options() + padded_rows() + reduce_only() + reduce_large():
        if w.name == name:
            return w
    raise KeyError(name)
