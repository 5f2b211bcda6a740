"""CUDA-graph capture of interleaved calls.

Adapted from the interleave test on page "[HIP] fix(custom-ar): gfx1250 fused all-reduce +
RMSNorm" (Changes / Test results: small and large fused calls mixed with plain
all-reduces on one communicator) and the graph checks on page "[HIP] [Perf] Specialize
partial tiles in two-stage custom all-reduce" (bench_allreduce_tail.py listing: outputs
poisoned with NaN before each replay, fresh inputs per sample, every captured call
checked).  One graph holds decode-sized and large fused calls, an FP8 call and plain
reduces on distinct buffers; each replay gets new inputs and is checked against the oracle.
"""
import numpy as np
import pytest
import torch

import tensor_all_reduce_gb300 as tar
from tensor_all_reduce_gb300 import synth

from gpu_helpers import assert_bits_equal, assert_fp8, assert_y_within_ulp, bits_of

pytestmark = pytest.mark.gpu


@pytest.fixture(scope="module")
def dev():
    if not torch.cuda.is_available():
        pytest.skip("no CUDA device")
    import __graft_entry__
    __graft_entry__.build()
    return torch.device("cuda", 0)


class FusedCall:
    def __init__(self, dev, n, m, h, dtype, gemma, quant):
        self.n, self.m, self.h, self.dtype, self.gemma, self.quant = n, m, h, dtype, gemma, quant
        t = torch.bfloat16 if dtype == "bf16" else torch.float16
        self.parts = [torch.empty((m, h), dtype=t, device=dev) for _ in range(n)]
        self.res = torch.empty((m, h), dtype=t, device=dev)
        self.w = torch.empty((h,), dtype=t, device=dev)
        self.out = torch.empty((m, h), dtype=t, device=dev)
        self.ro = torch.empty((m, h), dtype=t, device=dev)
        self.q = torch.empty((m, h), dtype=torch.uint8, device=dev) if quant else None
        self.sc = torch.empty((m,), dtype=torch.float32, device=dev) if quant else None

    def load(self, seed):
        self.inp = synth.fused_inputs(self.n, self.m, self.h, self.dtype, seed=seed, gemma=self.gemma)
        for d, s in zip(self.parts, self.inp["partials"]):
            d.copy_(s)
        self.res.copy_(self.inp["residual"])
        self.w.copy_(self.inp["weight"])

    def poison(self):
        self.out.fill_(float("nan"))
        self.ro.fill_(float("nan"))
        if self.quant:
            self.q.fill_(0x7F)
            self.sc.fill_(float("nan"))

    def call(self, ctx):
        ctx.fused_reduce_rmsnorm(self.parts, self.res, self.w, eps=1e-6, gemma=self.gemma, quant=self.quant,
                                 out=self.out, residual_out=self.ro, q_out=self.q, scale_out=self.sc)

    def check(self, orc):
        ref = orc.fused([synth.bits(p) for p in self.inp["partials"]], synth.bits(self.inp["residual"]),
                        synth.bits(self.inp["weight"]), 1e-6, self.gemma, self.quant, self.dtype)
        assert_bits_equal(bits_of(self.ro), ref["res_out"], "graph residual_out")
        y = bits_of(self.out)
        assert_y_within_ulp(y, ref["y"], self.dtype)
        if self.quant:
            assert_fp8(orc, self.q.cpu().numpy(), self.sc.cpu().numpy(), y, self.dtype, ref)


class ReduceCall:
    def __init__(self, dev, n, numel, dtype):
        self.n, self.numel, self.dtype = n, numel, dtype
        t = {"bf16": torch.bfloat16, "fp16": torch.float16, "fp32": torch.float32}[dtype]
        self.parts = [torch.empty((numel,), dtype=t, device=dev) for _ in range(n)]
        self.out = torch.empty((numel,), dtype=t, device=dev)

    def load(self, seed):
        self.inp = synth.reduce_inputs(self.n, self.numel, self.dtype, seed=seed)
        for d, s in zip(self.parts, self.inp):
            d.copy_(s)

    def poison(self):
        self.out.fill_(float("nan"))

    def call(self, ctx):
        ctx.reduce_sum(self.parts, out=self.out)

    def check(self, orc):
        ref = orc.reduce_sum([synth.bits(p) for p in self.inp], self.dtype)
        assert_bits_equal(synth.bits(self.out.cpu()), ref, "graph reduce")


def test_graph_interleaved_calls(dev, orc):
    calls = [
        FusedCall(dev, 4, 16, 6144, "bf16", False, False),     # decode-sized: one staged CTA per row
        ReduceCall(dev, 4, 1025 * 512, "fp16"),                 # tail path
        FusedCall(dev, 4, 384, 6144, "bf16", True, True),       # FP8 epilogue, persistent staged
        FusedCall(dev, 4, 1, 6144, "bf16", False, False),      # one token
        ReduceCall(dev, 4, 1024 * 512, "fp32"),
        FusedCall(dev, 8, 1024, 6144, "bf16", False, False),    # large M
        FusedCall(dev, 4, 7, 6145, "fp16", True, True),         # tail hidden size: element-wise form
        FusedCall(dev, 4, 64, 12288, "bf16", True, True),       # long rows: staged cluster form
        ReduceCall(dev, 5, 8192 * 16 * 152, "bf16"),            # large 16-bit sum: staged rows
    ]
    with tar.Context(0) as ctx:
        for i, c in enumerate(calls):
            c.load(seed=i)
        # eager warm-up, then capture on a side stream
        ran = []
        for c in calls:
            c.call(ctx)
            ran.append(ctx.last_variant)
        torch.cuda.synchronize()
        assert ran[0] == "fused_staged" and "scalar" in ran[6] and ran[7] == "fused_staged_cluster", ran
        if ctx.info(tar.AR_INFO_SM_COUNT) <= 152:
            assert ran[8] == "reduce_staged", ran
        g = torch.cuda.CUDAGraph()
        s = torch.cuda.Stream()
        s.wait_stream(torch.cuda.current_stream())
        with torch.cuda.graph(g, stream=s):
            for c in calls:
                c.call(ctx)
        torch.cuda.current_stream().wait_stream(s)
        torch.cuda.synchronize()
        for rep in range(12):
            for i, c in enumerate(calls):
                c.load(seed=1000 * (rep + 1) + i)
                c.poison()
            g.replay()
            torch.cuda.synchronize()
            for c in calls:
                c.check(orc)


# ---------------------------------------------------------------------------
# interleave stress: the mixed graph replayed 300 times with fresh inputs
# ---------------------------------------------------------------------------

class StressFused(FusedCall):
    """Inputs drawn on the device every replay; checked in full (check_rows None) or on
    `check_rows` sampled rows, plus a device-side scan that no NaN poison survived."""

    def __init__(self, dev, n, m, h, dtype, gemma, quant, check_rows=None):
        super().__init__(dev, n, m, h, dtype, gemma, quant)
        self.check_rows = check_rows

    def load(self, seed):
        synth.fill_fused_inputs_device(self.parts, self.res, self.w, seed, self.gemma)

    def check(self, orc, rng):
        assert not bool(torch.isnan(self.out).any()) and not bool(torch.isnan(self.ro).any()), "poison left"
        if self.quant:
            assert not bool((self.q == 0x7F).any()) and not bool(torch.isnan(self.sc).any()), "poison left"
        rows = (np.arange(self.m) if self.check_rows is None
                else np.sort(rng.choice(self.m, self.check_rows, replace=False)))
        idx = torch.from_numpy(rows).to(self.out.device)
        take = lambda t: synth.bits(t.index_select(0, idx).cpu())
        ref = orc.fused([take(p) for p in self.parts], take(self.res), synth.bits(self.w.cpu()), 1e-6, self.gemma,
                        self.quant, self.dtype)
        assert_bits_equal(take(self.ro), ref["res_out"], "graph residual_out")
        y = take(self.out)
        assert_y_within_ulp(y, ref["y"], self.dtype)
        if self.quant:
            assert_fp8(orc, self.q.index_select(0, idx).cpu().numpy(), self.sc.index_select(0, idx).cpu().numpy(),
                       y, self.dtype, ref)


class StressReduce(ReduceCall):
    """Plain reduce with device-drawn inputs; checked in full or on `check_runs` sampled
    contiguous runs of 4096 elements."""

    def __init__(self, dev, n, numel, dtype, check_runs=None):
        super().__init__(dev, n, numel, dtype)
        self.check_runs = check_runs

    def load(self, seed):
        synth.fill_reduce_inputs_device(self.parts, seed)

    def check(self, orc, rng):
        assert not bool(torch.isnan(self.out).any()), "poison left"
        if self.check_runs is None:
            sl = [slice(0, self.numel)]
        else:
            starts = rng.choice(self.numel // 4096, self.check_runs, replace=False) * 4096
            sl = [slice(int(a), int(a) + 4096) for a in starts]
        for s in sl:
            ref = orc.reduce_sum([synth.bits(p[s].cpu()) for p in self.parts], self.dtype)
            assert_bits_equal(synth.bits(self.out[s].cpu()), ref, "graph reduce")


def test_graph_interleaved_300_replays(dev, orc):
    """The mixed graph of decode-sized, large, FP8, element-wise, cluster and plain-reduce calls
    replayed 300 times; before every replay each call gets fresh inputs and NaN-poisoned
    outputs.  Small calls are checked in full on every replay, large ones on sampled rows."""
    calls = [
        StressFused(dev, 4, 16, 6144, "bf16", False, False),
        StressReduce(dev, 4, 1025 * 512, "fp16"),
        StressFused(dev, 4, 384, 6144, "bf16", True, True, check_rows=3),
        StressFused(dev, 4, 1, 6144, "bf16", False, False),
        StressReduce(dev, 4, 1024 * 512, "fp32"),
        StressFused(dev, 8, 1024, 6144, "bf16", False, False, check_rows=2),
        StressFused(dev, 4, 7, 6145, "fp16", True, True),
        StressFused(dev, 4, 64, 12288, "bf16", True, True, check_rows=2),
        StressReduce(dev, 5, 8192 * 16 * 152, "bf16", check_runs=2),
        StressFused(dev, 2, 3, 2880, "fp16", False, True),      # short fp16 rows with FP8
    ]
    rng = np.random.default_rng(2024)
    with tar.Context(0) as ctx:
        for i, c in enumerate(calls):
            c.load(seed=i)
            c.call(ctx)
        torch.cuda.synchronize()
        g = torch.cuda.CUDAGraph()
        s = torch.cuda.Stream()
        s.wait_stream(torch.cuda.current_stream())
        with torch.cuda.graph(g, stream=s):
            for c in calls:
                c.call(ctx)
        torch.cuda.current_stream().wait_stream(s)
        torch.cuda.synchronize()
        for rep in range(300):
            for i, c in enumerate(calls):
                c.load(seed=7919 * (rep + 1) + i)
                c.poison()
            g.replay()
            torch.cuda.synchronize()
            for c in calls:
                c.check(orc, rng)
        assert ctx.device_status() == 0
