"""GPU parity of ar_fused_reduce_rmsnorm_batch: several independent fused calls in one
launch, each checked against the oracle with the single-call bars (residual_out bit-exact,
y within one ulp, FP8 codes and scales exact given the kernel's own y)."""
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


@pytest.fixture(scope="module")
def ctx(dev):
    c = tar.Context(0)
    yield c
    c.close()


def _make(dev, shapes, dtype, n, gemma, quant, residual=True, seed0=0):
    calls, inps = [], []
    for i, (m, h) in enumerate(shapes):
        inp = synth.fused_inputs(n, m, h, dtype, seed=seed0 + 31 * i + m + h, gemma=gemma, residual=residual)
        inps.append(inp)
        calls.append({"partials": [p.to(dev) for p in inp["partials"]],
                      "residual": inp["residual"].to(dev) if residual else None,
                      "weight": inp["weight"].to(dev), "eps": 1e-6 * (1 + i), "gemma": gemma, "quant": quant})
    return calls, inps


def _check(orc, outs, inps, calls, dtype, quant):
    for (y, ro, q, sc), inp, c in zip(outs, inps, calls):
        ref = orc.fused([synth.bits(p) for p in inp["partials"]], synth.bits(inp["residual"]),
                        synth.bits(inp["weight"]), c["eps"], c["gemma"], quant, dtype)
        assert_bits_equal(bits_of(ro), ref["res_out"], "residual_out")
        yb = bits_of(y)
        assert_y_within_ulp(yb, ref["y"], dtype)
        if quant:
            assert_fp8(orc, q.cpu().numpy(), sc.cpu().numpy(), yb, dtype, ref)


DECODE = [(1, 6144), (16, 6144), (3, 4096), (64, 2880), (7, 7168), (1, 8192)]


@pytest.mark.parametrize("dtype", ["bf16", "fp16"])
@pytest.mark.parametrize("quant", [False, True])
@pytest.mark.parametrize("n", [1, 4, 8])
def test_batch_of_decode_calls(ctx, dev, orc, dtype, quant, n):
    calls, inps = _make(dev, DECODE, dtype, n, gemma=quant, quant=quant)
    outs = ctx.fused_reduce_rmsnorm_batch(calls)
    torch.cuda.synchronize()
    assert ctx.last_variant == "fused_batch"
    _check(orc, outs, inps, calls, dtype, quant)
    assert ctx.device_status() == 0


def test_batch_mixed_sizes_and_options(ctx, dev, orc):
    shapes = [(300, 6144), (1, 6144), (1000, 2048), (0, 6144), (33, 4096)]
    calls, inps = _make(dev, shapes, "bf16", 4, gemma=False, quant=False, residual=False)
    outs = ctx.fused_reduce_rmsnorm_batch(calls)
    torch.cuda.synchronize()
    assert ctx.last_variant == "fused_batch"
    for (y, ro, _, _), inp, c, (m, h) in zip(outs, inps, calls, shapes):
        if m == 0:
            continue
        ref = orc.fused([synth.bits(p) for p in inp["partials"]], None, synth.bits(inp["weight"]), c["eps"], False,
                        False, "bf16")
        assert_bits_equal(bits_of(ro), ref["res_out"], "residual_out")
        assert_y_within_ulp(bits_of(y), ref["y"], "bf16")


def test_batch_skip_norm_and_fp32_out(ctx, dev, orc):
    calls, inps = _make(dev, DECODE[:4], "bf16", 4, gemma=False, quant=True)
    for c in calls:
        c["skip_norm"] = True
        c["weight"] = None
    outs = ctx.fused_reduce_rmsnorm_batch(calls)
    torch.cuda.synchronize()
    for (y, ro, q, sc), inp in zip(outs, inps):
        ref = orc.fused_ex([synth.bits(p) for p in inp["partials"]], synth.bits(inp["residual"]), None, 0.0, False,
                           True, "bf16", skip_norm=True)
        assert_bits_equal(bits_of(y), ref["y"], "z")
        assert np.array_equal(q.cpu().numpy(), ref["q"]) and np.array_equal(sc.cpu().numpy(), ref["scale"])
    calls, inps = _make(dev, DECODE[:4], "bf16", 4, gemma=True, quant=False)
    for c in calls:
        c["out_fp32"] = True
    outs = ctx.fused_reduce_rmsnorm_batch(calls)
    torch.cuda.synchronize()
    for (y, ro, _, _), inp, c in zip(outs, inps, calls):
        ref = orc.fused_ex([synth.bits(p) for p in inp["partials"]], synth.bits(inp["residual"]),
                           synth.bits(inp["weight"]), c["eps"], True, False, "bf16", out_fp32=True)
        g, r = y.cpu().numpy().astype(np.float64), ref["y32"].astype(np.float64)
        assert np.all(np.abs(g - r) <= 2.0 ** -19 * np.abs(r) + 1e-30)


def test_batch_falls_back_to_separate_launches(ctx, dev, orc):
    calls, inps = _make(dev, [(4, 6144), (5, 6145)], "bf16", 2, gemma=False, quant=False)
    outs = ctx.fused_reduce_rmsnorm_batch(calls)
    torch.cuda.synchronize()
    assert ctx.last_variant == "fused_batch_sequential"
    _check(orc, outs, inps, calls, "bf16", False)


def test_batch_in_a_cuda_graph(ctx, dev, orc):
    calls, inps = _make(dev, DECODE, "bf16", 4, gemma=True, quant=True)
    outs = ctx.fused_reduce_rmsnorm_batch(calls)
    torch.cuda.synchronize()
    g = torch.cuda.CUDAGraph()
    s = torch.cuda.Stream()
    s.wait_stream(torch.cuda.current_stream())
    with torch.cuda.graph(g, stream=s):
        for c, (y, ro, q, sc) in zip(calls, outs):
            c.update(out=y, residual_out=ro, q_out=q, scale_out=sc)
        ctx.fused_reduce_rmsnorm_batch(calls)
    torch.cuda.current_stream().wait_stream(s)
    for rep in range(3):
        new = []
        for i, c in enumerate(calls):
            m, h = c["partials"][0].shape
            inp = synth.fused_inputs(4, m, h, "bf16", seed=7000 + 10 * rep + i, gemma=True)
            for d, src in zip(c["partials"], inp["partials"]):
                d.copy_(src)
            c["residual"].copy_(inp["residual"])
            c["weight"].copy_(inp["weight"])
            new.append(inp)
        for y, ro, q, sc in outs:
            y.fill_(float("nan"))
            ro.fill_(float("nan"))
        g.replay()
        torch.cuda.synchronize()
        _check(orc, outs, new, calls, "bf16", True)
