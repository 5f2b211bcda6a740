"""Padded (row-strided) inputs and outputs: the fused path on [m, h] views of wider
buffers (page "[HIP] fix(custom-ar): gfx1250 fused all-reduce + RMSNorm", Changes, sends
padded or strided rows to the unfused path; here they stay fused).  Results must equal the
oracle's on the contiguous copies, and the padding columns must stay untouched."""
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


VARIANTS = {"auto": {}, "row": {tar.AR_OPT_FORCE_VARIANT: tar.VARIANT_ROW},
            "staged": {tar.AR_OPT_FORCE_VARIANT: tar.VARIANT_STAGED},
            "cluster4": {tar.AR_OPT_CLUSTER_SIZE: 4},
            "scalar": {tar.AR_OPT_FORCE_VARIANT: tar.VARIANT_SCALAR}}


def _set(ctx, opts):
    for o in range(5):
        ctx.set_option(o, 0)
    for k, v in opts.items():
        ctx.set_option(k, v)


def _padded(t, pad, dev, fill=None):
    """A device [m, h] view, with row stride h + pad, of a wider buffer holding t (or `fill`)."""
    m, h = t.shape
    big = torch.empty((m, h + pad), dtype=t.dtype, device=dev)
    if fill is None:
        big.view(torch.uint8).fill_(0x5A)
        big[:, :h].copy_(t)
    else:
        big.view(torch.uint8).fill_(fill)
    return big, big[:, :h]


def _pads_intact(big, h, fill):
    raw = big[:, h:].contiguous().view(torch.uint8)
    return bool((raw == fill).all().item()) if raw.numel() else True


@pytest.mark.parametrize("variant", list(VARIANTS))
@pytest.mark.parametrize("pad_in,pad_out", [(8, 16), (64, 0), (0, 24), (3, 5)])
@pytest.mark.parametrize("quant", [False, True])
def test_padded_rows(ctx, dev, orc, variant, pad_in, pad_out, quant):
    _set(ctx, VARIANTS[variant])
    for m, h in ((700, 4096), (6, 2048)):
        inp = synth.fused_inputs(4, m, h, "bf16", seed=m + pad_in + 7 * pad_out, gemma=quant)
        parts = [_padded(p, pad_in, dev)[1] for p in inp["partials"]]
        res = _padded(inp["residual"], pad_in, dev)[1]
        y_big, y = _padded(inp["residual"], pad_out, dev, fill=0xA5)
        ro_big, ro = _padded(inp["residual"], pad_out, dev, fill=0xA5)
        q_big = torch.full((m, h + pad_out), 0xA5, dtype=torch.uint8, device=dev) if quant else None
        q = q_big[:, :h] if quant else None
        if variant == "staged" and (pad_in % 8 or pad_out % 8):
            # the staged kernel copies whole 16-byte-aligned rows: forcing it on unaligned
            # strides is refused before anything is launched
            with pytest.raises(tar.ArError) as e:
                ctx.fused_reduce_rmsnorm(parts, res, inp["weight"].to(dev), eps=1e-6, gemma=quant, quant=quant,
                                         out=y, residual_out=ro, q_out=q)
            assert e.value.status == tar.AR_ERR_UNSUPPORTED
            continue
        ctx.fused_reduce_rmsnorm(parts, res, inp["weight"].to(dev), eps=1e-6, gemma=quant, quant=quant, out=y,
                                 residual_out=ro, q_out=q)
        torch.cuda.synchronize()
        if (pad_in % 8) or (pad_out % 8) or variant == "scalar":
            assert "scalar" in ctx.last_variant
        for big in (y_big, ro_big) + ((q_big,) if quant else ()):
            assert _pads_intact(big, h, 0xA5), "a kernel wrote into the row padding"
        ref = orc.fused([synth.bits(p) for p in inp["partials"]], synth.bits(inp["residual"]),
                        synth.bits(inp["weight"]), 1e-6, quant, quant, "bf16")
        assert_bits_equal(bits_of(ro.contiguous()), ref["res_out"], "residual_out")
        yb = bits_of(y.contiguous())
        assert_y_within_ulp(yb, ref["y"], "bf16")


@pytest.mark.parametrize("variant", ["auto", "staged", "row"])
def test_padded_rows_fp8_codes(ctx, dev, orc, variant):
    _set(ctx, VARIANTS[variant])
    m, h, pad = 900, 6144, 64
    inp = synth.fused_inputs(4, m, h, "bf16", seed=3, gemma=True)
    parts = [_padded(p, pad, dev)[1] for p in inp["partials"]]
    res = _padded(inp["residual"], pad, dev)[1]
    y = _padded(inp["residual"], pad, dev, fill=0)[1]
    ro = _padded(inp["residual"], pad, dev, fill=0)[1]
    q = torch.zeros((m, h + pad), dtype=torch.uint8, device=dev)[:, :h]
    _, _, _, sc = ctx.fused_reduce_rmsnorm(parts, res, inp["weight"].to(dev), eps=1e-6, gemma=True, quant=True, out=y,
                                           residual_out=ro, q_out=q)
    torch.cuda.synchronize()
    ref = orc.fused([synth.bits(p) for p in inp["partials"]], synth.bits(inp["residual"]), synth.bits(inp["weight"]),
                    1e-6, True, True, "bf16")
    yb = bits_of(y.contiguous())
    assert_y_within_ulp(yb, ref["y"], "bf16")
    assert_fp8(orc, q.contiguous().cpu().numpy(), sc.cpu().numpy(), yb, "bf16", ref)


def test_padded_rows_batched(ctx, dev, orc):
    _set(ctx, {})
    calls, inps = [], []
    for i, (m, h) in enumerate(((16, 6144), (3, 4096))):
        inp = synth.fused_inputs(4, m, h, "bf16", seed=80 + i)
        inps.append(inp)
        calls.append({"partials": [_padded(p, 8 * (i + 1), dev)[1] for p in inp["partials"]],
                      "residual": _padded(inp["residual"], 8 * (i + 1), dev)[1], "weight": inp["weight"].to(dev),
                      "out": _padded(inp["residual"], 16, dev, fill=0)[1],
                      "residual_out": _padded(inp["residual"], 16, dev, fill=0)[1]})
    outs = ctx.fused_reduce_rmsnorm_batch(calls)
    torch.cuda.synchronize()
    assert ctx.last_variant == "fused_batch"
    for (y, ro, _, _), inp in zip(outs, inps):
        ref = orc.fused([synth.bits(p) for p in inp["partials"]], synth.bits(inp["residual"]),
                        synth.bits(inp["weight"]), 1e-6, False, False, "bf16")
        assert_bits_equal(bits_of(ro.contiguous()), ref["res_out"], "residual_out")
        assert_y_within_ulp(bits_of(y.contiguous()), ref["y"], "bf16")


@pytest.mark.parametrize("wl", synth.padded_rows(), ids=[w.name for w in synth.padded_rows()])
def test_padded_workload_full_size(ctx, dev, orc, wl):
    """The benchmark's padded-row workload at its full size, in the launch configuration the
    benchmark times (the automatic choice): the staged kernel on [m, h] views of [m, h + pad]
    buffers, checked against the oracle on the contiguous copies."""
    _set(ctx, {})
    inp = wl.inputs()
    m, h = wl.m, wl.h
    parts = [_padded(p, wl.pad, dev)[1] for p in inp["partials"]]
    res = _padded(inp["residual"], wl.pad, dev)[1]
    y_big, y = _padded(inp["residual"], wl.pad, dev, fill=0xA5)
    ro_big, ro = _padded(inp["residual"], wl.pad, dev, fill=0xA5)
    q_big = torch.full((m, h + wl.pad), 0xA5, dtype=torch.uint8, device=dev)
    sc = torch.empty((m,), dtype=torch.float32, device=dev)
    ctx.fused_reduce_rmsnorm(parts, res, inp["weight"].to(dev), eps=1e-6, gemma=wl.gemma, quant=wl.quant, out=y,
                             residual_out=ro, q_out=q_big[:, :h], scale_out=sc)
    torch.cuda.synchronize()
    assert ctx.last_variant == "fused_staged"
    ref = orc.fused([synth.bits(p) for p in inp["partials"]], synth.bits(inp["residual"]), synth.bits(inp["weight"]),
                    1e-6, wl.gemma, wl.quant, "bf16")
    assert_bits_equal(bits_of(ro), ref["res_out"], "residual_out")
    yb = bits_of(y)
    assert_y_within_ulp(yb, ref["y"], "bf16")
    assert_fp8(orc, q_big[:, :h].cpu().numpy(), sc.cpu().numpy(), yb, "bf16", ref)
    assert _pads_intact(y_big, h, 0xA5) and _pads_intact(ro_big, h, 0xA5) and _pads_intact(q_big, h, 0xA5)
