"""The fused call over host memory (ar_fused_reduce_rmsnorm_host): partials, residual,
weight and outputs in page-locked host memory, read and written by the kernel directly
across the CPU-GPU link.  Same bar as the device form against the oracle: residual_out
bit-exact, y within one 16-bit ulp, FP8 codes and scales exact on the kernel's own y.
Guard bytes around the host outputs must stay untouched, buffers may mix host and device
memory, and pageable host memory is refused without a launch."""
import ctypes

import numpy as np
import pytest
import torch

import tensor_all_reduce_gb300 as tar
from tensor_all_reduce_gb300 import synth

from gpu_helpers import assert_bits_equal, assert_fp8, assert_y_within_ulp, bits_of

pytestmark = pytest.mark.gpu

HOST_VARIANTS = ("fused_row_vec", "fused_cluster_vec", "fused_scalar", "fused_cluster_scalar")


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


def _reset(ctx):
    for o in range(5):
        ctx.set_option(o, 0)


def _pinned(t):
    return None if t is None else t.pin_memory()


def _guarded_pinned(shape, dtype, guard=4096):
    """A pinned [shape] view inside a larger pinned buffer whose both ends hold 0xA5 bytes."""
    n = int(np.prod(shape))
    buf = torch.empty(n + 2 * guard, dtype=dtype, pin_memory=True)
    buf.view(torch.uint8).fill_(0xA5)
    return buf, buf[guard:guard + n].view(shape)


def _guards_intact(buf, n, guard=4096):
    raw = buf.view(torch.uint8)
    es = buf.element_size()
    return bool((raw[:guard * es] == 0xA5).all()) and bool((raw[(guard + n) * es:] == 0xA5).all())


@pytest.mark.parametrize("dtype", ["bf16", "fp16"])
@pytest.mark.parametrize("m,h", [(1, 6144), (300, 6144), (37, 1001), (2800, 6144)])
@pytest.mark.parametrize("quant", [False, True])
def test_host_buffers_match_oracle(ctx, dev, orc, dtype, m, h, quant):
    _reset(ctx)
    inp = synth.fused_inputs(4, m, h, dtype, seed=m + h + quant, gemma=quant)
    parts = [_pinned(p) for p in inp["partials"]]
    res, w = _pinned(inp["residual"]), _pinned(inp["weight"])
    t = synth.TORCH_DTYPES[dtype]
    y_buf, y = _guarded_pinned((m, h), t)
    ro_buf, ro = _guarded_pinned((m, h), t)
    q_buf, q = _guarded_pinned((m, h), torch.uint8) if quant else (None, None)
    y, ro, q, sc = ctx.fused_reduce_rmsnorm_host(parts, res, w, eps=1e-6, gemma=quant, quant=quant, out=y,
                                                 residual_out=ro, q_out=q)
    torch.cuda.synchronize()
    assert ctx.last_variant in HOST_VARIANTS
    assert not y.is_cuda and not ro.is_cuda and (not quant or (not sc.is_cuda and sc.is_pinned()))
    for buf in (y_buf, ro_buf) + ((q_buf,) if quant else ()):
        assert _guards_intact(buf, m * h), "the kernel wrote outside an output in host memory"
    ref = orc.fused([synth.bits(p) for p in inp["partials"]], synth.bits(inp["residual"]),
                    synth.bits(inp["weight"]), 1e-6, quant, quant, dtype)
    assert_bits_equal(bits_of(ro), ref["res_out"], "residual_out")
    yb = bits_of(y)
    assert_y_within_ulp(yb, ref["y"], dtype)
    if quant:
        assert_fp8(orc, q.numpy(), sc.numpy(), yb, dtype, ref)


def test_host_and_device_buffers_mixed(ctx, dev, orc):
    _reset(ctx)
    m, h = 500, 4096
    inp = synth.fused_inputs(3, m, h, "bf16", seed=11, gemma=True)
    parts = [_pinned(inp["partials"][0]), inp["partials"][1].to(dev), _pinned(inp["partials"][2])]
    res, w = inp["residual"].to(dev), inp["weight"].to(dev)
    ro = torch.empty((m, h), dtype=torch.bfloat16, device=dev)
    y, ro, q, sc = ctx.fused_reduce_rmsnorm_host(parts, res, w, eps=1e-6, gemma=True, quant=True, residual_out=ro)
    torch.cuda.synchronize()
    assert ro.is_cuda and y.is_pinned() and q.is_pinned()
    ref = orc.fused([synth.bits(p) for p in inp["partials"]], synth.bits(inp["residual"]),
                    synth.bits(inp["weight"]), 1e-6, True, True, "bf16")
    assert_bits_equal(bits_of(ro), ref["res_out"], "residual_out")
    yb = bits_of(y)
    assert_y_within_ulp(yb, ref["y"], "bf16")
    assert_fp8(orc, q.numpy(), sc.numpy(), yb, "bf16", ref)


@pytest.mark.parametrize("group", [32, 128])
def test_host_per_group_fp8(ctx, dev, orc, group):
    _reset(ctx)
    m, h = 200, 6144
    inp = synth.fused_inputs(4, m, h, "bf16", seed=group, gemma=True)
    parts = [_pinned(p) for p in inp["partials"]]
    y, ro, q, sc = ctx.fused_reduce_rmsnorm_host(parts, _pinned(inp["residual"]), _pinned(inp["weight"]), eps=1e-6,
                                                 gemma=True, quant=True, group_size=group)
    torch.cuda.synchronize()
    assert sc.shape == (m, h // group)
    ref = orc.fused_ex([synth.bits(p) for p in inp["partials"]], synth.bits(inp["residual"]),
                       synth.bits(inp["weight"]), 1e-6, True, True, "bf16", group=group)
    assert_bits_equal(bits_of(ro), ref["res_out"], "residual_out")
    yb = bits_of(y)
    assert_y_within_ulp(yb, ref["y"], "bf16")
    q_ref, s_ref = orc.per_group_quant(yb, group, "bf16")   # the same decision on the kernel's y
    assert np.array_equal(sc.numpy().view(np.uint32), s_ref.view(np.uint32))
    assert np.array_equal(q.numpy(), q_ref)


def test_host_skip_norm_fp8_and_fp32_output(ctx, dev, orc):
    _reset(ctx)
    m, h = 300, 2880
    inp = synth.fused_inputs(4, m, h, "fp16", seed=5)
    parts = [_pinned(p) for p in inp["partials"]]
    y, ro, q, sc = ctx.fused_reduce_rmsnorm_host(parts, _pinned(inp["residual"]), None, eps=1e-6, quant=True,
                                                 skip_norm=True)
    torch.cuda.synchronize()
    ref = orc.fused_ex([synth.bits(p) for p in inp["partials"]], synth.bits(inp["residual"]), None, 0.0, False,
                       True, "fp16", skip_norm=True)
    assert_bits_equal(bits_of(ro), ref["res_out"], "residual_out")
    assert_bits_equal(bits_of(y), ref["y"], "output (= z)")
    assert np.array_equal(sc.numpy().view(np.uint32), ref["scale"].view(np.uint32))
    assert np.array_equal(q.numpy(), ref["q"])
    # fp32 output: the normalised row before rounding, against the oracle's binary32 value
    y32, ro, _, _ = ctx.fused_reduce_rmsnorm_host(parts, _pinned(inp["residual"]), _pinned(inp["weight"]), eps=1e-6,
                                                  out_fp32=True)
    torch.cuda.synchronize()
    ref = orc.fused_ex([synth.bits(p) for p in inp["partials"]], synth.bits(inp["residual"]),
                       synth.bits(inp["weight"]), 1e-6, False, False, "fp16", out_fp32=True)
    assert y32.dtype == torch.float32
    g, r = y32.numpy().astype(np.float64), ref["y32"].astype(np.float64)
    assert np.all(np.abs(g - r) <= 2.0 ** -19 * np.abs(r) + 1e-30)


def test_host_padded_rows(ctx, dev, orc):
    _reset(ctx)
    m, h, pad = 120, 4096, 64
    inp = synth.fused_inputs(4, m, h, "bf16", seed=21)

    def padded(t):
        big = torch.zeros((m, h + pad), dtype=t.dtype, pin_memory=True)
        big[:, :h].copy_(t)
        return big[:, :h]

    parts = [padded(p) for p in inp["partials"]]
    y_big = torch.full((m, h + pad), 7.0, dtype=torch.bfloat16, pin_memory=True)
    ro_big = torch.full((m, h + pad), 7.0, dtype=torch.bfloat16, pin_memory=True)
    ctx.fused_reduce_rmsnorm_host(parts, padded(inp["residual"]), _pinned(inp["weight"]), eps=1e-6,
                                  out=y_big[:, :h], residual_out=ro_big[:, :h])
    torch.cuda.synchronize()
    assert bool((y_big[:, h:] == 7.0).all()) and bool((ro_big[:, h:] == 7.0).all())
    ref = orc.fused([synth.bits(p) for p in inp["partials"]], synth.bits(inp["residual"]),
                    synth.bits(inp["weight"]), 1e-6, False, False, "bf16")
    assert_bits_equal(bits_of(ro_big[:, :h].contiguous()), ref["res_out"], "residual_out")
    assert_y_within_ulp(bits_of(y_big[:, :h].contiguous()), ref["y"], "bf16")


def test_host_call_in_cuda_graph(ctx, dev, orc):
    _reset(ctx)
    m, h = 256, 6144
    inp = synth.fused_inputs(4, m, h, "bf16", seed=31, gemma=True)
    parts = [_pinned(p) for p in inp["partials"]]
    res, w = _pinned(inp["residual"]), _pinned(inp["weight"])
    y = torch.empty((m, h), dtype=torch.bfloat16, pin_memory=True)
    ro = torch.empty((m, h), dtype=torch.bfloat16, pin_memory=True)
    q = torch.empty((m, h), dtype=torch.uint8, pin_memory=True)
    sc = torch.empty((m,), dtype=torch.float32, pin_memory=True)

    def call():
        ctx.fused_reduce_rmsnorm_host(parts, res, w, eps=1e-6, gemma=True, quant=True, out=y, residual_out=ro,
                                      q_out=q, scale_out=sc)

    call()
    torch.cuda.synchronize()
    g = torch.cuda.CUDAGraph()
    s = torch.cuda.Stream()
    s.wait_stream(torch.cuda.current_stream())
    with torch.cuda.graph(g, stream=s):
        call()
    torch.cuda.current_stream().wait_stream(s)
    for t in (y, ro, q, sc):
        t.view(torch.uint8).fill_(0)
    g.replay()
    torch.cuda.synchronize()
    ref = orc.fused([synth.bits(p) for p in inp["partials"]], synth.bits(inp["residual"]),
                    synth.bits(inp["weight"]), 1e-6, True, True, "bf16")
    assert_bits_equal(bits_of(ro), ref["res_out"], "residual_out")
    yb = bits_of(y)
    assert_y_within_ulp(yb, ref["y"], "bf16")
    assert_fp8(orc, q.numpy(), sc.numpy(), yb, "bf16", ref)


def test_host_refusals(ctx, dev):
    _reset(ctx)
    m, h = 16, 1024
    inp = synth.fused_inputs(2, m, h, "bf16", seed=1)
    pinned = [_pinned(p) for p in inp["partials"]]
    w = _pinned(inp["weight"])
    y = torch.empty((m, h), dtype=torch.bfloat16, pin_memory=True)
    pageable = inp["partials"][0].clone()          # ordinary (pageable) host memory
    assert not pageable.is_pinned()

    def status(partials, out, **kw):
        a = tar.make_fused_args([p.data_ptr() for p in partials], None, None, w.data_ptr(), out.data_ptr(),
                                1e-6, False, False, None, None, m, h, tar.AR_DTYPE_BF16, **kw)
        return tar.ar_fused_reduce_rmsnorm_host(ctx.handle, a, torch.cuda.current_stream().cuda_stream,
                                                raise_on_error=False)

    assert status(pinned, y) == tar.AR_OK
    assert status([pinned[0], pageable], y) == tar.AR_ERR_INVALID_ARG
    assert b"page-locked" in tar.load_library().ar_last_error(ctx.handle)
    y_pageable = torch.empty((m, h), dtype=torch.bfloat16)
    assert status(pinned, y_pageable) == tar.AR_ERR_INVALID_ARG
    ctx.set_option(tar.AR_OPT_FORCE_VARIANT, tar.VARIANT_STAGED)
    assert status(pinned, y) == tar.AR_ERR_UNSUPPORTED
    _reset(ctx)
    torch.cuda.synchronize()
    with pytest.raises(ValueError):                # the torch front end refuses pageable tensors itself
        ctx.fused_reduce_rmsnorm_host([pinned[0], pageable], None, w, out=y)
    assert ctx.device_status() == 0
