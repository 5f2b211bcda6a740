"""GPU parity of the fused path's further forms against the oracle.

* skip_norm: all-reduce + residual add + dynamic per-token FP8 without RMSNorm (the
  all-reduce followed by dynamic_per_token_scaled_quant of page "[HIP] fix(custom-ar):
  gfx1250 fused all-reduce + RMSNorm", Changes, without the norm).  The output is the
  rounded sum plus residual, bit-exact, and the FP8 codes and scales follow from it exactly.
* out_fp32: the normalised row stored in fp32 before its rounding.  Bar: relative error
  2^-19 against the oracle's binary32 rounding of the binary64 value.  Derivation: the fp32
  square-sum over h <= 8192 elements carries at most ~log2(h) * 2^-24 < 2^-20 relative
  error, its reciprocal square root halves that and adds at most 2 ulp (rsqrtf), and the two
  products add 2^-24 each: about 2^-20.7 in total, within the bar with a factor 3 to spare.
"""
import numpy as np
import pytest
import torch

import tensor_all_reduce_gb300 as tar
from tensor_all_reduce_gb300 import synth

from gpu_helpers import TDT, assert_bits_equal, bits_of, code_ordinal

pytestmark = pytest.mark.gpu

F32_REL_TOL = 2.0 ** -19


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
            "cluster4": {tar.AR_OPT_CLUSTER_SIZE: 4}, "staged": {tar.AR_OPT_FORCE_VARIANT: tar.VARIANT_STAGED},
            "scalar": {tar.AR_OPT_FORCE_VARIANT: tar.VARIANT_SCALAR}}


def _set(ctx, opts):
    for o in range(5):
        ctx.set_option(o, 0)
    for k, v in opts.items():
        ctx.set_option(k, v)


def _run(ctx, dev, inp, dtype, **kw):
    parts = [p.to(dev) for p in inp["partials"]]
    res = inp["residual"].to(dev) if inp["residual"] is not None else None
    w = inp["weight"].to(dev) if not kw.get("skip_norm") else None
    y, ro, q, sc = ctx.fused_reduce_rmsnorm(parts, res, w, eps=1e-6, **kw)
    torch.cuda.synchronize()
    return y, ro, q, sc


@pytest.mark.parametrize("variant", list(VARIANTS))
@pytest.mark.parametrize("dtype", ["bf16", "fp16"])
@pytest.mark.parametrize("residual", [True, False])
def test_skip_norm_with_fp8(ctx, dev, orc, variant, dtype, residual):
    _set(ctx, VARIANTS[variant])
    for m, h in ((700, 4096), (5, 2880)):
        inp = synth.fused_inputs(4, m, h, dtype, seed=m + h, residual=residual)
        y, ro, q, sc = _run(ctx, dev, inp, dtype, skip_norm=True, quant=True)
        ref = orc.fused_ex([synth.bits(p) for p in inp["partials"]], synth.bits(inp["residual"]), None, 0.0, False,
                           True, dtype, skip_norm=True)
        assert_bits_equal(bits_of(ro), ref["res_out"], "residual_out")
        assert_bits_equal(bits_of(y), ref["y"], "output (= z)")
        assert np.array_equal(sc.cpu().numpy().view(np.uint32), ref["scale"].view(np.uint32))
        assert np.array_equal(q.cpu().numpy(), ref["q"])


@pytest.mark.parametrize("variant", list(VARIANTS))
@pytest.mark.parametrize("dtype", ["bf16", "fp16"])
@pytest.mark.parametrize("quant", [False, True])
def test_fp32_output(ctx, dev, orc, variant, dtype, quant):
    _set(ctx, VARIANTS[variant])
    for m, h in ((700, 4096), (3, 6144)):
        inp = synth.fused_inputs(4, m, h, dtype, seed=3 * m + h, gemma=quant)
        y32, ro, q, sc = _run(ctx, dev, inp, dtype, out_fp32=True, quant=quant, gemma=quant)
        ref = orc.fused_ex([synth.bits(p) for p in inp["partials"]], synth.bits(inp["residual"]),
                           synth.bits(inp["weight"]), 1e-6, quant, quant, dtype, out_fp32=True)
        assert y32.dtype == torch.float32
        assert_bits_equal(bits_of(ro), ref["res_out"], "residual_out")
        g, r = y32.cpu().numpy().astype(np.float64), ref["y32"].astype(np.float64)
        err = np.abs(g - r)
        assert np.all(err <= F32_REL_TOL * np.abs(r) + 1e-30), f"max rel err {np.max(err / np.maximum(np.abs(r), 1e-30))}"
        if quant:
            # FP8 still quantises the 16-bit-rounded row: codes within one code, scales within
            # one 16-bit ulp of amax of the oracle's (the kernel's rounded row is not an output)
            s_g, s_r = sc.cpu().numpy().astype(np.float64), ref["scale"].astype(np.float64)
            tol = 2.0 ** -7 if dtype == "bf16" else 2.0 ** -10
            assert np.all(np.abs(s_g - s_r) <= tol * s_r * 1.0001)
            same = s_g == s_r
            assert same.mean() > 0.99
            d = np.abs(code_ordinal(q.cpu().numpy()) - code_ordinal(ref["q"]))
            assert d.max(initial=0) <= 1


def test_skip_norm_fp32_output_is_z(ctx, dev, orc):
    _set(ctx, {})
    inp = synth.fused_inputs(3, 900, 2048, "bf16", seed=8)
    y32, ro, _, _ = _run(ctx, dev, inp, "bf16", skip_norm=True, out_fp32=True)
    z = torch.from_numpy(bits_of(ro).view(np.int16)).view(torch.bfloat16).float().numpy()
    assert np.array_equal(y32.cpu().numpy(), z)


OPTION_WORKLOADS = [w for w in synth.options() if not w.group]   # per-group: test_gpu_groupquant.py


@pytest.mark.parametrize("wl", OPTION_WORKLOADS, ids=[w.name for w in OPTION_WORKLOADS])
def test_option_workloads_full_size(ctx, dev, orc, wl):
    _set(ctx, {})
    inp = wl.inputs()
    kw = dict(skip_norm=wl.skip_norm, out_fp32=wl.out_fp32, quant=wl.quant, want_out=wl.mirror or not wl.quant)
    y, ro, q, sc = _run(ctx, dev, inp, wl.dtype, **kw)
    ref = orc.fused_ex([synth.bits(p) for p in inp["partials"]], synth.bits(inp["residual"]),
                       None if wl.skip_norm else synth.bits(inp["weight"]), 1e-6, False, wl.quant, wl.dtype,
                       skip_norm=wl.skip_norm, out_fp32=wl.out_fp32)
    assert_bits_equal(bits_of(ro), ref["res_out"], "residual_out")
    if wl.quant:
        assert np.array_equal(q.cpu().numpy(), ref["q"])
        assert np.array_equal(sc.cpu().numpy(), ref["scale"])
    if wl.out_fp32:
        g, r = y.cpu().numpy().astype(np.float64), ref["y32"].astype(np.float64)
        assert np.all(np.abs(g - r) <= F32_REL_TOL * np.abs(r) + 1e-30)
