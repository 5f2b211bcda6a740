"""The cluster form of the staged kernel: rows longer than one CTA holds (more than 8192
elements) are split over 2, 4 or 8 CTAs of a thread-block cluster, each staging its slice of
every row by bulk copies; the square-sum and the amax are combined through distributed
shared memory (the in-GPU form of page "[OUTDATED] perf: optimize fused AllReduce + RMSNorm
(custom_all_reduce)", Technical Details / 2stage: split the hidden dimension, then combine).
Same bar as every fused form against the oracle; the form can also be forced on shorter
rows, where it is checked with every option, and its bounded waits fail without a fault."""
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


def _set(ctx, opts):
    for o in range(5):
        ctx.set_option(o, 0)
    for k, v in opts.items():
        ctx.set_option(k, v)


def _run_and_check(ctx, dev, orc, n, m, h, dtype, quant, **kw):
    inp = synth.fused_inputs(n, m, h, dtype, seed=n + m + h, gemma=quant)
    parts = [p.to(dev) for p in inp["partials"]]
    y, ro, q, sc = ctx.fused_reduce_rmsnorm(parts, inp["residual"].to(dev), inp["weight"].to(dev), eps=1e-6,
                                            gemma=quant, quant=quant, **kw)
    torch.cuda.synchronize()
    ref = orc.fused([synth.bits(p) for p in inp["partials"]], synth.bits(inp["residual"]),
                    synth.bits(inp["weight"]), 1e-6, quant, quant, dtype)
    assert_bits_equal(bits_of(ro), ref["res_out"], "residual_out")
    yb = bits_of(y)
    assert_y_within_ulp(yb, ref["y"], dtype)
    if quant:
        assert_fp8(orc, q.cpu().numpy(), sc.cpu().numpy(), yb, dtype, ref)


@pytest.mark.parametrize("h", [12288, 16384, 24576, 65536])
@pytest.mark.parametrize("m", [1, 37, 700])
@pytest.mark.parametrize("quant", [False, True])
def test_wide_rows_take_the_cluster_form(ctx, dev, orc, h, m, quant):
    _set(ctx, {})
    _run_and_check(ctx, dev, orc, 4, m, h, "bf16", quant)
    assert ctx.last_variant == "fused_staged_cluster"
    assert ctx.device_status() == 0


@pytest.mark.parametrize("n", [1, 3, 8])
@pytest.mark.parametrize("dtype", ["bf16", "fp16"])
def test_wide_rows_every_n(ctx, dev, orc, n, dtype):
    _set(ctx, {})
    _run_and_check(ctx, dev, orc, n, 300, 16384, dtype, True)
    assert ctx.last_variant == "fused_staged_cluster"


@pytest.mark.parametrize("cl", [2, 4, 8])
@pytest.mark.parametrize("stages", [1, 2])
def test_forced_on_short_rows(ctx, dev, orc, cl, stages):
    _set(ctx, {tar.AR_OPT_FORCE_VARIANT: tar.VARIANT_STAGED, tar.AR_OPT_CLUSTER_SIZE: cl, tar.AR_OPT_STAGES: stages})
    for m, h in ((900, 6144), (5, 4096), (160, 2048)):
        _run_and_check(ctx, dev, orc, 4, m, h, "bf16", True)
        assert ctx.last_variant == "fused_staged_cluster"
    _set(ctx, {})


def test_forced_with_every_option(ctx, dev, orc):
    """Per-group FP8, no-norm FP8, fp32 output and padded rows through the cluster form."""
    _set(ctx, {tar.AR_OPT_FORCE_VARIANT: tar.VARIANT_STAGED, tar.AR_OPT_CLUSTER_SIZE: 2})
    m, h = 400, 6144
    inp = synth.fused_inputs(4, m, h, "bf16", seed=5, gemma=True)
    parts = [p.to(dev) for p in inp["partials"]]
    res, w = inp["residual"].to(dev), inp["weight"].to(dev)
    bits = [synth.bits(p) for p in inp["partials"]]
    # per-group FP8, groups of 128 (the 384-pack slices hold whole groups)
    y, ro, q, sc = ctx.fused_reduce_rmsnorm(parts, res, w, eps=1e-6, gemma=True, quant=True, group_size=128)
    torch.cuda.synchronize()
    assert ctx.last_variant == "fused_staged_cluster"
    ref = orc.fused_ex(bits, synth.bits(inp["residual"]), synth.bits(inp["weight"]), 1e-6, True, True, "bf16",
                       group=128)
    assert_bits_equal(bits_of(ro), ref["res_out"], "residual_out")
    yb = bits_of(y)
    assert_y_within_ulp(yb, ref["y"], "bf16")
    q_ref, s_ref = orc.per_group_quant(yb, 128, "bf16")
    assert np.array_equal(sc.cpu().numpy().view(np.uint32), s_ref.view(np.uint32))
    assert np.array_equal(q.cpu().numpy(), q_ref)
    # all-reduce + residual + per-token FP8 without the norm: exact
    y, ro, q, sc = ctx.fused_reduce_rmsnorm(parts, res, None, eps=1e-6, quant=True, skip_norm=True)
    torch.cuda.synchronize()
    ref = orc.fused_ex(bits, synth.bits(inp["residual"]), None, 0.0, False, True, "bf16", skip_norm=True)
    assert_bits_equal(bits_of(y), ref["y"], "output (= z)")
    assert np.array_equal(sc.cpu().numpy().view(np.uint32), ref["scale"].view(np.uint32))
    assert np.array_equal(q.cpu().numpy(), ref["q"])
    # fp32 output
    y32, ro, _, _ = ctx.fused_reduce_rmsnorm(parts, res, w, eps=1e-6, out_fp32=True)
    torch.cuda.synchronize()
    ref = orc.fused_ex(bits, synth.bits(inp["residual"]), synth.bits(inp["weight"]), 1e-6, False, False, "bf16",
                       out_fp32=True)
    g, r = y32.cpu().numpy().astype(np.float64), ref["y32"].astype(np.float64)
    assert np.all(np.abs(g - r) <= 2.0 ** -19 * np.abs(r) + 1e-30)
    # padded rows (strides that keep 16-byte row starts)
    pad = 64
    big = [torch.zeros((m, h + pad), dtype=torch.bfloat16, device=dev) for _ in range(5)]
    for b, t in zip(big, parts + [res]):
        b[:, :h].copy_(t)
    y_big = torch.full((m, h + 8), 3.0, dtype=torch.bfloat16, device=dev)
    ro_big = torch.full((m, h + 8), 3.0, dtype=torch.bfloat16, device=dev)
    ctx.fused_reduce_rmsnorm([b[:, :h] for b in big[:4]], big[4][:, :h], w, eps=1e-6, out=y_big[:, :h],
                             residual_out=ro_big[:, :h])
    torch.cuda.synchronize()
    assert ctx.last_variant == "fused_staged_cluster"
    assert bool((y_big[:, h:] == 3.0).all()) and bool((ro_big[:, h:] == 3.0).all())
    ref = orc.fused(bits, synth.bits(inp["residual"]), synth.bits(inp["weight"]), 1e-6, False, False, "bf16")
    assert_bits_equal(bits_of(ro_big[:, :h].contiguous()), ref["res_out"], "residual_out")
    assert_y_within_ulp(bits_of(y_big[:, :h].contiguous()), ref["y"], "bf16")
    _set(ctx, {})


def test_forced_refusals(ctx, dev):
    """Rows that do not split into whole 16-byte packs per CTA, or slices that would cut a
    per-group FP8 group, are refused before any launch."""
    _set(ctx, {tar.AR_OPT_FORCE_VARIANT: tar.VARIANT_STAGED, tar.AR_OPT_CLUSTER_SIZE: 4})
    inp = synth.fused_inputs(2, 8, 2056, "bf16", seed=1)          # 257 packs: not a multiple of 4
    parts = [p.to(dev) for p in inp["partials"]]
    with pytest.raises(tar.ArError) as e:
        ctx.fused_reduce_rmsnorm(parts, inp["residual"].to(dev), inp["weight"].to(dev))
    assert e.value.status == tar.AR_ERR_UNSUPPORTED
    inp = synth.fused_inputs(2, 8, 1536, "bf16", seed=2)          # 48-pack slices cut 32-pack groups
    parts = [p.to(dev) for p in inp["partials"]]
    with pytest.raises(tar.ArError) as e:
        ctx.fused_reduce_rmsnorm(parts, inp["residual"].to(dev), inp["weight"].to(dev), quant=True,
                                 group_size=256)
    assert e.value.status == tar.AR_ERR_UNSUPPORTED
    ctx.set_option(tar.AR_OPT_CLUSTER_SIZE, 16)                   # the staged clusters have 2 to 8 CTAs
    with pytest.raises(tar.ArError) as e:
        ctx.fused_reduce_rmsnorm(parts, inp["residual"].to(dev), inp["weight"].to(dev))
    assert e.value.status == tar.AR_ERR_UNSUPPORTED
    _set(ctx, {})


def test_pdl_chain_through_the_cluster_form(ctx, dev, orc):
    """Each call reads the previous call's residual_out (programmatic dependent launch on)."""
    _set(ctx, {})
    n, m, h, K = 4, 200, 16384, 4
    steps = [synth.fused_inputs(n, m, h, "bf16", seed=300 + k) for k in range(K)]
    res0 = synth.fused_inputs(1, m, h, "bf16", seed=7)["partials"][0]
    ref_res, refs = synth.bits(res0), []
    for st in steps:
        r = orc.fused([synth.bits(p) for p in st["partials"]], ref_res, synth.bits(st["weight"]), 1e-6, False,
                      False, "bf16")
        refs.append(r)
        ref_res = r["res_out"]
    res = res0.to(dev)
    outs = []
    for st in steps:
        y, ro, _, _ = ctx.fused_reduce_rmsnorm([p.to(dev) for p in st["partials"]], res, st["weight"].to(dev),
                                               eps=1e-6)
        outs.append((y, ro))
        res = ro
    torch.cuda.synchronize()
    assert ctx.last_variant == "fused_staged_cluster"
    for (y, ro), r in zip(outs, refs):
        assert_bits_equal(bits_of(ro), r["res_out"], "residual_out")
        assert_y_within_ulp(bits_of(y), r["y"], "bf16")


def test_cluster_wait_that_runs_out_is_reported(dev, orc):
    inp = synth.fused_inputs(4, 300, 16384, "bf16", seed=93)
    parts = [p.to(dev) for p in inp["partials"]]
    res, w = inp["residual"].to(dev), inp["weight"].to(dev)
    with tar.Context(0) as c:
        c.set_option(tar.AR_OPT_WAIT_CYCLES, 2_000_000)          # about a millisecond
        c.set_option(tar.AR_OPT_TEST_STALL, 1)
        c.fused_reduce_rmsnorm(parts, res, w, eps=1e-6)
        torch.cuda.synchronize()
        assert c.last_variant == "fused_staged_cluster"
        assert c.device_status() == 1
        c.set_option(tar.AR_OPT_TEST_STALL, 0)
        y, ro, _, _ = c.fused_reduce_rmsnorm(parts, res, w, eps=1e-6)
        torch.cuda.synchronize()
        ref = orc.fused([synth.bits(p) for p in inp["partials"]], synth.bits(inp["residual"]),
                        synth.bits(inp["weight"]), 1e-6, False, False, "bf16")
        assert_bits_equal(bits_of(ro), ref["res_out"], "residual_out")
        assert_y_within_ulp(bits_of(y), ref["y"], "bf16")
        assert c.device_status() == 0
