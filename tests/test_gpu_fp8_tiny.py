"""FP8 epilogue on rows and groups of tiny magnitude (bf16 maxima between 2^-133 and 2^-118).

There, scale = amax / 448 is a binary32 subnormal (or close to one) whose reciprocal
overflows, so a quotient formed from the reciprocal would be NaN or infinite.  The kernels
take the IEEE division for maxima below 2^-80; this file checks, on every kernel form and
entry point (row, cluster, staged, staged cluster, element-wise, batch, allocation-free,
host buffers), that codes and scales then equal the oracle's quantisation of the kernel's
own y exactly, that no NaN code (0x7F / 0xFF) is written, and that residual_out and y
keep their usual bars.  Three ways such rows arise:

* all-reduce + FP8 without the norm on rows of tiny sums (y = z);
* per-group FP8 where some groups hold tiny values next to groups of normal size;
* RMSNorm with a near-zero weight row, so every y of the row is tiny.

Source of the epilogue: page "[HIP] fix(custom-ar): gfx1250 fused all-reduce + RMSNorm",
Changes (per-token FP8 of the rounded output with the steps of
dynamic_per_token_scaled_quant; the same codes and scales as the unfused path).
"""
import numpy as np
import pytest
import torch

import tensor_all_reduce_gb300 as tar
from tensor_all_reduce_gb300 import synth

from gpu_helpers import assert_bits_equal, assert_y_within_ulp, bits_of

pytestmark = pytest.mark.gpu

BF16 = torch.bfloat16


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


def _scaled(t, mags):
    """bf16 tensor t times per-row (or per-column) powers of two, rounded to bf16."""
    return (t.float() * mags).to(BF16)


def tiny_rows_inputs(m, h, seed):
    """Rows whose partials and residual are N(0,1) times 2^k, k from -133 to -118 (some rows
    of normal size and one all-zero row in between)."""
    inp = synth.fused_inputs(4, m, h, "bf16", seed=seed)
    ks = torch.tensor([[-133 + (r % 16)] if r % 5 != 4 else [0] for r in range(m)], dtype=torch.float32)
    mags = torch.pow(2.0, ks)
    inp["partials"] = [_scaled(p, mags) for p in inp["partials"]]
    inp["residual"] = _scaled(inp["residual"], mags)
    if m > 3:
        for p in inp["partials"]:
            p[3].zero_()
        inp["residual"][3].zero_()
    return inp


def tiny_groups_inputs(m, h, group, seed):
    """RMSNorm (plain) with a weight whose groups alternate between normal size and 2^-125..
    2^-131 times 1 + 0.1 N(0,1): the normalised row has tiny groups next to normal ones."""
    inp = synth.fused_inputs(4, m, h, "bf16", seed=seed)
    g = torch.arange(h) // group
    ks = torch.where(g % 2 == 1, -125.0 - (g % 7).float(), torch.zeros(h))
    inp["weight"] = _scaled(inp["weight"], torch.pow(2.0, ks))
    return inp


def tiny_weight_inputs(m, h, seed):
    """RMSNorm (plain) with a near-zero weight row (2^-127 times 1 + 0.1 N(0,1), partly
    subnormal): every normalised value is tiny."""
    inp = synth.fused_inputs(4, m, h, "bf16", seed=seed)
    inp["weight"] = _scaled(inp["weight"], torch.tensor(2.0 ** -127))
    return inp


CASES = {
    "nonorm_tiny_rows": dict(make=lambda m, h: tiny_rows_inputs(m, h, 31), skip_norm=True, group=0),
    "nonorm_tiny_rows_group16": dict(make=lambda m, h: tiny_rows_inputs(m, h, 32), skip_norm=True, group=16),
    "tiny_groups_group32": dict(make=lambda m, h: tiny_groups_inputs(m, h, 32, 33), skip_norm=False, group=32),
    "tiny_weight_row": dict(make=lambda m, h: tiny_weight_inputs(m, h, 34), skip_norm=False, group=0),
}


def _oracle(orc, inp, case):
    return orc.fused_ex([synth.bits(p) for p in inp["partials"]], synth.bits(inp["residual"]),
                        None if case["skip_norm"] else synth.bits(inp["weight"]), 1e-6, False, True, "bf16",
                        skip_norm=case["skip_norm"], group=case["group"])


def _check(orc, case, ref, y_bits, ro_bits, q, sc):
    assert_bits_equal(ro_bits, ref["res_out"], "residual_out")
    if case["skip_norm"]:
        assert_bits_equal(y_bits, ref["y"], "output (= z)")
    else:
        assert_y_within_ulp(y_bits, ref["y"], "bf16")
    assert not np.any((q & 0x7F) == 0x7F), "a NaN code was written"
    if case["group"]:
        q_ref, s_ref = orc.per_group_quant(y_bits, case["group"], "bf16")
    else:
        q_ref, s_ref = orc.per_token_quant(y_bits, "bf16")
    assert np.array_equal(sc.view(np.uint32), s_ref.view(np.uint32)), "scales differ from the oracle's"
    assert np.array_equal(q, q_ref), "codes differ from the oracle's quantisation of the kernel's y"
    # the inputs do reach the range where the reciprocal of the scale overflows
    assert np.any((s_ref > 0) & (s_ref < np.float32(2.0 ** -126)))


def _args(inp_dev, outs, case, m, h):
    parts, res, w = inp_dev
    y, ro, q, sc = outs
    return tar.make_fused_args([p.data_ptr() for p in parts], res.data_ptr(), ro.data_ptr(),
                               None if case["skip_norm"] else w.data_ptr(), y.data_ptr(), 1e-6, False, True,
                               q.data_ptr(), sc.data_ptr(), m, h, tar.AR_DTYPE_BF16, skip_norm=case["skip_norm"],
                               group_size=case["group"])


def _alloc(dev, m, h, group, pinned=False):
    kw = dict(pin_memory=True) if pinned else dict(device=dev)
    y = torch.full((m, h), float("nan"), dtype=BF16, **kw)
    ro = torch.full((m, h), float("nan"), dtype=BF16, **kw)
    q = torch.full((m, h), 0x7F, dtype=torch.uint8, **kw)
    sc = torch.full((m, h // group) if group else (m,), float("nan"), dtype=torch.float32, **kw)
    return y, ro, q, sc


def _to_dev(inp, dev):
    return [p.to(dev) for p in inp["partials"]], inp["residual"].to(dev), inp["weight"].to(dev)


def _host(outs):
    y, ro, q, sc = outs
    return bits_of(y), bits_of(ro), q.cpu().numpy(), sc.cpu().numpy()


FORMS = {
    "row": ({tar.AR_OPT_FORCE_VARIANT: tar.VARIANT_ROW}, "fused_row_vec"),
    "cluster4": ({tar.AR_OPT_CLUSTER_SIZE: 4}, "fused_cluster_vec"),
    "staged": ({tar.AR_OPT_FORCE_VARIANT: tar.VARIANT_STAGED}, "fused_staged"),
    "scalar": ({tar.AR_OPT_FORCE_VARIANT: tar.VARIANT_SCALAR}, "fused_scalar"),
}
# the element-wise form splits rows over a cluster when there are fewer rows than SMs
ALSO = {"fused_scalar": "fused_cluster_scalar"}


@pytest.mark.parametrize("case_name", list(CASES))
@pytest.mark.parametrize("form", list(FORMS))
def test_tiny_fp8_every_kernel_form(ctx, dev, orc, case_name, form):
    case = CASES[case_name]
    opts, variant = FORMS[form]
    if case["group"] and form == "cluster4":
        variant = "fused_row_vec"        # per-group FP8 keeps a row in one CTA
    _set(ctx, opts)
    m, h = 40, 2048
    inp = case["make"](m, h)
    parts, res, w = _to_dev(inp, dev)
    outs = _alloc(dev, m, h, case["group"])
    y, ro, q, sc = outs
    ctx.fused_reduce_rmsnorm(parts, res, None if case["skip_norm"] else w, eps=1e-6, quant=True, out=y,
                             residual_out=ro, q_out=q, scale_out=sc, skip_norm=case["skip_norm"],
                             group_size=case["group"])
    torch.cuda.synchronize()
    assert ctx.last_variant in (variant, ALSO.get(variant)), ctx.last_variant
    _check(orc, case, _oracle(orc, inp, case), *_host(outs))
    _set(ctx, {})


@pytest.mark.parametrize("case_name", ["nonorm_tiny_rows", "tiny_weight_row"])
def test_tiny_fp8_staged_cluster(ctx, dev, orc, case_name):
    """Rows longer than one CTA holds: the staged cluster form (two CTAs per row)."""
    case = CASES[case_name]
    _set(ctx, {tar.AR_OPT_FORCE_VARIANT: tar.VARIANT_STAGED, tar.AR_OPT_CLUSTER_SIZE: 2})
    m, h = 20, 16384
    inp = case["make"](m, h)
    parts, res, w = _to_dev(inp, dev)
    outs = _alloc(dev, m, h, 0)
    y, ro, q, sc = outs
    ctx.fused_reduce_rmsnorm(parts, res, None if case["skip_norm"] else w, eps=1e-6, quant=True, out=y,
                             residual_out=ro, q_out=q, scale_out=sc, skip_norm=case["skip_norm"])
    torch.cuda.synchronize()
    assert ctx.last_variant == "fused_staged_cluster"
    _check(orc, case, _oracle(orc, inp, case), *_host(outs))
    _set(ctx, {})


@pytest.mark.parametrize("case_name", list(CASES))
def test_tiny_fp8_batch(ctx, dev, orc, case_name):
    case = CASES[case_name]
    _set(ctx, {})
    calls, keep = [], []
    for k, (m, h) in enumerate(((7, 2048), (16, 4096), (1, 1024))):
        inp = case["make"](m, h)
        parts, res, w = _to_dev(inp, dev)
        outs = _alloc(dev, m, h, case["group"])
        y, ro, q, sc = outs
        calls.append({"partials": parts, "residual": res, "weight": None if case["skip_norm"] else w,
                      "eps": 1e-6, "quant": True, "out": y, "residual_out": ro, "q_out": q, "scale_out": sc,
                      "skip_norm": case["skip_norm"], "group_size": case["group"]})
        keep.append((inp, outs))
    ctx.fused_reduce_rmsnorm_batch(calls)
    torch.cuda.synchronize()
    assert ctx.last_variant == "fused_batch"
    for inp, outs in keep:
        _check(orc, case, _oracle(orc, inp, case), *_host(outs))


@pytest.mark.parametrize("case_name", list(CASES))
def test_tiny_fp8_host_buffers(ctx, dev, orc, case_name):
    case = CASES[case_name]
    _set(ctx, {})
    m, h = 24, 2048
    inp = case["make"](m, h)
    parts = [p.pin_memory() for p in inp["partials"]]
    res, w = inp["residual"].pin_memory(), inp["weight"].pin_memory()
    outs = _alloc(dev, m, h, case["group"], pinned=True)
    y, ro, q, sc = outs
    ctx.fused_reduce_rmsnorm_host(parts, res, None if case["skip_norm"] else w, eps=1e-6, quant=True, out=y,
                                  residual_out=ro, q_out=q, scale_out=sc, skip_norm=case["skip_norm"],
                                  group_size=case["group"])
    torch.cuda.synchronize()
    _check(orc, case, _oracle(orc, inp, case), *_host(outs))


@pytest.mark.parametrize("case_name", list(CASES))
def test_tiny_fp8_noalloc(dev, orc, case_name):
    case = CASES[case_name]
    m, h = 300, 4096
    inp = case["make"](m, h)
    d = _to_dev(inp, dev)
    outs = _alloc(dev, m, h, case["group"])
    args = _args(d, outs, case, m, h)
    tar.ar_fused_reduce_rmsnorm_noalloc(args, torch.cuda.current_stream().cuda_stream)
    torch.cuda.synchronize()
    _check(orc, case, _oracle(orc, inp, case), *_host(outs))
