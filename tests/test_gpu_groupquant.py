"""GPU parity of the per-group FP8 epilogue (AR_QUANT_FP8_E4M3_PER_GROUP).

Reading (the pages name per-group fused forms without a group size or scale rule): every
run of G consecutive elements of a row gets scale amax_group / 448 and its codes by the
per-token rules.  Checked against the oracle on every kernel variant: residual_out
bit-exact, y within one ulp, and, given the kernel's own y, every code and scale exact.
"""
import ctypes

import numpy as np
import pytest
import torch

import tensor_all_reduce_gb300 as tar
from tensor_all_reduce_gb300 import synth

from gpu_helpers import assert_bits_equal, assert_y_within_ulp, bits_of

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
            "scalar": {tar.AR_OPT_FORCE_VARIANT: tar.VARIANT_SCALAR}}


def _set(ctx, opts):
    for o in range(5):
        ctx.set_option(o, 0)
    for k, v in opts.items():
        ctx.set_option(k, v)


def _check(orc, inp, y, ro, q, sc, dtype, group, gemma, skip_norm=False):
    ref = orc.fused_ex([synth.bits(p) for p in inp["partials"]], synth.bits(inp["residual"]),
                       None if skip_norm else synth.bits(inp["weight"]), 1e-6, gemma, True, dtype,
                       skip_norm=skip_norm, group=group)
    assert_bits_equal(bits_of(ro), ref["res_out"], "residual_out")
    yb = bits_of(y)
    assert_y_within_ulp(yb, ref["y"], dtype)
    q_ref, s_ref = orc.per_group_quant(yb, group, dtype)      # the same decision on the kernel's y
    assert np.array_equal(sc.cpu().numpy().view(np.uint32), s_ref.view(np.uint32))
    assert np.array_equal(q.cpu().numpy(), q_ref)


@pytest.mark.parametrize("variant", list(VARIANTS))
@pytest.mark.parametrize("group", [8, 32, 128, 256])
@pytest.mark.parametrize("dtype", ["bf16", "fp16"])
def test_per_group_every_variant(ctx, dev, orc, variant, group, dtype):
    _set(ctx, VARIANTS[variant])
    for m, h in ((700, 4096), (5, 6144), (3, 1024)):
        inp = synth.fused_inputs(4, m, h, dtype, seed=m + h + group, gemma=True)
        inp["partials"][0][1, :group] = 0           # a zero group (with the residual zeroed too)
        inp["residual"][1, :group] = 0
        for p in inp["partials"][1:]:
            p[1, :group] = 0
        parts = [p.to(dev) for p in inp["partials"]]
        y, ro, q, sc = ctx.fused_reduce_rmsnorm(parts, inp["residual"].to(dev), inp["weight"].to(dev), eps=1e-6,
                                                gemma=True, quant=True, group_size=group)
        torch.cuda.synchronize()
        assert sc.shape == (m, h // group)
        _check(orc, inp, y, ro, q, sc, dtype, group, True)
        assert (sc[1, 0] == 0).item() and (q[1, :group] == 0).all().item()


def test_per_group_without_norm(ctx, dev, orc):
    _set(ctx, {})
    inp = synth.fused_inputs(4, 900, 6144, "bf16", seed=5)
    parts = [p.to(dev) for p in inp["partials"]]
    y, ro, q, sc = ctx.fused_reduce_rmsnorm(parts, inp["residual"].to(dev), None, quant=True, skip_norm=True,
                                            group_size=64)
    torch.cuda.synchronize()
    _check(orc, inp, y, ro, q, sc, "bf16", 64, False, skip_norm=True)


def test_per_group_batched_and_allocation_free(ctx, dev, orc):
    _set(ctx, {})
    calls, inps = [], []
    for i, (m, h) in enumerate(((16, 6144), (1, 4096), (40, 2048))):
        inp = synth.fused_inputs(4, m, h, "bf16", seed=60 + i, gemma=True)
        inps.append(inp)
        calls.append({"partials": [p.to(dev) for p in inp["partials"]], "residual": inp["residual"].to(dev),
                      "weight": inp["weight"].to(dev), "eps": 1e-6, "gemma": True, "quant": True, "group_size": 128})
    outs = ctx.fused_reduce_rmsnorm_batch(calls)
    torch.cuda.synchronize()
    assert ctx.last_variant == "fused_batch"
    for (y, ro, q, sc), inp in zip(outs, inps):
        _check(orc, inp, y, ro, q, sc, "bf16", 128, True)
    # the context-free entry point takes the same arguments
    lib = tar.load_library()
    lib.ar_fused_reduce_rmsnorm_noalloc.argtypes = [ctypes.POINTER(tar.ArFusedArgs), ctypes.c_void_p]
    lib.ar_fused_reduce_rmsnorm_noalloc.restype = ctypes.c_int
    inp = inps[0]
    c = calls[0]
    m, h = c["partials"][0].shape
    y = torch.empty((m, h), dtype=torch.bfloat16, device=dev)
    ro = torch.empty_like(y)
    q = torch.empty((m, h), dtype=torch.uint8, device=dev)
    sc = torch.empty((m, h // 128), dtype=torch.float32, device=dev)
    a = tar.make_fused_args([p.data_ptr() for p in c["partials"]], c["residual"].data_ptr(), ro.data_ptr(),
                            c["weight"].data_ptr(), y.data_ptr(), 1e-6, True, True, q.data_ptr(), sc.data_ptr(), m, h,
                            tar.AR_DTYPE_BF16, group_size=128)
    assert lib.ar_fused_reduce_rmsnorm_noalloc(ctypes.byref(a), torch.cuda.current_stream().cuda_stream) == tar.AR_OK
    torch.cuda.synchronize()
    _check(orc, inp, y, ro, q, sc, "bf16", 128, True)


def test_per_group_workload_full_size(ctx, dev, orc):
    _set(ctx, {})
    wl = synth.by_name("n4_m2800_h6144_bf16_gemma_fp8_group128")
    inp = wl.inputs()
    parts = [p.to(dev) for p in inp["partials"]]
    y, ro, q, sc = ctx.fused_reduce_rmsnorm(parts, inp["residual"].to(dev), inp["weight"].to(dev), eps=1e-6,
                                            gemma=True, quant=True, group_size=wl.group)
    torch.cuda.synchronize()
    _check(orc, inp, y, ro, q, sc, "bf16", wl.group, True)
