"""The allocation-free entry point, ar_fused_reduce_rmsnorm_noalloc.

It serves callers that cannot call cudaMalloc where they need the op (an engine whose
device memory is all planned up front, code inside a stream capture, a loop that must not
let an allocation synchronise the device).  It takes no context and keeps the staged
kernel's status word in a static device array.  Here it is called through the C ABI: twice
in a row against the context-based ar_fused_reduce_rmsnorm on the same inputs, and against
the oracle with the parity bars of the other tests (residual_out bit-exact, y within one
ulp, FP8 codes and scales exact on the kernel's own y), over both element types, the
no-norm form with a NULL weight, fp32 output, per-group FP8, padded rows and the empty call.

This file is collected last on purpose: it must pass alone in a fresh process and after
every other test.
"""
import ctypes

import numpy as np
import pytest
import torch

import tensor_all_reduce_gb300 as tar
from tensor_all_reduce_gb300 import synth

from gpu_helpers import TDT, assert_bits_equal, assert_y_within_ulp, bits_of, code_ordinal

pytestmark = pytest.mark.gpu


@pytest.fixture(scope="module")
def lib():
    if not torch.cuda.is_available():
        pytest.skip("no CUDA device")
    import __graft_entry__
    __graft_entry__.build()
    lib = tar.load_library()
    lib.ar_fused_reduce_rmsnorm_noalloc.argtypes = [ctypes.POINTER(tar.ArFusedArgs), ctypes.c_void_p]
    lib.ar_fused_reduce_rmsnorm_noalloc.restype = ctypes.c_int
    return lib


def _noalloc_call(lib, parts, res, w, y, ro, q, sc, gemma, quant, dtype_code):
    m, h = parts[0].shape
    args = tar.make_fused_args([p.data_ptr() for p in parts], res.data_ptr(), ro.data_ptr(), w.data_ptr(),
                               y.data_ptr(), 1e-6, gemma, quant, None if q is None else q.data_ptr(),
                               None if sc is None else sc.data_ptr(), m, h, dtype_code)
    return lib.ar_fused_reduce_rmsnorm_noalloc(ctypes.byref(args), torch.cuda.current_stream().cuda_stream)


def test_noalloc_matches_context_entry_point_on_two_calls(lib):
    dev = torch.device("cuda", 0)
    cases = [(4, 1000, 4096, True, True), (8, 300, 6144, False, False)]
    with tar.Context(0) as ctx:
        for call, (n, m, h, quant, gemma) in enumerate(cases):
            inp = synth.fused_inputs(n, m, h, "bf16", seed=100 + call, gemma=gemma)
            parts = [p.to(dev) for p in inp["partials"]]
            res, w = inp["residual"].to(dev), inp["weight"].to(dev)
            y1, ro1, q1, s1 = ctx.fused_reduce_rmsnorm(parts, res, w, eps=1e-6, gemma=gemma, quant=quant)
            y2 = torch.full_like(y1, float("nan"))
            ro2 = torch.full_like(ro1, float("nan"))
            q2 = torch.full((m, h), 0x7F, dtype=torch.uint8, device=dev) if quant else None
            s2 = torch.full((m,), float("nan"), dtype=torch.float32, device=dev) if quant else None
            torch.cuda.synchronize()
            free_before = torch.cuda.mem_get_info(dev)[0]
            st = _noalloc_call(lib, parts, res, w, y2, ro2, q2, s2, gemma, quant, tar.AR_DTYPE_BF16)
            torch.cuda.synchronize()
            assert st == tar.AR_OK, tar.status_string(st)
            if call > 0:   # after the first call's one-time set-up nothing is allocated
                assert torch.cuda.mem_get_info(dev)[0] == free_before
            assert_bits_equal(bits_of(ro2), bits_of(ro1), "residual_out")
            assert_y_within_ulp(bits_of(y2), bits_of(y1), "bf16")
            if quant:
                a, b = s2.cpu().numpy().astype(np.float64), s1.cpu().numpy().astype(np.float64)
                assert np.all(np.abs(a - b) <= 1e-6 * np.abs(b))
                d = np.abs(code_ordinal(q2.cpu().numpy()) - code_ordinal(q1.cpu().numpy()))
                assert d.max() <= 1


def test_noalloc_refuses_what_the_staged_kernel_cannot_do(lib):
    dev = torch.device("cuda", 0)
    for h in (6145, 16384):                      # not a multiple of 8 / wider than 8192
        inp = synth.fused_inputs(2, 4, h, "bf16", seed=1)
        parts = [p.to(dev) for p in inp["partials"]]
        res, w = inp["residual"].to(dev), inp["weight"].to(dev)
        y, ro = torch.empty_like(parts[0]), torch.empty_like(parts[0])
        st = _noalloc_call(lib, parts, res, w, y, ro, None, None, False, False, tar.AR_DTYPE_BF16)
        assert st == tar.AR_ERR_UNSUPPORTED
    # argument errors are those of the context entry point
    inp = synth.fused_inputs(2, 4, 64, "bf16", seed=2)
    parts = [p.to(dev) for p in inp["partials"]]
    res, w = inp["residual"].to(dev), inp["weight"].to(dev)
    y = torch.empty_like(parts[0])
    st = _noalloc_call(lib, parts, res, w, y, y, None, None, False, False, tar.AR_DTYPE_BF16)
    assert st == tar.AR_ERR_OVERLAP                 # residual_out == out


DT_CODE = {"bf16": tar.AR_DTYPE_BF16, "fp16": tar.AR_DTYPE_F16}
F32_REL_TOL = 2.0 ** -19     # the fp32-output bar of the context entry's tests


def _noalloc(lib, parts, res, w, y, ro, q, sc, dtype, *, gemma=False, quant=False, skip_norm=False,
             out_fp32=False, group=0, ld_in=0, ld_out=0, m=None, h=None):
    m = parts[0].shape[0] if m is None else m
    h = parts[0].shape[1] if h is None else h
    ptr = lambda t: None if t is None else t.data_ptr()
    args = tar.make_fused_args([p.data_ptr() for p in parts], ptr(res), ptr(ro), ptr(w), ptr(y), 1e-6, gemma, quant,
                               ptr(q), ptr(sc), m, h, DT_CODE[dtype], skip_norm=skip_norm, out_fp32=out_fp32,
                               group_size=group, ld_in=ld_in, ld_out=ld_out)
    return lib.ar_fused_reduce_rmsnorm_noalloc(ctypes.byref(args), torch.cuda.current_stream().cuda_stream)


FORMS = {
    "gemma_fp8_mirror": dict(gemma=True, quant=True),
    "plain": dict(),
    "nonorm_fp8": dict(quant=True, skip_norm=True),
    "f32out_fp8": dict(quant=True, out_fp32=True),
    "group64_fp8": dict(gemma=True, quant=True, group=64),
}


@pytest.mark.parametrize("dtype", ["bf16", "fp16"])
@pytest.mark.parametrize("form", list(FORMS))
def test_noalloc_matches_the_oracle(lib, orc, dtype, form):
    dev = torch.device("cuda", 0)
    kw = FORMS[form]
    n, m, h = 4, 333, 6144
    inp = synth.fused_inputs(n, m, h, dtype, seed=200 + len(form), gemma=kw.get("gemma", False))
    parts = [p.to(dev) for p in inp["partials"]]
    res = inp["residual"].to(dev)
    w = None if kw.get("skip_norm") else inp["weight"].to(dev)
    y = torch.full((m, h), float("nan"), dtype=torch.float32 if kw.get("out_fp32") else TDT[dtype], device=dev)
    ro = torch.full((m, h), float("nan"), dtype=TDT[dtype], device=dev)
    q = torch.full((m, h), 0x7F, dtype=torch.uint8, device=dev) if kw.get("quant") else None
    g = kw.get("group", 0)
    sc = torch.full((m, h // g) if g else (m,), float("nan"), dtype=torch.float32, device=dev) if q is not None else None
    st = _noalloc(lib, parts, res, w, y, ro, q, sc, dtype, **kw)
    torch.cuda.synchronize()
    assert st == tar.AR_OK, tar.status_string(st)
    ref = orc.fused_ex([synth.bits(p) for p in inp["partials"]], synth.bits(inp["residual"]),
                       None if w is None else synth.bits(inp["weight"]), 1e-6, kw.get("gemma", False),
                       kw.get("quant", False), dtype, skip_norm=kw.get("skip_norm", False),
                       out_fp32=kw.get("out_fp32", False), group=g)
    ro_b = bits_of(ro)
    assert_bits_equal(ro_b, ref["res_out"], "residual_out")
    if kw.get("out_fp32"):
        yg, yr = y.cpu().numpy().astype(np.float64), ref["y32"].astype(np.float64)
        assert np.all(np.abs(yg - yr) <= F32_REL_TOL * np.abs(yr) + 1e-30)
    elif kw.get("skip_norm"):
        assert_bits_equal(bits_of(y), ref["y"], "output (= z)")
    else:
        assert_y_within_ulp(bits_of(y), ref["y"], dtype)
    if q is not None:
        if kw.get("out_fp32"):        # the 16-bit rounded row is not an output: scales within one ulp of amax
            tol = 2.0 ** -7 if dtype == "bf16" else 2.0 ** -10
            s_g, s_r = sc.cpu().numpy().astype(np.float64), ref["scale"].astype(np.float64)
            assert np.all(np.abs(s_g - s_r) <= tol * s_r * 1.0001)
            d = np.abs(code_ordinal(q.cpu().numpy()) - code_ordinal(ref["q"]))
            assert d.max(initial=0) <= 1
        else:
            yb = ro_b if kw.get("skip_norm") else bits_of(y)
            q_ref, s_ref = orc.per_group_quant(yb, g, dtype) if g else orc.per_token_quant(yb, dtype)
            assert np.array_equal(sc.cpu().numpy().view(np.uint32), s_ref.view(np.uint32))
            assert np.array_equal(q.cpu().numpy(), q_ref)


def test_noalloc_padded_rows(lib, orc):
    """Row strides ld_in / ld_out above h: the results of the contiguous call, the padding untouched."""
    dev = torch.device("cuda", 0)
    n, m, h, li, lo = 4, 200, 4096, 4096 + 24, 4096 + 64
    inp = synth.fused_inputs(n, m, h, "bf16", seed=77, gemma=True)
    pad_in = [torch.full((m, li), 7.0, dtype=torch.bfloat16, device=dev) for _ in range(n + 1)]
    for buf, src in zip(pad_in, inp["partials"] + [inp["residual"]]):
        buf[:, :h].copy_(src.to(dev))
    outs = [torch.full((m, lo), 3.0, dtype=torch.bfloat16, device=dev) for _ in range(2)]
    qbuf = torch.full((m, lo), 0x55, dtype=torch.uint8, device=dev)
    sc = torch.empty((m,), dtype=torch.float32, device=dev)
    w = inp["weight"].to(dev)
    parts = [b[:, :h] for b in pad_in[:n]]
    st = _noalloc(lib, parts, pad_in[n][:, :h], w, outs[0][:, :h], outs[1][:, :h], qbuf[:, :h], sc, "bf16",
                  gemma=True, quant=True, ld_in=li, ld_out=lo)
    torch.cuda.synchronize()
    assert st == tar.AR_OK, tar.status_string(st)
    ref = orc.fused([synth.bits(p) for p in inp["partials"]], synth.bits(inp["residual"]), synth.bits(inp["weight"]),
                    1e-6, True, True, "bf16")
    assert_bits_equal(bits_of(outs[1][:, :h]), ref["res_out"], "residual_out")
    yb = bits_of(outs[0][:, :h])
    assert_y_within_ulp(yb, ref["y"], "bf16")
    q_ref, s_ref = orc.per_token_quant(yb, "bf16")
    assert np.array_equal(qbuf[:, :h].cpu().numpy(), q_ref)
    assert np.array_equal(sc.cpu().numpy().view(np.uint32), s_ref.view(np.uint32))
    assert bool((outs[0][:, h:] == 3.0).all()) and bool((outs[1][:, h:] == 3.0).all())
    assert bool((qbuf[:, h:] == 0x55).all())


def test_noalloc_empty_call(lib):
    """m = 0: AR_OK with nothing launched; only the weight has to be a real pointer."""
    dev = torch.device("cuda", 0)
    w = torch.ones(64, dtype=torch.bfloat16, device=dev)
    args = tar.make_fused_args([0, 0], None, None, w.data_ptr(), None, 1e-6, False, False, None, None, 0, 64,
                               tar.AR_DTYPE_BF16)
    st = lib.ar_fused_reduce_rmsnorm_noalloc(ctypes.byref(args), torch.cuda.current_stream().cuda_stream)
    torch.cuda.synchronize()
    assert st == tar.AR_OK
