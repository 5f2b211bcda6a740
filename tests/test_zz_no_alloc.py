"""The allocation-free entry point, ar_fused_reduce_rmsnorm_noalloc.

It serves callers that cannot call cudaMalloc where they need the op (an engine whose
device memory is all planned up front, code inside a stream capture, a loop that must not
let an allocation synchronise the device).  It takes no context and keeps the staged
kernel's status word in a static device array.  Here it is called through the C ABI twice
in a row and each result is checked against the context-based ar_fused_reduce_rmsnorm on
the same inputs, with the parity bars of the other tests: residual_out bit-exact, y within
one ulp, FP8 codes within one code and scales within 1e-6 relative.

This file is collected last on purpose: it must pass alone in a fresh process and after
every other test.
"""
import ctypes

import numpy as np
import pytest
import torch

import tensor_all_reduce_gb300 as tar
from tensor_all_reduce_gb300 import synth

from gpu_helpers import assert_bits_equal, assert_y_within_ulp, bits_of, code_ordinal

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
