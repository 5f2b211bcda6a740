"""Failure detection without a GPU fault.

The staged kernels wait on shared-memory barriers that their own bulk copies complete, and
every wait is bounded.  The test hook AR_OPT_TEST_STALL arms each CTA's first stage without
issuing its copies: nothing completes that barrier, the wait runs out after the (shortened)
bound, the CTA records code 1 in the context's status word and returns.  The host reads the
code, and the same context then computes correctly again.  No trap, no fault, no endless
loop is involved.
"""
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


@pytest.mark.parametrize("stages", [1, 2])
def test_wait_that_runs_out_is_reported_and_context_recovers(dev, orc, stages):
    inp = synth.fused_inputs(4, 600, 4096, "bf16", seed=91)
    parts = [p.to(dev) for p in inp["partials"]]
    res, w = inp["residual"].to(dev), inp["weight"].to(dev)
    with tar.Context(0) as ctx:
        assert ctx.device_status() == 0
        ctx.set_option(tar.AR_OPT_FORCE_VARIANT, tar.VARIANT_STAGED)
        ctx.set_option(tar.AR_OPT_STAGES, stages)
        ctx.set_option(tar.AR_OPT_WAIT_CYCLES, 2_000_000)        # about a millisecond
        ctx.set_option(tar.AR_OPT_TEST_STALL, 1)
        ctx.fused_reduce_rmsnorm(parts, res, w, eps=1e-6)
        torch.cuda.synchronize()                                  # the kernel gave up and returned
        assert ctx.device_status() == 1
        assert ctx.device_status() == 0                           # reading clears it
        # the same context, without the hook: correct results and a clean status
        ctx.set_option(tar.AR_OPT_TEST_STALL, 0)
        y, ro, _, _ = ctx.fused_reduce_rmsnorm(parts, res, w, eps=1e-6)
        torch.cuda.synchronize()
        ref = orc.fused([synth.bits(p) for p in inp["partials"]], synth.bits(inp["residual"]),
                        synth.bits(inp["weight"]), 1e-6, False, False, "bf16")
        assert_bits_equal(bits_of(ro), ref["res_out"], "residual_out")
        assert_y_within_ulp(bits_of(y), ref["y"], "bf16")
        assert ctx.device_status() == 0


def test_batched_wait_that_runs_out_is_reported(dev):
    with tar.Context(0) as ctx:
        ctx.set_option(tar.AR_OPT_WAIT_CYCLES, 2_000_000)
        ctx.set_option(tar.AR_OPT_TEST_STALL, 1)
        calls = []
        for i in range(3):
            inp = synth.fused_inputs(2, 4, 2048, "bf16", seed=i)
            calls.append({"partials": [p.to(dev) for p in inp["partials"]], "residual": inp["residual"].to(dev),
                          "weight": inp["weight"].to(dev)})
        ctx.fused_reduce_rmsnorm_batch(calls)
        torch.cuda.synchronize()
        assert ctx.last_variant == "fused_batch"
        assert ctx.device_status() == 1
