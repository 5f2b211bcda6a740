"""Programmatic dependent launch (AR_OPT_PDL): kernels may be scheduled before their
predecessor on the stream finishes, and each waits for it before reading memory.

These chains make every call read what the previous call wrote: call k+1's residual is
call k's residual_out (bit-exact on both sides, so the oracle can follow the same chain),
and a plain reduce's output is the first partial of the next fused call.  Run eagerly and
captured in a CUDA graph, across the staged (few and many rows) and row kernels.
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


def _chain_oracle(orc, first_res, steps, n, m, h):
    """Oracle side of the chain: returns [(res_out_k, y_k)] for k = 0..steps-1."""
    out = []
    res = synth.bits(first_res)
    for k, st in enumerate(steps):
        parts = [synth.bits(p) for p in st["partials"]]
        if st["reduce_first"]:
            parts[0] = orc.reduce_sum([synth.bits(p) for p in st["reduce_in"]], "bf16").reshape(m, h)
        r = orc.fused(parts, res, synth.bits(st["weight"]), 1e-6, False, False, "bf16")
        out.append((r["res_out"], r["y"]))
        res = r["res_out"]
    return out


@pytest.mark.parametrize("pdl", [1, 0])
@pytest.mark.parametrize("m", [16, 300, 1000])
@pytest.mark.parametrize("graph", [False, True])
def test_pdl_chain_reads_predecessor_outputs(dev, orc, m, graph, pdl):
    n, h, K = 4, 6144, 6
    steps = []
    for k in range(K):
        inp = synth.fused_inputs(n, m, h, "bf16", seed=500 + k)
        st = {"partials": inp["partials"], "weight": inp["weight"], "reduce_first": k % 2 == 1}
        if st["reduce_first"]:
            st["reduce_in"] = synth.reduce_inputs(3, m * h, "bf16", seed=900 + k)
        steps.append(st)
    first_res = synth.fused_inputs(1, m, h, "bf16", seed=77)["partials"][0]
    ref = _chain_oracle(orc, first_res, steps, n, m, h)

    with tar.Context(0) as ctx:
        ctx.set_option(tar.AR_OPT_PDL, pdl)
        d_parts = [[p.to(dev) for p in st["partials"]] for st in steps]
        d_w = [st["weight"].to(dev) for st in steps]
        d_red_in = [[p.to(dev).view(m, h) for p in st["reduce_in"]] if st["reduce_first"] else None for st in steps]
        d_red_out = [torch.empty((m, h), dtype=torch.bfloat16, device=dev) for _ in steps]
        res0 = first_res.to(dev)
        d_ro = [torch.empty((m, h), dtype=torch.bfloat16, device=dev) for _ in steps]
        d_y = [torch.empty((m, h), dtype=torch.bfloat16, device=dev) for _ in steps]

        def run():
            res = res0
            for k, st in enumerate(steps):
                parts = list(d_parts[k])
                if st["reduce_first"]:
                    ctx.reduce_sum([p.view(-1) for p in d_red_in[k]], out=d_red_out[k].view(-1))
                    parts[0] = d_red_out[k]
                ctx.fused_reduce_rmsnorm(parts, res, d_w[k], eps=1e-6, out=d_y[k], residual_out=d_ro[k])
                res = d_ro[k]

        run()
        torch.cuda.synchronize()
        if graph:
            for t in d_ro + d_y + d_red_out:
                t.fill_(float("nan"))
            g = torch.cuda.CUDAGraph()
            s = torch.cuda.Stream()
            s.wait_stream(torch.cuda.current_stream())
            with torch.cuda.graph(g, stream=s):
                run()
            torch.cuda.current_stream().wait_stream(s)
            for _ in range(3):
                for t in d_ro + d_y + d_red_out:
                    t.fill_(float("nan"))
                g.replay()
            torch.cuda.synchronize()
        for k in range(K):
            assert_bits_equal(bits_of(d_ro[k]), ref[k][0], f"residual_out of call {k}")
            assert_y_within_ulp(bits_of(d_y[k]), ref[k][1], "bf16", f"y of call {k}")
        assert ctx.device_status() == 0
