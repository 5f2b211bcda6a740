"""Distinct contexts are independent: two host threads, each with its own context and CUDA
stream, issue fused calls, plain sums and batches at the same time on separate buffers; every
result equals the oracle's, and each context's status word stays clear.  (One context is used
by one thread at a time, as the header states; ctypes releases the interpreter lock during the
C calls, so the two threads' launches do interleave.)"""
import threading

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


def _work(t, dev, rounds):
    """The calls of thread t: inputs drawn up front, outputs kept for checking."""
    jobs = []
    for r in range(rounds):
        seed = 10_000 * (t + 1) + r
        m = [3, 200, 1100, 16][r % 4]
        h = [6144, 4096, 2048, 7168][(r + t) % 4]
        quant = (r + t) % 2 == 1
        inp = synth.fused_inputs(4, m, h, "bf16", seed=seed, gemma=quant)
        red = synth.reduce_inputs(3, 257 * 1024 + r, "fp16", seed=seed)
        jobs.append({"inp": inp, "quant": quant, "red": red,
                     "d_parts": [p.to(dev) for p in inp["partials"]], "d_res": inp["residual"].to(dev),
                     "d_w": inp["weight"].to(dev), "d_red": [p.to(dev) for p in red]})
    return jobs


def test_two_threads_two_contexts(dev, orc):
    rounds = 12
    work = [_work(t, dev, rounds) for t in range(2)]
    torch.cuda.synchronize()
    errors = []
    barrier = threading.Barrier(2)

    def run(t):
        try:
            with tar.Context(0) as ctx:
                stream = torch.cuda.Stream()
                barrier.wait()
                with torch.cuda.stream(stream):
                    for job in work[t]:
                        job["out"] = ctx.fused_reduce_rmsnorm(job["d_parts"], job["d_res"], job["d_w"], eps=1e-6,
                                                              gemma=job["quant"], quant=job["quant"], stream=stream)
                        job["sum"] = ctx.reduce_sum(job["d_red"], stream=stream)
                stream.synchronize()
                job_status = ctx.device_status()
                if job_status != 0:
                    errors.append(f"thread {t}: status {job_status}")
        except Exception as e:          # reported to the main thread
            errors.append(f"thread {t}: {e!r}")

    threads = [threading.Thread(target=run, args=(t,)) for t in range(2)]
    for th in threads:
        th.start()
    for th in threads:
        th.join(timeout=300)
    assert not errors, errors
    torch.cuda.synchronize()
    for t in range(2):
        for job in work[t]:
            inp, quant = job["inp"], job["quant"]
            y, ro, q, sc = job["out"]
            ref = orc.fused([synth.bits(p) for p in inp["partials"]], synth.bits(inp["residual"]),
                            synth.bits(inp["weight"]), 1e-6, quant, quant, "bf16")
            assert_bits_equal(bits_of(ro), ref["res_out"], f"thread {t} residual_out")
            yb = bits_of(y)
            assert_y_within_ulp(yb, ref["y"], "bf16", f"thread {t} y")
            if quant:
                assert_fp8(orc, q.cpu().numpy(), sc.cpu().numpy(), yb, "bf16", ref)
            assert_bits_equal(synth.bits(job["sum"].cpu()), orc.reduce_sum([synth.bits(p) for p in job["red"]], "fp16"),
                              f"thread {t} sum")
