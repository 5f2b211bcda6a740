"""The benchmark's multi-rank logic on CPU: two gloo ranks, each an independent replica.

The path has no exchange between GPUs (rows are independent and every rank holds its own
partials), so ranks only meet at the timing barriers and in the max over ranks.
"""
import json
import os
import socket
import subprocess
import sys

import pytest
import torch.multiprocessing as mp

ROOT = os.path.dirname(os.path.dirname(os.path.abspath(__file__)))


def _free_port():
    with socket.socket() as s:
        s.bind(("127.0.0.1", 0))
        return s.getsockname()[1]


def _worker(rank, world, port, q):
    os.environ.update(MASTER_ADDR="127.0.0.1", MASTER_PORT=str(port), RANK=str(rank), WORLD_SIZE=str(world),
                      LOCAL_RANK=str(rank))
    sys.path.insert(0, ROOT)
    import bench
    dist = bench.init_dist(world, "gloo")
    local_ms = 10.0 + 5.0 * rank           # rank 1 is the slow replica
    bench.barrier(world)
    m = bench.max_over_ranks(local_ms, world)
    q.put((rank, m, bench.job_us_per_call(m, 100, world)))
    dist.destroy_process_group()


def test_max_over_two_gloo_ranks():
    ctx = mp.get_context("spawn")
    q = ctx.Queue()
    port = _free_port()
    procs = [ctx.Process(target=_worker, args=(r, 2, port, q)) for r in range(2)]
    for p in procs:
        p.start()
    for p in procs:
        p.join(120)
        assert p.exitcode == 0
    got = sorted(q.get(timeout=5) for _ in range(2))
    # both ranks see the slowest replica's time; the job time per call spans both ranks' calls
    assert [g[1] for g in got] == [15.0, 15.0]
    assert got[0][2] == pytest.approx(15.0 * 1000 / 200)


def test_rotation_sets_cover_l2():
    sys.path.insert(0, ROOT)
    import bench
    l2 = 126 * 2**20
    assert bench.rotation_sets(258 * 10**6, l2) == 2
    assert bench.rotation_sets(10**9, l2) == 1
    assert bench.rotation_sets(98_304, l2, cap=4096) == 4032
    assert bench.rotation_sets(10, l2, cap=64) == 64


def test_reference_arm_under_two_ranks_only_rank0_prints():
    env = dict(os.environ, PYTHONPATH=ROOT)
    port = _free_port()
    cmd = [sys.executable, "-m", "torch.distributed.run", "--nnodes=1", "--nproc-per-node=2",
           "--master-addr=127.0.0.1", f"--master-port={port}", os.path.join(ROOT, "bench.py"),
           "--impl", "reference", "--gpus", "2", "--steps", "3", "--warmup", "3",
           "--workload", "n4_m16_h6144_bf16_plain"]
    r = subprocess.run(cmd, cwd=ROOT, env=env, capture_output=True, text=True, timeout=300)
    assert r.returncode == 0, r.stderr[-2000:]
    lines = [json.loads(line) for line in r.stdout.splitlines() if line.startswith("{")]
    assert len(lines) == 1
    line = lines[0]
    assert line["impl"] == "reference" and line["unit"] == "us/call" and line["higher_is_better"] is False
    assert line["cpu_baseline"]["kind"] == "oracle" and line["e2e"]["h2d_bytes_per_step"] == 0
    sys.path.insert(0, ROOT)
    import bench
    from tensor_all_reduce_gb300 import synth
    assert line["config"] == bench.workload_config(synth.by_name("n4_m16_h6144_bf16_plain"), 2)
    assert line["rows_per_step"] == 16 and "whole call" in line["cpu_baseline"]["sample"]
    # ms_per_step is the time a step took: steps x ms_per_step fits in the process's run time
    assert line["ms_per_step"] * line["steps"] < 300_000


def test_cpu_baseline_reports_serial_and_all_cores():
    sys.path.insert(0, ROOT)
    import bench
    import oracle
    from tensor_all_reduce_gb300 import synth
    wl = synth.by_name("n4_m16_h6144_bf16_plain")
    us, cores = bench.oracle_all_cores_us(bench.OracleInputs(wl), oracle.get(), runs=2)
    assert us > 0 and cores == bench.host_cores()
    cpu = bench.cpu_baseline(wl, budget_s=5.0)
    assert cpu["kind"] == "oracle" and cpu["cores"] == 1 and cpu["value"] > 0
    assert "whole calls" in cpu["sample"]
    assert cpu["all_cores"]["cores"] == cores and cpu["all_cores"]["unit"] == cpu["unit"]


def test_host_timings_take_whole_calls_when_they_fit():
    sys.path.insert(0, ROOT)
    import bench
    from tensor_all_reduce_gb300 import synth
    wl = synth.by_name("n8_m4096_h6144_bf16_plain")
    assert bench.rows_for_budget(wl, 3.5, 25, 150.0) == wl.m           # 87.5 s of whole calls
    rows = bench.rows_for_budget(wl, 10.0, 25, 150.0)                  # 250 s: a row sample
    assert 1 <= rows < wl.m and rows * 10.0 / wl.m * 25 <= 150.0


def test_headline_is_the_largest_configuration():
    sys.path.insert(0, ROOT)
    import bench
    from tensor_all_reduce_gb300 import synth
    wl = synth.by_name(bench.HEADLINE)
    sizes = [w.algorithmic_bytes() for _, w in bench.config_workloads()]
    assert wl.algorithmic_bytes() == max(sizes) and len(sizes) == 15
    assert [t for t, _ in bench.config_workloads()] == ["C1"] + ["C2"] * 6 + ["C3"] * 4 + ["C4"] * 3 + ["C5"]


def _leaving_worker(rank, world, port, q):
    import time
    os.environ.update(MASTER_ADDR="127.0.0.1", MASTER_PORT=str(port), RANK=str(rank), WORLD_SIZE=str(world),
                      LOCAL_RANK=str(rank))
    sys.path.insert(0, ROOT)
    import bench
    try:
        bench.init_dist(world, "gloo", timeout_s=20)
        bench.barrier(world)             # one step done together
    except Exception as e:
        q.put(("setup failed: " + type(e).__name__, -1.0))
        os._exit(0)
    if rank == 1:
        os._exit(0)                      # leaves between steps, without joining the next barrier
    t0 = time.time()
    try:
        bench.barrier(world)
        q.put(("no error", time.time() - t0))
    except Exception as e:               # the survivor learns of it as an error, not a hang
        q.put((type(e).__name__, time.time() - t0))
    os._exit(0)


def test_a_rank_that_leaves_is_an_error_on_the_other():
    port = _free_port()
    ctx = mp.get_context("spawn")
    q = ctx.SimpleQueue()                # put() writes synchronously: safe before os._exit
    ps = [ctx.Process(target=_leaving_worker, args=(r, 2, port, q)) for r in range(2)]
    for p in ps:
        p.start()
    for p in ps:
        p.join(timeout=120)
    assert not q.empty(), "the surviving rank reported nothing"
    kind, waited = q.get()
    assert not kind.startswith("setup failed"), kind
    assert kind != "no error"
    assert 0 <= waited < 60


def test_reference_arm_line_single_process():
    env = dict(os.environ, PYTHONPATH=ROOT)
    for k in ("WORLD_SIZE", "RANK", "LOCAL_RANK"):
        env.pop(k, None)
    cmd = [sys.executable, os.path.join(ROOT, "bench.py"), "--impl", "reference", "--steps", "3", "--warmup", "3",
           "--workload", "n4_m16_h6144_bf16_plain"]
    r = subprocess.run(cmd, cwd=ROOT, env=env, capture_output=True, text=True, timeout=300)
    assert r.returncode == 0, r.stderr[-2000:]
    line = json.loads([x for x in r.stdout.splitlines() if x.startswith("{")][-1])
    for key in ("metric", "value", "unit", "n_gpus", "steps", "warmup", "ms_per_step", "higher_is_better", "scaling",
                "vs_baseline", "dtype", "data", "config", "cpu_baseline", "e2e"):
        assert key in line, key
    assert line["impl"] == "reference" and line["steps"] == 3 and line["n_gpus"] == 1
    assert line["cpu_baseline"]["cores"] == 1 and line["cpu_baseline"]["cpu"]
    assert line["e2e"]["value"] == line["value"] and line["e2e"]["h2d_bytes_per_step"] == 0


def test_kernel_source_hash_ignores_comments_only():
    sys.path.insert(0, ROOT)
    import bench
    a = "int f(int x) { // add one\n  return x + 1; /* done */ }\n"
    b = "int f(int x) {\n    return x + 1;\n}\n"
    c = "int f(int x) { return x + 2; }"
    assert bench._code_only(a) == bench._code_only(b)
    assert bench._code_only(a) != bench._code_only(c)
    assert len(bench.kernel_source_hash()) == 16
