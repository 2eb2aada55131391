"""The N > 1 host logic of bench.py on CPU: two gloo ranks.

Every call of the library runs on one GPU; `bench.py --gpus N` runs N
independent replicas (one process per GPU) and reports the whole job: the
slowest rank's time (max over ranks) and the work of all ranks.  These tests
run that logic with world size 2 on the gloo backend, and the reference arm's
rule that only rank 0 works and prints.
"""
import importlib.util
import io
import json
import os
import socket
import contextlib

import pytest

ROOT = os.path.dirname(os.path.dirname(os.path.abspath(__file__)))


def _bench():
    spec = importlib.util.spec_from_file_location("bench_under_test", os.path.join(ROOT, "bench.py"))
    mod = importlib.util.module_from_spec(spec)
    spec.loader.exec_module(mod)
    return mod


def _free_port():
    with socket.socket() as s:
        s.bind(("127.0.0.1", 0))
        return s.getsockname()[1]


def _rank_main(rank, world, port, out_q):
    import torch
    import torch.distributed as dist
    os.environ.update(MASTER_ADDR="127.0.0.1", MASTER_PORT=str(port))
    dist.init_process_group("gloo", rank=rank, world_size=world)
    try:
        bench = _bench()
        dev = torch.device("cpu")
        dist.barrier()
        local_ms = [12.5, 30.0][rank]
        got = bench.max_over_ranks(local_ms, world, dev)
        tf = bench.whole_job_tflops(world, 6.0e9, got)
        out_q.put((rank, got, tf))
        dist.barrier()
    finally:
        dist.destroy_process_group()


def test_max_over_ranks_and_whole_job_value_with_two_gloo_ranks():
    import torch.multiprocessing as mp
    ctx = mp.get_context("spawn")
    q = ctx.Queue()
    port = _free_port()
    procs = [ctx.Process(target=_rank_main, args=(r, 2, port, q)) for r in range(2)]
    for p in procs:
        p.start()
    for p in procs:
        p.join(timeout=120)
    assert all(p.exitcode == 0 for p in procs), [p.exitcode for p in procs]
    res = sorted(q.get(timeout=10) for _ in range(2))
    for rank, got, tf in res:
        # both ranks see the slower rank's time; the value counts both ranks' work
        assert got == 30.0, (rank, got)
        assert tf == pytest.approx(2 * 6.0e9 / 30.0e-3 / 1e12)


def test_single_rank_needs_no_process_group():
    bench = _bench()
    assert bench.max_over_ranks(7.0, 1, None) == 7.0
    assert bench.whole_job_tflops(1, 1.0e12, 1000.0) == pytest.approx(1.0)


def test_reference_arm_runs_on_rank_zero_only(monkeypatch):
    """Under torchrun only rank 0 runs the oracle and prints one JSON line;
    the other ranks return 0 without work or output."""
    bench = _bench()
    args = bench.main.__globals__["argparse"].Namespace(steps=1, warmup=0, ref_budget=0.5)
    w = bench.fa_inputs.WORKLOADS["s256"]
    monkeypatch.setenv("WORLD_SIZE", "2")
    monkeypatch.setenv("RANK", "1")
    buf = io.StringIO()
    with contextlib.redirect_stdout(buf):
        assert bench.run_reference(args, w) == 0
    assert buf.getvalue() == ""
    monkeypatch.setenv("RANK", "0")
    buf = io.StringIO()
    with contextlib.redirect_stdout(buf):
        assert bench.run_reference(args, w) == 0
    lines = [l for l in buf.getvalue().splitlines() if l.strip()]
    assert len(lines) == 1
    line = json.loads(lines[0])
    assert line["impl"] == "reference" and line["n_gpus"] == 2
    assert line["value"] > 0 and line["e2e"]["h2d_bytes_per_step"] == 0
