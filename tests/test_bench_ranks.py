"""bench.py's multi-rank host logic on CPU with two gloo ranks (no GPU).

Replicas run independent work with no data-path collective; the only
exchange is the timing: every rank takes the slowest rank's time, and rank 0
alone prints.  Rendezvous is on 127.0.0.1.
"""
import json
import os
import socket
import subprocess
import sys

import pytest

torch = pytest.importorskip("torch")

ROOT = os.path.dirname(os.path.dirname(os.path.abspath(__file__)))


def free_port() -> int:
    s = socket.socket()
    s.bind(("127.0.0.1", 0))
    port = s.getsockname()[1]
    s.close()
    return port


def _rank_main(rank, ws, port, q):
    os.environ.update(MASTER_ADDR="127.0.0.1", MASTER_PORT=str(port), RANK=str(rank), WORLD_SIZE=str(ws),
                      LOCAL_RANK=str(rank))
    sys.path.insert(0, ROOT)
    import bench
    try:
        bench.init_dist(ws)
        assert torch.distributed.get_backend() == "gloo"
        got = bench.max_over_ranks(10.0 * (rank + 1), ws, "cpu")
        torch.distributed.barrier()
        torch.distributed.destroy_process_group()
        q.put((rank, got, bench.dist_env()))
    except Exception as e:  # reported to the parent rather than hanging it
        q.put((rank, repr(e), None))


def test_two_gloo_ranks_take_the_slowest_rank_time():
    import torch.multiprocessing as mp
    ctx = mp.get_context("spawn")
    q = ctx.Queue()
    port = free_port()
    procs = [ctx.Process(target=_rank_main, args=(r, 2, port, q)) for r in range(2)]
    for p in procs:
        p.start()
    try:
        res = sorted(q.get(timeout=180) for _ in range(2))
    finally:
        for p in procs:
            p.join(timeout=60)
            if p.is_alive():
                p.kill()
    assert [p.exitcode for p in procs] == [0, 0]
    assert [r[1] for r in res] == [20.0, 20.0], res
    assert [r[2] for r in res] == [(2, 0, 0), (2, 1, 1)]


def test_single_rank_needs_no_process_group():
    sys.path.insert(0, ROOT)
    import bench
    assert bench.max_over_ranks(3.5, 1, "cpu") == 3.5


def test_reference_arm_under_two_ranks_prints_one_line_from_rank_0():
    port = free_port()
    cmd = [sys.executable, "-m", "torch.distributed.run", "--nnodes=1", "--nproc-per-node", "2",
           "--master-addr", "127.0.0.1", "--master-port", str(port),
           "bench.py", "--impl", "reference", "--config", "tiny", "--gpus", "2", "--steps", "2", "--warmup", "1"]
    env = dict(os.environ, OMP_NUM_THREADS="2")
    r = subprocess.run(cmd, cwd=ROOT, capture_output=True, text=True, timeout=600, env=env)
    assert r.returncode == 0, r.stderr[-3000:]
    lines = [ln for ln in r.stdout.splitlines() if ln.startswith("{")]
    assert len(lines) == 1, r.stdout[-3000:]
    d = json.loads(lines[0])
    assert d["impl"] == "reference" and d["value"] > 0
    assert d["cpu_baseline"]["kind"] == "oracle" and d["e2e"]["h2d_bytes_per_step"] == 0


def test_reference_arm_on_the_prefill_workload_reports_the_gpu_arms_unit():
    r = subprocess.run([sys.executable, "bench.py", "--config", "prefill_35b", "--impl", "reference",
                        "--steps", "1", "--warmup", "0"], cwd=ROOT, capture_output=True, text=True, timeout=600)
    assert r.returncode == 0, r.stderr[-3000:]
    d = json.loads([ln for ln in r.stdout.splitlines() if ln.startswith("{")][-1])
    assert d["impl"] == "reference" and d["unit"] == "TFLOP/s" and d["value"] > 0
    assert d["config"]["workload"] == "prefill_35b" and d["cpu_baseline"]["kind"] == "oracle"


def test_reference_arm_keeps_each_steps_experts_when_its_store_is_full():
    """The oracle's store of quantised experts is bounded: evicting the least recently used never drops an expert
    the current step routes to, over more steps than the store holds."""
    sys.path.insert(0, ROOT)
    import bench
    import workloads as W
    cfg = W.scaled(W.CONFIGS["tiny"], layers=3)
    ref = bench.OracleToken(cfg, keep=2)
    for s in range(6):
        assert ref.step(s) >= 0.0
        assert len(ref.q) <= max(2, cfg.layers * min(cfg.E, cfg.T * cfg.k))


def test_reference_arm_stops_at_its_time_budget(monkeypatch):
    """Asked for more steps than fit the budget, the reference arm times whole steps until the budget is spent and
    reports how many it timed and how many were asked."""
    sys.path.insert(0, ROOT)
    import bench
    monkeypatch.setattr(bench, "REF_BUDGET_S", 0.0)
    monkeypatch.setattr(sys, "argv", ["bench.py", "--impl", "reference", "--config", "tiny", "--steps", "50",
                                      "--warmup", "0"])
    import contextlib
    import io
    out = io.StringIO()
    with contextlib.redirect_stdout(out):
        bench.main()
    d = json.loads([ln for ln in out.getvalue().splitlines() if ln.startswith("{")][-1])
    assert d["steps"] == 1 and d["steps_requested"] == 50 and d["value"] > 0
