"""Multi-rank plumbing of bench.py on CPU (gloo, world size 2).

The decode path shards over the batch with no collective: every rank runs an
independent replica and the bench takes the slowest rank's time.  These tests
cover the host side of that on CPU: rendezvous, the barrier, the max-over-ranks
reduction, the whole-job aggregation, and that only rank 0 runs the reference
arm.  No GPU is touched.
"""
import importlib.util
import json
import os
import socket
import sys

import numpy as np
import pytest
import torch.multiprocessing as mp

ROOT = os.path.dirname(os.path.dirname(os.path.abspath(__file__)))


def _load_bench():
    spec = importlib.util.spec_from_file_location("bench_under_test", os.path.join(ROOT, "bench.py"))
    mod = importlib.util.module_from_spec(spec)
    sys.path.insert(0, ROOT)
    spec.loader.exec_module(mod)
    return mod


def _free_port() -> int:
    with socket.socket() as s:
        s.bind(("127.0.0.1", 0))
        return s.getsockname()[1]


def _rank_main(rank, world, port, q):
    os.environ.update({"WORLD_SIZE": str(world), "RANK": str(rank), "LOCAL_RANK": str(rank),
                       "MASTER_ADDR": "127.0.0.1", "MASTER_PORT": str(port),
                       "MLA_BENCH_BACKEND": "gloo"})
    bench = _load_bench()
    r, w, local, dist = bench.dist_setup(world)
    try:
        bench.barrier(dist, None)
        # each rank "timed" a different duration; the job time is the slowest
        t = bench.max_over_ranks(dist, 1.5 + rank)
        # whole-job throughput: units of all ranks over the slowest rank's time
        units_per_rank = 1000
        value = units_per_rank * w / t
        q.put((r, w, local, t, value))
    finally:
        dist.destroy_process_group()


def test_two_rank_gloo_max_and_aggregate():
    ctx = mp.get_context("spawn")
    q = ctx.Queue()
    port = _free_port()
    procs = [ctx.Process(target=_rank_main, args=(r, 2, port, q)) for r in range(2)]
    for p in procs:
        p.start()
    for p in procs:
        p.join(timeout=120)
    assert all(p.exitcode == 0 for p in procs)
    got = sorted(q.get(timeout=5) for _ in range(2))
    assert [g[0] for g in got] == [0, 1]
    for r, w, local, t, value in got:
        assert w == 2 and local == r
        assert t == pytest.approx(2.5)              # max over ranks
        assert value == pytest.approx(2000 / 2.5)   # both ranks' units / slowest time


def test_world_size_mismatch_is_rejected(monkeypatch):
    bench = _load_bench()
    monkeypatch.setenv("WORLD_SIZE", "2")
    with pytest.raises(SystemExit):
        bench.dist_setup(1)


def test_reference_arm_runs_on_rank_zero_only(monkeypatch, capsys):
    bench = _load_bench()
    monkeypatch.setenv("RANK", "1")
    args = bench.argparse.Namespace(gpus=2, steps=1, warmup=3, impl="reference",
                                    workload=bench.mi.V2_DECODE.name, cpu_budget=1.0,
                                    no_cpu_baseline=True)
    assert bench.run_reference(args, bench.mi.V2_DECODE) == 0
    assert capsys.readouterr().out == ""       # no work, no line on the other ranks


def test_prefill_flop_count_matches_brute_force():
    bench = _load_bench()
    spec = bench.mi.PrefillSpec("tiny", seed=0, B=2, H=3, T_q=4, seqlens=(4, 9), d_h=8, d_c=16, d_r=4)
    seqlens = np.array(spec.seqlens, dtype=np.int32)
    w = bench.prefill_work(spec, seqlens)
    rebuild = sum(L * spec.H * 2 * (2 * spec.d_c * spec.d_h) for L in spec.seqlens)
    attn = 0
    for L in spec.seqlens:
        for t in range(spec.T_q):
            for s in range(L):
                if s <= L - spec.T_q + t:        # causal: keys up to the query's position
                    attn += spec.H * (2 * (spec.d_h + spec.d_r) + 2 * spec.d_h)
    assert w["rebuild_flops"] == rebuild and w["attn_flops"] == attn
    assert w["flops"] == rebuild + attn


def test_prefill_reference_arm_rank_zero_only_and_line(monkeypatch, capsys):
    bench = _load_bench()
    spec = bench.mi.PrefillSpec("tiny_prefill", seed=3, B=1, H=2, T_q=40, seqlens=(70,))
    args = bench.argparse.Namespace(gpus=2, steps=1, warmup=3, impl="reference",
                                    workload=spec.name, cpu_budget=1.0, no_cpu_baseline=True)
    monkeypatch.setenv("RANK", "1")
    assert bench.run_prefill_reference(args, spec) == 0
    assert capsys.readouterr().out == ""
    monkeypatch.setenv("RANK", "0")
    assert bench.run_prefill_reference(args, spec) == 0
    line = json.loads(capsys.readouterr().out)
    assert line["impl"] == "reference" and line["unit"] == "TFLOP/s" and line["value"] > 0
    assert line["cpu_baseline"]["kind"] == "oracle" and line["e2e"]["h2d_bytes_per_step"] == 0
