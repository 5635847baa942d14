"""The multi-rank path of bench.py on CPU (gloo, world size 2): ranks are
independent replicas, the step time is the max over ranks, the job value counts
every rank's pseudo-tokens, and the reference arm runs on rank 0 only."""
import argparse
import io
import json
import multiprocessing as mp
import os
import socket
import sys
from contextlib import redirect_stdout

import pytest

from conftest import ROOT


def _free_port():
    with socket.socket() as s:
        s.bind(("127.0.0.1", 0))
        return s.getsockname()[1]


def _env(rank, world, port):
    os.environ.update(RANK=str(rank), WORLD_SIZE=str(world), LOCAL_RANK=str(rank),
                      MASTER_ADDR="127.0.0.1", MASTER_PORT=str(port))
    if ROOT not in sys.path:
        sys.path.insert(0, ROOT)


def _timing_worker(rank, world, port, q):
    _env(rank, world, port)
    import torch
    import bench
    r, w, local, dist = bench.dist_setup(world)
    m = bench.max_over_ranks(1.5 + rank, dist, torch.device("cpu"))
    bench.barrier(dist)
    q.put((rank, r, w, m, bench.job_value(w, 1000, m)))
    dist.destroy_process_group()


def _reference_worker(rank, world, port, q):
    _env(rank, world, port)
    import bench
    import iha_inputs as gi
    args = argparse.Namespace(gpus=world, steps=1, warmup=3, ref_tokens=4)
    buf = io.StringIO()
    with redirect_stdout(buf):
        bench.run_reference(args, gi.WORKLOADS["tiny_f32_nomask"])
    q.put((rank, buf.getvalue()))


def _run(target, world=2):
    ctx = mp.get_context("spawn")
    q = ctx.Queue()
    port = _free_port()
    ps = [ctx.Process(target=target, args=(r, world, port, q)) for r in range(world)]
    for p in ps:
        p.start()
    out = [q.get(timeout=120) for _ in ps]
    for p in ps:
        p.join(timeout=60)
        assert p.exitcode == 0
    return sorted(out)


def test_two_ranks_take_the_max_step_time_and_count_both_replicas():
    out = _run(_timing_worker)
    for rank, r, w, m, value in out:
        assert r == rank and w == 2
        assert m == 2.5                        # max(1.5, 2.5)
        assert value == pytest.approx(2 * 1000 / 2.5e-3)


def test_reference_arm_prints_on_rank_zero_only():
    out = _run(_reference_worker)
    (r0, text0), (r1, text1) = out
    assert r0 == 0 and r1 == 1
    assert text1.strip() == ""
    line = json.loads(text0.strip().splitlines()[-1])
    assert line["impl"] == "reference" and line["cpu_baseline"]["kind"] == "oracle"
    assert line["value"] > 0 and line["e2e"]["h2d_bytes_per_step"] == 0
