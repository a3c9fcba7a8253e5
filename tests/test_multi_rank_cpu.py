"""The multi-rank path of bench.py on CPU: two gloo ranks on 127.0.0.1.

The hot path has no exchange step, so several GPUs run independent replicas;
the ranks only meet to time (barrier, then the slowest rank's time) and rank 0
alone prints. This checks that logic without a GPU: the max over ranks, the
whole-job throughput formula, and that the reference arm prints on rank 0 only
and exits 0 on the others.
"""
import contextlib
import io
import json
import multiprocessing as mp
import os
import socket
import sys
import types

import pytest

ROOT = os.path.dirname(os.path.dirname(os.path.abspath(__file__)))


def _free_port():
    with socket.socket() as s:
        s.bind(("127.0.0.1", 0))
        return s.getsockname()[1]


def _worker(rank, world, port, out):
    os.environ.update(MASTER_ADDR="127.0.0.1", MASTER_PORT=str(port), RANK=str(rank), WORLD_SIZE=str(world),
                      LOCAL_RANK=str(rank))
    sys.path.insert(0, ROOT)
    import torch.distributed as tdist

    import bench

    tdist.init_process_group("gloo", rank=rank, world_size=world)
    try:
        slowest = bench.max_over_ranks(1.0 + rank, world)
        tdist.barrier()
        args = types.SimpleNamespace(workload="tiny_decode", warmup=1, steps=2, gpus=world, impl="reference")
        buf = io.StringIO()
        with contextlib.redirect_stdout(buf):
            rc = bench.run_reference(args)
        tdist.barrier()
        out.put((rank, slowest, rc, buf.getvalue()))
    finally:
        tdist.destroy_process_group()


def test_two_gloo_ranks_replica_timing_and_reference_arm():
    world = 2
    ctx = mp.get_context("spawn")
    out = ctx.Queue()
    port = _free_port()
    procs = [ctx.Process(target=_worker, args=(r, world, port, out)) for r in range(world)]
    for p in procs:
        p.start()
    res = {}
    try:
        for _ in range(world):
            rank, slowest, rc, text = out.get(timeout=240)
            res[rank] = (slowest, rc, text)
    finally:
        for p in procs:
            p.join(timeout=60)
            if p.is_alive():
                p.kill()
    assert all(p.exitcode == 0 for p in procs)
    # every rank sees the slowest rank's time
    assert res[0][0] == res[1][0] == pytest.approx(2.0)
    # both ranks exit 0; only rank 0 prints, one JSON line
    assert res[0][1] == 0 and res[1][1] == 0
    assert res[1][2] == ""
    lines = [l for l in res[0][2].splitlines() if l.strip()]
    assert len(lines) == 1
    d = json.loads(lines[0])
    assert d["impl"] == "reference" and d["n_gpus"] == world and d["steps"] == 2
    assert d["cpu_baseline"]["kind"] == "oracle" and d["cpu_baseline"]["value"] == d["value"] > 0
    assert d["e2e"]["h2d_bytes_per_step"] == 0 and d["e2e"]["d2h_bytes_per_step"] == 0


def test_replica_throughput_counts_every_rank():
    sys.path.insert(0, ROOT)
    import bench

    # 4 replicas x 3 steps x 32 tokens in (at most) 0.5 s
    assert bench.replica_throughput(32, 3, 4, 0.5) == pytest.approx(32 * 3 * 4 / 0.5)
    assert bench.max_over_ranks(0.25, 1) == 0.25
