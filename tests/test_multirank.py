"""The benchmark's multi-replica path, on CPU with gloo (world size 2).

On N GPUs bench.py runs one replica of the workload per GPU (the logical
ranks of the ring already live in one GPU's HBM), barriers around the timed
region, takes the slowest replica's time with an all-reduce MAX and reports
N x bytes / that time from rank 0.  These tests run the same helpers in two
gloo processes; the reference arm must print only on rank 0.
"""
import io
import contextlib
import os
import socket

import pytest
import torch
import torch.distributed as dist
import torch.multiprocessing as mp

from tests.conftest import ROOT


def _free_port():
    with socket.socket() as s:
        s.bind(("127.0.0.1", 0))
        return s.getsockname()[1]


def _worker(rank, world, port, q):
    os.environ.update(MASTER_ADDR="127.0.0.1", MASTER_PORT=str(port), RANK=str(rank), WORLD_SIZE=str(world))
    import sys
    sys.path.insert(0, ROOT)
    import bench
    dist.init_process_group("gloo", rank=rank, world_size=world)
    try:
        dist.barrier()
        ms = 1.0 + rank * 0.5                 # rank 1 is the slow replica
        ms_max = bench.max_over_ranks(ms, dist, "cpu")
        value = bench.replicas_value(world, 2.0e9, ms_max)
        args = bench.parse_args_for_tests(["--impl", "reference", "--gpus", str(world), "--steps", "1", "--warmup", "0"])
        spec = bench.workload_spec("f32_64mib", 8, 8 * 64)
        out = io.StringIO()
        with contextlib.redirect_stdout(out):
            rc = bench.run_reference(args, spec, rank, world)
        q.put((rank, ms_max, value, rc, out.getvalue()))
    finally:
        dist.destroy_process_group()


def test_replica_harness_two_gloo_ranks():
    ctx = mp.get_context("spawn")
    q = ctx.Queue()
    port = _free_port()
    procs = [ctx.Process(target=_worker, args=(r, 2, port, q)) for r in range(2)]
    for p in procs:
        p.start()
    res = sorted(q.get(timeout=300) for _ in procs)
    for p in procs:
        p.join(timeout=60)
        assert p.exitcode == 0
    for rank, ms_max, value, rc, out in res:
        assert ms_max == pytest.approx(1.5)                 # the slowest replica
        assert value == pytest.approx(2 * 2.0e9 / 1.5e-3 / 1e9)
        assert rc == 0
    assert '"impl": "reference"' in res[0][4]               # rank 0 prints the line
    assert res[1][4] == ""                                  # other ranks exit without work
    import json
    line = json.loads(res[0][4].strip().splitlines()[-1])
    for key in ("metric", "value", "unit", "n_gpus", "steps", "warmup", "ms_per_step", "higher_is_better",
                "scaling", "vs_baseline", "dtype", "data", "config", "cpu_baseline", "e2e"):
        assert key in line, key
    assert line["n_gpus"] == 2 and line["higher_is_better"] is True and line["vs_baseline"] is None
    assert line["cpu_baseline"]["kind"] == "oracle" and line["cpu_baseline"]["value"] == line["value"]
    assert line["e2e"]["h2d_bytes_per_step"] == 0 and line["e2e"]["d2h_bytes_per_step"] == 0
    assert line["e2e"]["value"] == line["value"] and line["e2e"]["unit"] == line["unit"]
    assert "workload" in line["config"]
