"""The benchmark's multi-rank path on CPU: two gloo ranks, each with its own
replica, exactly as torchrun launches bench.py with --gpus 2 (no collective in
the data path; only the barrier and the max-over-ranks timing reduction)."""
import json
import os
import socket
import subprocess
import sys

import pytest

from conftest import ROOT


def _free_port():
    with socket.socket() as s:
        s.bind(("127.0.0.1", 0))
        return s.getsockname()[1]


WORKER = r"""
import json, os, sys
sys.path.insert(0, {root!r})
import torch.distributed as dist
dist.init_process_group("gloo", init_method="env://")
import bench
world, rank, local = bench.dist_setup()
assert (world, rank, local) == (2, int(os.environ["RANK"]), int(os.environ["LOCAL_RANK"]))
bench.barrier(world)
slowest = bench.max_over_ranks(1.5 if rank == 0 else 2.5, world, "cpu")
rate = bench.aggregate_rate(world, 14336, 1024, slowest)
print(json.dumps({{"rank": rank, "slowest": slowest, "rate": rate}}), flush=True)
dist.destroy_process_group()
"""


def _launch(code, extra_env=None):
    port = _free_port()
    procs = []
    for rank in range(2):
        env = dict(os.environ, MASTER_ADDR="127.0.0.1", MASTER_PORT=str(port),
                   RANK=str(rank), LOCAL_RANK=str(rank), WORLD_SIZE="2")
        env.update(extra_env or {})
        procs.append(subprocess.Popen([sys.executable, "-c", code], env=env,
                                      stdout=subprocess.PIPE, stderr=subprocess.PIPE,
                                      text=True, cwd=ROOT))
    outs = [p.communicate(timeout=240) for p in procs]
    for p, (o, e) in zip(procs, outs):
        assert p.returncode == 0, e
    return [o for o, _ in outs]


def test_two_rank_barrier_and_max_reduction():
    outs = _launch(WORKER.format(root=ROOT))
    lines = [json.loads(o.strip().splitlines()[-1]) for o in outs]
    for ln in lines:
        assert ln["slowest"] == 2.5          # both ranks see the slowest rank
        assert ln["rate"] == pytest.approx(2 * 14336 * 1024 / 2.5)
    assert sorted(ln["rank"] for ln in lines) == [0, 1]


def test_reference_arm_prints_on_rank_zero_only():
    """`bench.py --impl reference` under two ranks: rank 0 times the oracle
    on a bounded sample and prints one JSON line; rank 1 exits 0 silently."""
    code = (f"import sys; sys.path.insert(0, {ROOT!r}); "
            "sys.argv = ['bench.py', '--impl', 'reference', '--gpus', '2', "
            "'--steps', '3', '--warmup', '3', '--workload', 'single', "
            "'--ref-groups', '1']; import bench; bench.main()")
    outs = _launch(code)
    line = json.loads(outs[0].strip().splitlines()[-1])
    assert line["impl"] == "reference" and line["unit"] == "group-steps/s"
    assert line["n_gpus"] == 2 and line["value"] > 0
    assert line["e2e"]["h2d_bytes_per_step"] == 0
    assert line["cpu_baseline"]["kind"] == "oracle"
    assert outs[1].strip() == ""
