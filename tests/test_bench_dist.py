"""bench.py's multi-rank host logic on CPU (gloo, world size 2): each rank
times its own replica of the workload; the job time is the maximum over
ranks and the work is the sum (weak scaling, no data-path collective)."""
import json
import os
import socket
import subprocess
import sys

import pytest

ROOT = os.path.dirname(os.path.dirname(os.path.abspath(__file__)))

WORKER = r"""
import os, sys, json
sys.path.insert(0, {root!r})
import torch.distributed as dist
import bench
dist.init_process_group("gloo")
rank, world = dist.get_rank(), dist.get_world_size()
# rank r pretends its replica took (r + 1) seconds for (r + 1) * 10 FLOP
t, f = bench.aggregate(float(rank + 1), float((rank + 1) * 10), world)
bench.barrier(world)
print(json.dumps({{"rank": rank, "t": t, "f": f}}), flush=True)
dist.destroy_process_group()
"""


def _free_port():
    with socket.socket() as s:
        s.bind(("127.0.0.1", 0))
        return s.getsockname()[1]


def test_aggregate_max_time_sum_work_gloo():
    port = _free_port()
    procs = []
    for r in range(2):
        env = dict(os.environ, MASTER_ADDR="127.0.0.1", MASTER_PORT=str(port), RANK=str(r),
                   WORLD_SIZE="2", LOCAL_RANK=str(r))
        procs.append(subprocess.Popen([sys.executable, "-c", WORKER.format(root=ROOT)], env=env,
                                      stdout=subprocess.PIPE, stderr=subprocess.PIPE, text=True))
    outs = []
    for p in procs:
        out, err = p.communicate(timeout=120)
        assert p.returncode == 0, err
        outs.append(json.loads(out.strip().splitlines()[-1]))
    for o in outs:
        assert o["t"] == 2.0 and o["f"] == 30.0


def test_single_rank_aggregate_is_identity():
    sys.path.insert(0, ROOT)
    import bench
    assert bench.aggregate(1.5, 7.0, 1) == (1.5, 7.0)


def test_reference_arm_on_other_ranks_prints_nothing(monkeypatch, capsys):
    sys.path.insert(0, ROOT)
    import bench
    monkeypatch.setenv("RANK", "1")
    monkeypatch.setenv("WORLD_SIZE", "2")
    assert bench.main(["--impl", "reference", "--workload", "tiny", "--steps", "1",
                       "--warmup", "3"]) == 0
    assert capsys.readouterr().out == ""


def test_make_workload_default_c_tile():
    """Every bench workload resolves; the per-tile cost defaults from its head dim."""
    sys.path.insert(0, ROOT)
    import types
    import bench
    from packed_varlen_attention_cu_gb300 import api
    for name in bench.WORKLOADS:
        args = types.SimpleNamespace(workload=name, pack_tokens=0, c_tile=None)
        w, desc = bench.make_workload(args)
        assert args.c_tile == api.default_c_tile(w.head_dim) == 32768 * 128 // w.head_dim
        assert desc
    args = types.SimpleNamespace(workload="128k", pack_tokens=32768, c_tile=777)
    w, _ = bench.make_workload(args)
    assert w.total_tokens == 32768 and args.c_tile == 777
