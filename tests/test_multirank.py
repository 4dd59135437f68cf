"""Multi-rank path on CPU (gloo, world size 2).

Under torchrun each rank owns a contiguous range of experts of the stack and
prepares and decodes that sub-stack on its own GPU (no data-path collective);
the only cross-rank steps are a barrier and the max over ranks of the timed
region.  These tests run the shard assignment (expert ranges and routing
views) and that reduction on two gloo ranks, and launch the reference arm
under torchrun with two ranks (rank 0 alone prints)."""
import json
import os
import socket
import subprocess
import sys

import pytest
import torch
import torch.distributed as dist
import torch.multiprocessing as mp

ROOT = os.path.dirname(os.path.dirname(os.path.abspath(__file__)))


def _free_port():
    with socket.socket() as s:
        s.bind(("127.0.0.1", 0))
        return s.getsockname()[1]


def _worker(rank, world, port, out):
    os.environ.update(MASTER_ADDR="127.0.0.1", MASTER_PORT=str(port))
    dist.init_process_group("gloo", rank=rank, world_size=world)
    sys.path.insert(0, ROOT)
    import bench
    dist.barrier()
    got = bench.reduce_max(torch, dist, 10.0 + 3.5 * rank, "cpu")
    out[rank] = got
    dist.destroy_process_group()


def test_reduce_max_over_two_gloo_ranks():
    port = _free_port()
    with mp.Manager() as m:
        out = m.dict()
        mp.spawn(_worker, args=(2, port, out), nprocs=2, join=True)
        assert dict(out) == {0: 13.5, 1: 13.5}


def _shard_worker(rank, world, port, out):
    os.environ.update(MASTER_ADDR="127.0.0.1", MASTER_PORT=str(port))
    dist.init_process_group("gloo", rank=rank, world_size=world)
    sys.path.insert(0, ROOT)
    from lossless_nvfp4_scale_gb300 import shard, synth
    E = 37                                          # not a multiple of the world size
    dense = torch.from_numpy(synth.random_rows(5, E * 3, 8).reshape(E, 3, 8))
    start = torch.from_numpy(synth.routing(E=E, active=6, tokens=20, seed=2))
    e0, e1 = shard.expert_range(E, world, rank)
    sub = shard.shard_dense(dense, e0, e1)
    view = shard.routing_view(start, e0, e1)
    # every rank's pieces, gathered on every rank
    ranges = [None] * world
    dist.all_gather_object(ranges, (e0, e1))
    subs = [None] * world
    dist.all_gather_object(subs, sub.clone())
    views = [None] * world
    dist.all_gather_object(views, view.clone())
    ok_partition = ranges[0][0] == 0 and ranges[-1][1] == E and all(
        a[1] == b[0] and a[0] < a[1] for a, b in zip(ranges, ranges[1:]))
    ok_dense = torch.equal(torch.cat(subs), dense)
    # a rank's routing view marks exactly its own experts' activity
    active = (start[1:] > start[:-1])
    ok_views = all(torch.equal(v[1:] > v[:-1], active[r0:r1]) and v.shape[0] == r1 - r0 + 1
                   for v, (r0, r1) in zip(views, ranges))
    ok_ptr = view.data_ptr() == start.data_ptr() + e0 * start.element_size()
    out[rank] = (ranges, ok_partition, ok_dense, ok_views, ok_ptr)
    dist.destroy_process_group()


def test_shard_assignment_over_two_gloo_ranks():
    port = _free_port()
    with mp.Manager() as m:
        out = m.dict()
        mp.spawn(_shard_worker, args=(2, port, out), nprocs=2, join=True)
        res = dict(out)
    assert res[0][0] == res[1][0] == [(0, 19), (19, 37)]
    for rank in (0, 1):
        assert res[rank][1:] == (True, True, True, True)


def test_expert_range_partitions():
    import importlib
    shard = importlib.import_module("lossless_nvfp4_scale_gb300.shard")
    for E in (1, 7, 8, 384, 512):
        for world in range(1, min(E, 9) + 1):
            rs = [shard.expert_range(E, world, r) for r in range(world)]
            assert rs[0][0] == 0 and rs[-1][1] == E
            sizes = [b - a for a, b in rs]
            assert max(sizes) - min(sizes) <= 1 and min(sizes) >= 1
            assert all(a[1] == b[0] for a, b in zip(rs, rs[1:]))
    with pytest.raises(ValueError):
        shard.expert_range(4, 8, 0)


def test_reference_arm_under_torchrun_prints_once():
    port = _free_port()
    cmd = [sys.executable, "-m", "torch.distributed.run", "--nnodes=1", "--nproc-per-node", "2",
           "--master-addr", "127.0.0.1", "--master-port", str(port),
           os.path.join(ROOT, "bench.py"), "--impl", "reference", "--gpus", "2", "--steps", "1",
           "--warmup", "3"]
    r = subprocess.run(cmd, capture_output=True, text=True, cwd=ROOT, timeout=300)
    assert r.returncode == 0, r.stderr[-2000:]
    lines = [ln for ln in r.stdout.splitlines() if ln.startswith("{")]
    assert len(lines) == 1
    d = json.loads(lines[0])
    assert d["impl"] == "reference" and d["cpu_baseline"]["kind"] == "oracle"
    assert d["unit"] == "GB/s" and d["higher_is_better"] is True
