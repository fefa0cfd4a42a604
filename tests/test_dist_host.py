"""The N > 1 path of bench.py on the host: two gloo ranks on CPU.

Every (b, h) is independent, so replicas run with no collective on the data
path; the only cross-rank steps are the barrier around the timed region and
the max of the step time over ranks.  Checked here with world_size 2.
"""
import json
import os
import socket
import sys
import types

import pytest
import torch.multiprocessing as mp

ROOT = os.path.dirname(os.path.dirname(os.path.abspath(__file__)))


def _free_port():
    s = socket.socket()
    s.bind(("127.0.0.1", 0))
    port = s.getsockname()[1]
    s.close()
    return port


def _worker(rank, world, port, outdir):
    os.environ.update({"MASTER_ADDR": "127.0.0.1", "MASTER_PORT": str(port), "WORLD_SIZE": str(world),
                       "RANK": str(rank), "LOCAL_RANK": str(rank)})
    sys.path.insert(0, ROOT)
    import bench
    import torch.distributed as dist
    r, w, local, pg = bench.dist_setup(types.SimpleNamespace(gpus=world))
    # per-rank step times; the job time is the slowest rank's
    ms = 10.0 + 3.0 * r
    bench.barrier(pg)
    ms_max = bench.max_over_ranks(ms, pg)
    value = bench.weak_scaling_value(w, 117.05e12, ms_max)
    with open(os.path.join(outdir, "rank%d.json" % r), "w") as f:
        json.dump({"rank": r, "world": w, "local": local, "pg": pg, "ms_max": ms_max, "value": value,
                   "backend": dist.get_backend()}, f)
    dist.destroy_process_group()


def test_two_gloo_ranks_max_and_value(tmp_path):
    world = 2
    mp.spawn(_worker, args=(world, _free_port(), str(tmp_path)), nprocs=world, join=True)
    res = [json.load(open(tmp_path / ("rank%d.json" % r))) for r in range(world)]
    for r, d in enumerate(res):
        assert d["rank"] == r and d["world"] == world and d["local"] == r and d["pg"] is True
        assert d["backend"] == "gloo"
        assert d["ms_max"] == 13.0                      # max over ranks, identical everywhere
        assert d["value"] == pytest.approx(2 * 117.05e12 / 13e-3 / 1e12)


def test_single_rank_is_identity():
    sys.path.insert(0, ROOT)
    import bench
    assert bench.max_over_ranks(4.5, False) == 4.5
    assert bench.weak_scaling_value(1, 1e12, 1000.0) == pytest.approx(1.0)   # 1e12 flop in 1 s


def test_reference_arm_only_rank0_works(monkeypatch, capsys):
    sys.path.insert(0, ROOT)
    import bench
    monkeypatch.setenv("RANK", "1")
    bench.run_reference(types.SimpleNamespace(gpus=2, steps=1, warmup=0))
    assert capsys.readouterr().out == ""
