"""The benchmark's multi-GPU path (replicas, one process per GPU under torchrun)
exercised on CPU: two gloo ranks run the same coordination code the GPU runs
use -- rank-seeded weight sets, barriers around the timed region, the slowest
rank's time for every rank, one JSON line from rank 0 -- with no GPU."""

import contextlib
import io
import json
import os
import socket
import sys

import pytest

ROOT = os.path.dirname(os.path.dirname(os.path.abspath(__file__)))


def _free_port():
    with socket.socket() as s:
        s.bind(("127.0.0.1", 0))
        return s.getsockname()[1]


def _rank_main(rank, world, port, out_dir):
    os.environ.update(MASTER_ADDR="127.0.0.1", MASTER_PORT=str(port), RANK=str(rank),
                      WORLD_SIZE=str(world), LOCAL_RANK=str(rank))
    sys.path.insert(0, ROOT)
    import bench
    r, w, local = bench.dist_env()
    rep = bench.Replicas(r, w, local, backend="gloo")
    rep.barrier()
    slowest = rep.slowest(10.0 * (r + 1), "cpu")     # rank r "took" 10 (r + 1) ms
    rep.barrier()
    buf = io.StringIO()
    with contextlib.redirect_stdout(buf):
        rep.emit({"rank": r, "value": world * 1.0 / slowest})
    seeds = [rep.seed(1000, i) for i in range(4)]
    rep.close()
    with open(os.path.join(out_dir, "rank%d.json" % r), "w") as f:
        json.dump({"slowest": slowest, "printed": buf.getvalue(), "seeds": seeds}, f)


def test_two_gloo_ranks_share_the_slowest_time_and_print_once(tmp_path):
    mp = pytest.importorskip("torch.multiprocessing")
    pytest.importorskip("torch.distributed")
    world = 2
    mp.start_processes(_rank_main, args=(world, _free_port(), str(tmp_path)), nprocs=world,
                       join=True, start_method="spawn")
    res = [json.load(open(tmp_path / ("rank%d.json" % r))) for r in range(world)]
    assert [x["slowest"] for x in res] == [20.0, 20.0]
    assert json.loads(res[0]["printed"]) == {"rank": 0, "value": 0.1}
    assert res[1]["printed"] == ""
    seeds = res[0]["seeds"] + res[1]["seeds"]
    assert len(set(seeds)) == len(seeds)                # every rank and set its own weights


def test_single_process_needs_no_process_group():
    sys.path.insert(0, ROOT)
    import bench
    rep = bench.Replicas(0, 1, 0)
    assert rep.dist is None
    rep.barrier()
    assert rep.slowest(3.5, "cpu") == 3.5
    assert rep.seed(1000) == 1000 and rep.seed(1000, 1) == 1000 + 7919
    rep.close()


def test_reference_arm_on_other_ranks_exits_without_work(monkeypatch):
    sys.path.insert(0, ROOT)
    import bench
    monkeypatch.setattr(sys, "argv", ["bench.py", "--impl", "reference"])
    args = bench.parse_args()
    spec = bench.workload_spec(args)
    buf = io.StringIO()
    with contextlib.redirect_stdout(buf):
        assert bench.run_reference(args, spec, 1) == 0
    assert buf.getvalue() == ""
