"""Replica aggregation of the benchmark on CPU: two gloo ranks, each timing its
own replica, agree on the slowest rank's time and the whole-job throughput."""
import os
import socket

import pytest
import torch.multiprocessing as mp


def _free_port():
    with socket.socket() as s:
        s.bind(("127.0.0.1", 0))
        return s.getsockname()[1]


def _rank_main(rank, world, port, out):
    import torch.distributed as dist
    import bench
    os.environ.update(MASTER_ADDR="127.0.0.1", MASTER_PORT=str(port))
    dist.init_process_group("gloo", rank=rank, world_size=world)
    my_ms = [12.5, 20.0][rank]
    ms = bench.max_over_ranks(my_ms, world, "cpu")
    line = bench.headline(100, 1, world, ms)
    assert line["n_gpus"] == world and line["scaling"] == "weak"
    assert line["ms_per_step"] == ms / 100
    out[rank] = (ms, line["value"])
    dist.barrier()
    dist.destroy_process_group()


def test_two_replicas_agree_on_max_time_and_job_throughput():
    ctx = mp.get_context("spawn")
    mgr = ctx.Manager()
    out = mgr.dict()
    port = _free_port()
    procs = [ctx.Process(target=_rank_main, args=(r, 2, port, out)) for r in range(2)]
    for p in procs:
        p.start()
    for p in procs:
        p.join(120)
        assert p.exitcode == 0
    assert out[0] == out[1] == (20.0, 100 * 1 * 2 / 0.02)


def test_launch_plan_for_gpus():
    import bench
    # no launcher: one GPU runs in place, N GPUs re-launch as N local ranks
    assert bench.launch_plan(1, {}, ["--steps", "5"]) == ("single", None)
    mode, cmd = bench.launch_plan(2, {}, ["--gpus", "2", "--steps", "5"], port=29555)
    assert mode == "spawn"
    assert cmd[1:3] == ["-m", "torch.distributed.run"]
    assert cmd[cmd.index("--nproc-per-node") + 1] == "2"
    assert cmd[cmd.index("--master-addr") + 1] == "127.0.0.1"
    assert cmd[-5] == os.path.abspath(bench.__file__)
    assert cmd[-4:] == ["--gpus", "2", "--steps", "5"]
    # under a launcher: one process per rank, and --gpus must match its world size
    assert bench.launch_plan(2, {"WORLD_SIZE": "2"}, []) == ("ranks", None)
    assert bench.launch_plan(1, {"WORLD_SIZE": "1"}, []) == ("single", None)
    with pytest.raises(SystemExit):
        bench.launch_plan(2, {"WORLD_SIZE": "4"}, [])


def test_single_rank_is_its_own_time():
    import bench
    assert bench.max_over_ranks(3.0, 1) == 3.0
    assert bench.job_throughput(10, 4, 1, 1000.0) == pytest.approx(40.0)
