"""The replica path of bench.py across two ranks, on CPU with the gloo backend.

With N GPUs every rank runs its own replica of the call; the job takes as long as its
slowest rank, so the timing fields are reduced with an element-wise maximum, and only
rank 0 reports.  The reference arm (the oracle on the host) runs on rank 0 alone; the
other ranks return without work.
"""
import json
import os
import socket
from types import SimpleNamespace

import torch.distributed as dist
import torch.multiprocessing as mp

WORLD = 2


def _free_port():
    with socket.socket() as s:
        s.bind(("127.0.0.1", 0))
        return s.getsockname()[1]


def _worker(rank, world, port, out_dir):
    os.environ.update(MASTER_ADDR="127.0.0.1", MASTER_PORT=str(port), RANK=str(rank),
                      WORLD_SIZE=str(world), LOCAL_RANK=str(rank))
    dist.init_process_group("gloo", rank=rank, world_size=world)
    try:
        import bench
        import workloads

        got = {"env": list(bench.dist_env())}
        # rank r reports times (1 + r, 5 - r, 3): the job's are (world, 5, 3)
        got["max"] = bench.reduce_max([1.0 + rank, 5.0 - rank, 3.0], world, "cpu")
        dist.barrier()
        args = SimpleNamespace(steps=1, warmup=0)
        got["reference_is_none"] = (bench.run_reference(args, workloads.BY_NAME["tiny"], rank)
                                    is None)
        with open(os.path.join(out_dir, f"rank{rank}.json"), "w") as f:
            json.dump(got, f)
    finally:
        dist.destroy_process_group()


def test_replicas_reduce_to_the_slowest_rank(tmp_path):
    mp.spawn(_worker, args=(WORLD, _free_port(), str(tmp_path)), nprocs=WORLD, join=True)
    res = [json.loads((tmp_path / f"rank{r}.json").read_text()) for r in range(WORLD)]
    for r, got in enumerate(res):
        assert got["env"] == [WORLD, r, r]
        assert got["max"] == [float(WORLD), 5.0, 3.0]   # every rank sees the job's maximum
    # rank 0 runs the oracle as the reference arm; the others return at once
    assert res[0]["reference_is_none"] is False
    assert all(got["reference_is_none"] for got in res[1:])


def test_single_rank_reduction_is_the_identity():
    import bench

    assert bench.reduce_max([2.5, 0.25], 1, "cpu") == [2.5, 0.25]


def test_launch_count_claim():
    import bench

    # hashed plan (one kernel) + the apply kernel
    assert bench.kernel_launches_per_call(8192, 129280) == 2
    # 17 id bits -> two 9-bit passes: pack, the digit histogram, one sweep per pass, the
    # listing, plus the apply kernel
    assert bench.kernel_launches_per_call(65536, 129280) == 1 + 1 + 2 + 1 + 1
    # a one-row table needs no radix pass: pack, listing, apply
    assert bench.kernel_launches_per_call(65536, 1) == 1 + 1 + 1
