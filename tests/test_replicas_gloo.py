"""Multi-GPU runs are replicas: every rank decodes its own copy of the
workload and the job time is the slowest rank's.  This checks that logic with
two gloo ranks on CPU: the max-over-ranks reduction bench.py uses, and that
two ranks given the same workload and seed produce identical draws (the
oracle stands in for the device, which this test does not need)."""
import os
import socket

import numpy as np
import pytest
import torch.multiprocessing as mp


def _free_port():
    with socket.socket() as s:
        s.bind(("127.0.0.1", 0))
        return s.getsockname()[1]


def _rank_main(rank, world, port, out_dir):
    os.environ.update(MASTER_ADDR="127.0.0.1", MASTER_PORT=str(port), RANK=str(rank), WORLD_SIZE=str(world),
                      LOCAL_RANK=str(rank))
    import sys
    root = os.path.dirname(os.path.dirname(os.path.abspath(__file__)))
    sys.path.insert(0, root)
    import torch.distributed as dist
    import bench
    import oracle
    import synth
    dist.init_process_group("gloo", rank=rank, world_size=world)
    try:
        assert bench.dist_env() == (world, rank, rank)
        # each rank times its own replica; the job time is the largest
        assert bench.max_over_ranks(10.0 + rank) == 10.0 + world - 1
        inp = synth.generate(synth.tiny("systematic"), 0)
        P = oracle.Problem.from_inputs(inp)
        est, J, _ = oracle.decode(P, "systematic", inp.wl.S, 3, 0)
        np.save(os.path.join(out_dir, f"J{rank}.npy"), J)
        np.save(os.path.join(out_dir, f"est{rank}.npy"), est)
        dist.barrier()
    finally:
        dist.destroy_process_group()


def test_two_gloo_ranks_are_independent_replicas(tmp_path, oracle_lib):
    world = 2
    mp.start_processes(_rank_main, args=(world, _free_port(), str(tmp_path)), nprocs=world, join=True,
                       start_method="spawn")
    assert np.array_equal(np.load(tmp_path / "J0.npy"), np.load(tmp_path / "J1.npy"))
    assert np.array_equal(np.load(tmp_path / "est0.npy"), np.load(tmp_path / "est1.npy"))


def test_single_process_max_is_identity():
    import bench
    assert bench.max_over_ranks(3.5) == 3.5
