"""The multi-GPU host logic on CPU: two gloo ranks shard the streams of a workload, each runs
the oracle on its own streams, and the union equals a single-process run; the max-over-ranks
timing reduction behaves as the benchmark uses it."""

import os
import socket

import numpy as np
import pytest
import torch.distributed as dist
import torch.multiprocessing as mp

from sparse_slot_memory_gb300.sharding import shard_streams


def test_shard_streams_partition():
    for P in (1, 3, 8, 32, 33):
        for world in (1, 2, 3, 8):
            got = [s for r in range(world) for s in shard_streams(P, r, world)]
            assert got == list(range(P))
    with pytest.raises(ValueError):
        shard_streams(4, 2, 2)


def _free_port():
    with socket.socket() as s:
        s.bind(("127.0.0.1", 0))
        return s.getsockname()[1]


def _rank_main(rank, world, port, out_dir):
    import oracle
    from synth import WORKLOADS, make_inputs, scaled

    os.environ.update(MASTER_ADDR="127.0.0.1", MASTER_PORT=str(port))
    dist.init_process_group("gloo", rank=rank, world_size=world)
    w = scaled(WORKLOADS["uniform_c128"], P=4, T=256, S=512, hd=8, name="mr")
    mine = list(shard_streams(w.P, rank, world))
    x = make_inputs(w, streams=mine)
    o = oracle.phase1(x["k_idx"], x["q_idx"], x["k_val"], x["q_val"], x["g"], S=w.S, val_dtype=w.val_dtype,
                      pairs=False)
    np.save(os.path.join(out_dir, f"logk_{rank}.npy"), o["log_k"])
    import torch
    t = torch.tensor([float(rank + 1)])
    dist.all_reduce(t, op=dist.ReduceOp.MAX)
    assert t.item() == float(world)
    dist.barrier()
    dist.destroy_process_group()


def test_two_gloo_ranks_match_single_process(tmp_path):
    import oracle
    from synth import WORKLOADS, make_inputs, scaled

    world, port = 2, _free_port()
    mp.start_processes(_rank_main, args=(world, port, str(tmp_path)), nprocs=world, start_method="spawn")
    w = scaled(WORKLOADS["uniform_c128"], P=4, T=256, S=512, hd=8, name="mr")
    x = make_inputs(w)
    full = oracle.phase1(x["k_idx"], x["q_idx"], x["k_val"], x["q_val"], x["g"], S=w.S, val_dtype=w.val_dtype,
                         pairs=False)["log_k"].reshape(w.steps, w.P, w.C, w.W)
    for r in range(world):
        got = np.load(tmp_path / f"logk_{r}.npy")
        streams = list(shard_streams(w.P, r, world))
        np.testing.assert_array_equal(got.reshape(w.steps, len(streams), w.C, w.W), full[:, streams])
