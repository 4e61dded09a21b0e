"""The element-range partition across ranks, on CPU with gloo (world size 2).

The volume term is element-local, so ranks that each evaluate one contiguous
element range need no exchange; the only collective of the benchmark is the
max-over-ranks of its timed region.  Each rank here takes the element range
that bench.py --split gives it (bench.rank_work), evaluates it with the oracle
(CPU) and rank 0 gathers the pieces: they must reproduce the single-process
result bitwise, and the max reduction must return the slowest rank's value.
"""
import os
import socket

import numpy as np
import pytest
import torch
import torch.distributed as dist
import torch.multiprocessing as mp

import bench
import oracle
import workloads as wl


def _free_port():
    s = socket.socket()
    s.bind(("127.0.0.1", 0))
    port = s.getsockname()[1]
    s.close()
    return port


def _rank_main(rank, world, port, cfg_args, result_path):
    os.environ["MASTER_ADDR"] = "127.0.0.1"
    os.environ["MASTER_PORT"] = str(port)
    dist.init_process_group("gloo", rank=rank, world_size=world)
    try:
        cfg = wl.small_config(*cfg_args[0], K=cfg_args[1], warp=True)
        # the bench's --split arithmetic decides this rank's element range
        e0, ec = bench.rank_work(cfg.K, world, rank, split=True)
        assert (e0, ec) == bench.element_shard(cfg.K, world, rank)
        g = wl.generate_elements(cfg, np.arange(e0, e0 + ec))
        gc = {k: v.numpy() for k, v in g.items()}
        Ja, _ = oracle.metrics(cfg.N, ec, gc["x"], gc["y"], gc["z"])
        out = oracle.volume(cfg.N, ec, gc["q"], Ja, gc["phi"], nthreads=1)
        # gather variable-size pieces: pad to the largest range
        np3 = cfg.Nq ** 3
        cap = (cfg.K // world + 1) * np3
        buf = torch.zeros((5, cap), dtype=torch.float64)
        buf[:, :ec * np3] = torch.from_numpy(out)
        pieces = [torch.zeros_like(buf) for _ in range(world)] if rank == 0 else None
        dist.gather(buf, pieces, dst=0)
        slow = bench.max_over_ranks(float(10 + rank))
        if rank == 0:
            full = []
            for r in range(world):
                _, c = bench.element_shard(cfg.K, world, r)
                full.append(pieces[r][:, :c * np3].numpy())
            np.save(result_path, np.concatenate(full, axis=1))
            with open(result_path + ".max", "w") as f:
                f.write(repr(slow))
    finally:
        dist.destroy_process_group()


def test_element_shard_covers_range():
    for K in (1, 2, 7, 13, 100, 8192):
        for world in (1, 2, 3, 8):
            rng = [bench.element_shard(K, world, r) for r in range(world)]
            pos = 0
            for e0, ec in rng:
                assert e0 == pos and ec >= 0
                pos += ec
            assert pos == K
            assert max(c for _, c in rng) - min(c for _, c in rng) <= 1


def test_split_and_replica_work():
    """--split: each rank its element_shard range and the job one mesh (strong
    scaling); replicas: each rank the whole mesh and the job one per rank."""
    for K in (1, 15, 8192):
        for world in (1, 2, 4, 8):
            ranges = [bench.rank_work(K, world, r, split=True) for r in range(world)]
            assert ranges == [bench.element_shard(K, world, r) for r in range(world)]
            assert sum(c for _, c in ranges) == K
            assert all(bench.rank_work(K, world, r, split=False) == (0, K) for r in range(world))
            n = K * 64
            assert bench.job_nodes(n, world, split=True) == n
            assert bench.job_nodes(n, world, split=False) == world * n


def test_two_rank_partition_matches_single_process(tmp_path):
    oracle.build()
    cfg_args = ((3,), (5, 3, 1))  # N = 3, 15 elements: a ragged split 8 + 7
    world = 2
    port = _free_port()
    result = str(tmp_path / "gathered.npy")
    mp.start_processes(_rank_main, args=(world, port, cfg_args, result), nprocs=world, join=True,
                       start_method="spawn")
    gathered = np.load(result)
    cfg = wl.small_config(*cfg_args[0], K=cfg_args[1], warp=True)
    g = wl.generate(cfg)
    Ja, _ = oracle.metrics(cfg.N, cfg.K, g["x"].numpy(), g["y"].numpy(), g["z"].numpy())
    ref = oracle.volume(cfg.N, cfg.K, g["q"].numpy(), Ja, g["phi"].numpy(), nthreads=1)
    assert np.array_equal(gathered, ref)
    with open(result + ".max") as f:
        assert float(f.read()) == 11.0
