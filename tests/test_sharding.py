"""Multi-rank host logic on CPU: two gloo ranks shard an attention batch by
sequence and by head, compute their shards with the oracle, and the gathered
result must equal the single-process result; the job time is the maximum over
ranks.  No GPU is used."""
import os
import socket

import numpy as np
import pytest
import torch.distributed as dist
import torch.multiprocessing as mp

from online_softmax_06_gb300 import sharding


def test_shard_range_partitions_exactly():
    for n in range(0, 40):
        for world in range(1, 9):
            seen = []
            for r in range(world):
                b, e = sharding.shard_range(n, r, world)
                assert 0 <= b <= e <= n
                seen.extend(range(b, e))
            assert seen == list(range(n))
            sizes = [e - b for b, e in (sharding.shard_range(n, r, world) for r in range(world))]
            assert max(sizes) - min(sizes) <= 1
    with pytest.raises(ValueError):
        sharding.shard_range(4, 2, 2)


def test_job_throughput():
    assert sharding.job_throughput([10.0, 10.0], 1000.0) == 20.0
    with pytest.raises(ValueError):
        sharding.job_throughput([1.0], 0.0)


def _free_port():
    with socket.socket() as s:
        s.bind(("127.0.0.1", 0))
        return s.getsockname()[1]


def _rank_main(rank, world, port, out_dir):
    import oracle
    import workloads
    os.environ["MASTER_ADDR"] = "127.0.0.1"
    os.environ["MASTER_PORT"] = str(port)
    dist.init_process_group("gloo", rank=rank, world_size=world)
    try:
        B, N, H, d = 4, 37, 6, 8
        Q, K, V = workloads.attention_inputs((B, N, H, d), seed=5, dtype="f32")
        # shard by sequence
        b0, b1 = sharding.batch_shard(B, rank, world)
        O, lse = oracle.attention_dense(Q[b0:b1], K[b0:b1], V[b0:b1], 0.3, True)
        np.save(os.path.join(out_dir, f"batch_O_{rank}.npy"), O)
        np.save(os.path.join(out_dir, f"batch_lse_{rank}.npy"), lse)
        # shard by head
        h0, h1 = sharding.head_shard(H, rank, world)
        O, lse = oracle.attention_dense(np.ascontiguousarray(Q[:, :, h0:h1]),
                                        np.ascontiguousarray(K[:, :, h0:h1]),
                                        np.ascontiguousarray(V[:, :, h0:h1]), 0.3, True)
        np.save(os.path.join(out_dir, f"head_O_{rank}.npy"), O)
        np.save(os.path.join(out_dir, f"head_lse_{rank}.npy"), lse)
        # the job time is the slowest rank's
        ms = sharding.reduce_max_ms(10.0 + 5.0 * rank, dist)
        np.save(os.path.join(out_dir, f"ms_{rank}.npy"), np.array([ms]))
        dist.barrier()
    finally:
        dist.destroy_process_group()


def test_two_rank_sharding_matches_single_process(tmp_path):
    import oracle
    import workloads
    world = 2
    mp.spawn(_rank_main, args=(world, _free_port(), str(tmp_path)), nprocs=world, join=True)
    B, N, H, d = 4, 37, 6, 8
    Q, K, V = workloads.attention_inputs((B, N, H, d), seed=5, dtype="f32")
    O_ref, lse_ref = oracle.attention_dense(Q, K, V, 0.3, True)
    O_b = np.concatenate([np.load(tmp_path / f"batch_O_{r}.npy") for r in range(world)], axis=0)
    l_b = np.concatenate([np.load(tmp_path / f"batch_lse_{r}.npy") for r in range(world)], axis=0)
    assert np.array_equal(O_b, O_ref) and np.array_equal(l_b, lse_ref)
    O_h = np.concatenate([np.load(tmp_path / f"head_O_{r}.npy") for r in range(world)], axis=2)
    l_h = np.concatenate([np.load(tmp_path / f"head_lse_{r}.npy") for r in range(world)], axis=1)
    assert np.array_equal(O_h, O_ref) and np.array_equal(l_h, lse_ref)
    for r in range(world):
        assert float(np.load(tmp_path / f"ms_{r}.npy")[0]) == 15.0
