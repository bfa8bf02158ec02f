"""Host logic of the N > 1 bench path, on CPU with gloo (world size 2): each
rank encodes its own documents (weak scaling, nothing exchanged on the data
path) and the reported numbers are the max of the times and the sum of the
work over ranks."""
import os
import socket

import numpy as np
import pytest

import workloads


def _free_port() -> int:
    with socket.socket() as s:
        s.bind(("127.0.0.1", 0))
        return s.getsockname()[1]


def _rank_main(rank: int, world: int, port: int, out_dir: str):
    import torch.distributed as dist

    import bench
    os.environ.update(MASTER_ADDR="127.0.0.1", MASTER_PORT=str(port))
    dist.init_process_group("gloo", rank=rank, world_size=world)
    first, n = bench.shard(1, rank, 64)
    data, offsets = workloads.docs(1, first, n)
    # per-rank stand-ins for the measured times; the counts are the rank's own
    times = [10.0 + rank, 5.0 * (rank + 1), 20.0 - rank]
    counts = [float(data.size), float(rank + 1), float(n)]
    got_t, got_c = bench.reduce_ranks(dist, "cpu", times, counts)
    np.save(os.path.join(out_dir, f"rank{rank}.npy"),
            np.array([first, n, data.size, *got_t, *got_c], dtype=np.float64))
    dist.barrier()
    dist.destroy_process_group()


def test_two_rank_shards_and_reduction(tmp_path):
    import torch.multiprocessing as mp
    world = 2
    mp.start_processes(_rank_main, args=(world, _free_port(), str(tmp_path)), nprocs=world, start_method="spawn")
    r = [np.load(tmp_path / f"rank{k}.npy") for k in range(world)]
    # disjoint, contiguous shards of the same generator
    assert r[0][0] == 0 and r[1][0] == r[0][1]
    # both ranks see the same reduced values: max of times, sum of counts
    for k in range(world):
        assert list(r[k][3:6]) == [11.0, 10.0, 20.0]
        assert r[k][6] == r[0][2] + r[1][2]
        assert r[k][7] == 3.0 and r[k][8] == r[0][1] + r[1][1]
    # the two shards are different documents
    a, _ = workloads.docs(1, 0, 64)
    b, _ = workloads.docs(1, 64, 64)
    assert not np.array_equal(a[:1000], b[:1000])


def test_reduce_without_process_group_is_identity():
    import bench
    assert bench.reduce_ranks(None, "cpu", [1.0, 2.0], [3.0]) == ([1.0, 2.0], [3.0])


@pytest.mark.parametrize("rank", [0, 1, 3])
def test_shard_is_rank_offset(rank):
    import bench
    assert bench.shard(5, rank, 100) == (rank * 100, 100)
