"""Host logic of the multi-replica benchmark on CPU: two gloo ranks exchange
their timing and byte counts the way bench.py does (max of times, sum of
bytes), with barriers around the timed region, and no data-path collective."""
import os
import socket

import pytest
import torch.multiprocessing as mp


def _free_port() -> int:
    with socket.socket() as s:
        s.bind(("127.0.0.1", 0))
        return s.getsockname()[1]


def _rank_main(rank, world, port, results):
    os.environ.update(MASTER_ADDR="127.0.0.1", MASTER_PORT=str(port), RANK=str(rank),
                      WORLD_SIZE=str(world), LOCAL_RANK=str(rank))
    import bench
    r, w, _ = bench.dist_env()
    assert (r, w) == (rank, world)
    dist = bench.init_dist(w, "gloo")
    bench.barrier(dist)
    # each replica processed its own batch: different local times and bytes
    local_ms = 10.0 + 5.0 * rank
    local_bytes = 1e9 * (rank + 1)
    ms_max = bench.reduce_scalar(local_ms, "max", dist)
    total = bench.reduce_scalar(local_bytes, "sum", dist)
    bench.barrier(dist)
    results[rank] = (ms_max, total)
    dist.destroy_process_group()


def test_two_rank_replica_aggregation():
    world = 2
    port = _free_port()
    with mp.Manager() as m:
        results = m.dict()
        mp.spawn(_rank_main, args=(world, port, results), nprocs=world, join=True)
        res = dict(results)
    assert res[0] == res[1] == (15.0, 3e9)


def test_single_rank_needs_no_process_group(monkeypatch):
    import bench
    for k in ("RANK", "WORLD_SIZE", "LOCAL_RANK"):
        monkeypatch.delenv(k, raising=False)
    assert bench.dist_env() == (0, 1, 0)
    assert bench.init_dist(1, "gloo") is None
    assert bench.reduce_scalar(3.5, "max", None) == 3.5


@pytest.mark.parametrize("argv,expect", [
    ([], ("ours", 1, 2000)),
    (["--impl", "reference", "--steps", "7"], ("reference", 1, 7)),
    (["--gpus", "8"], ("ours", 8, 2000)),
])
def test_bench_arguments(argv, expect):
    import bench
    a = bench.parse_args(argv)
    assert (a.impl, a.gpus, a.steps) == expect
    assert a.config == "long"


def test_bench_byte_accounting_counts_partials_of_split_sequences_only():
    """Algorithmic bytes of the decode call and of its main kernel on a small
    CPU workload, written out by hand: one sequence of 1 token (one
    partition, its output row written by the kernel), one of 65 tokens (two
    partitions of 64: partial states written by the kernel, read by the
    reduce)."""
    import bench
    import workload as wl
    w = wl.make("tiny", device="cpu", lengths=[1, 65], seed=1)
    el, H, Hkv, D, bs = 2, w.num_heads, w.num_kv_heads, w.head_size, w.block_size
    kv = (1 + 65) * Hkv * D * el * 2
    q = 2 * H * D * el
    tables = (1 + 5) * 4 + 2 * 4          # blocks in use (bs 16) + seq_lens
    partial = H * (D + 2) * 4             # one (sequence, head) partial state
    assert bench.kv_bytes(w) == kv
    assert bench.decode_launch_bytes(w, False, 64) == kv + 2 * q + tables
    assert bench.decode_launch_bytes(w, True, 64) == kv + 2 * q + tables + 2 * 2 * partial
    row = H * D * el
    assert bench.decode_kernel_bytes(w, True, 64) == kv + q + tables + row + 2 * partial
    assert bench.decode_kernel_bytes(w, False, 64) == kv + 2 * q + tables
