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


def test_bench_byte_accounting_follows_the_split_work_list():
    """Algorithmic bytes of the decode call and of its main kernel, written
    out by hand for two small CPU workloads.

    head_size 64 (the CUDA-core kernel): one sequence of 1 token and one of
    65 tokens (partitions of 64): every partition writes a partial state,
    the reduce reads them all and writes both output rows.

    head_size 128 (the tensor-core kernel, 4 kv heads per CTA, 2 head
    groups): one sequence of 1 token (writes its output directly) and one of
    321 tokens = 6 partitions of 64, 5 full ones.  With a grid of 2 CTAs the
    list keeps ceil(3 * 2 / (2 seqs * 2 groups)) - 1 = 1 trailing single
    full partition, so partitions 0-3 form one run, 4 is single, 5 is the
    last: 3 partial states, 3 covered partitions marked empty."""
    import bench
    import workload as wl
    w = wl.make("tiny", device="cpu", lengths=[1, 65], seed=1)
    el, H, Hkv, D = 2, w.num_heads, w.num_kv_heads, w.head_size
    kv = (1 + 65) * Hkv * D * el * 2
    q = 2 * H * D * el
    tables = (1 + 5) * 4 + 2 * 4          # blocks in use (bs 16) + seq_lens
    state = H * (D + 2) * 4               # one partition's partial state, all heads
    assert bench.kv_bytes(w) == kv
    assert bench.split_partials(w, 64, sms=2) == (3 * state, 3 * state, q)
    assert bench.decode_launch_bytes(w, False, 64) == kv + 2 * q + tables
    assert bench.decode_launch_bytes(w, True, 64) == kv + 2 * q + tables + 6 * state
    assert bench.decode_kernel_bytes(w, True, 64) == kv + q + tables + 3 * state

    w = wl.make("gqa8b", device="cpu", lengths=[1, 321], seed=1)
    H, Hkv, D = w.num_heads, w.num_kv_heads, w.head_size
    assert (H, Hkv, D) == (32, 8, 128)
    written = H * (3 * (D + 2) * 4 + 3 * 8)
    read = H * (6 * 8 + 3 * D * 4)
    row = H * D * el
    assert bench.split_partials(w, 64, sms=2) == (written, read, row)
