"""Edge cases of the CUDA path: empty sequences, guard bands, device-side
range guards, streams, partition-size invariance, determinism and batch
invariance.  Bad ids/lengths/slots below are ones the kernels' own bounds
checks turn into an error bit without dereferencing them."""
import numpy as np
import pytest
import torch

import workload as wl
from tests._parity import (check_agree, check_attention, check_lse, oracle_decode,
                           oracle_decode_lse, splitk_workspace)

pytestmark = pytest.mark.gpu


@pytest.fixture(scope="module")
def pa():
    from __graft_entry__ import build_library
    build_library()
    import paged_kv_cache_136_gb300 as pa
    pa.pa_device_errors(clear=True)
    return pa


def _decode(pa, w, split, partition_size=512, max_seq_len=None, out=None, stream=None):
    out = torch.empty_like(w.q) if out is None else out
    if split:
        msl = int(w.seq_lens.max().item()) if max_seq_len is None else max_seq_len
        ws = splitk_workspace(pa, w, msl, partition_size)
        pa.pa_decode_splitk(out, w.q, w.kv_cache, w.block_tables, w.seq_lens, w.scale,
                            w.block_size, msl, ws, partition_size, stream=stream)
    else:
        pa.pa_decode(out, w.q, w.kv_cache, w.block_tables, w.seq_lens, w.scale, w.block_size,
                     stream=stream)
    return out


@pytest.mark.parametrize("split", [False, True])
def test_empty_sequences_give_zero_rows(pa, split):
    w = wl.make("gqa8b", device="cuda", poison=True, lengths=[0, 5, 0, 130], seed=3)
    out = _decode(pa, w, split, partition_size=64)
    torch.cuda.synchronize()
    assert torch.count_nonzero(out[0]) == 0 and torch.count_nonzero(out[2]) == 0
    check_attention(out, oracle_decode(w), what="empty rows")
    assert pa.pa_device_errors() == 0


def test_all_sequences_empty_split(pa):
    w = wl.make("tiny", device="cuda", lengths=[0, 0], seed=4)
    out = _decode(pa, w, True, partition_size=64, max_seq_len=0)
    torch.cuda.synchronize()
    assert torch.count_nonzero(out) == 0


@pytest.mark.parametrize("split", [False, True])
def test_output_guard_bands_untouched(pa, split):
    w = wl.make("tiny", device="cuda", poison=True)
    n = w.q.numel()
    buf = torch.full((n + 2048,), 7.0, dtype=w.dtype, device="cuda")
    out = buf[1024:1024 + n].view_as(w.q)
    _decode(pa, w, split, partition_size=64, out=out)
    torch.cuda.synchronize()
    assert bool((buf[:1024] == 7.0).all()) and bool((buf[1024 + n:] == 7.0).all())
    check_attention(out, oracle_decode(w), what="guarded out")


def test_bad_block_id_sets_flag_and_is_not_read(pa):
    w = wl.make("tiny", device="cuda", seed=5)
    bt = w.block_tables.clone()
    bt[3, 2] = w.num_blocks + 5          # seq 3 (64 tokens) uses blocks 0..3
    bt[1, 0] = -7
    out = torch.empty_like(w.q)
    pa.pa_decode(out, w.q, w.kv_cache, bt, w.seq_lens, w.scale, w.block_size)
    flags = pa.pa_device_errors(clear=True)
    assert flags & pa.DEVERR_BLOCK_ID
    # Rows that use only valid ids are still right.
    ref = oracle_decode(w)
    check_attention(out[[0, 2]], ref[[0, 2]], what="valid rows next to bad ids")


def test_seq_len_beyond_table_is_clamped_and_flagged(pa):
    w = wl.make("tiny", device="cuda", seed=6)
    sl = w.seq_lens.clone()
    sl[0] = w.block_tables.shape[1] * w.block_size + 100
    sl[1] = -3
    out = torch.empty_like(w.q)
    pa.pa_decode(out, w.q, w.kv_cache, w.block_tables, sl, w.scale, w.block_size)
    assert pa.pa_device_errors(clear=True) & pa.DEVERR_SEQ_LEN
    assert torch.count_nonzero(out[1]) == 0


def test_seq_len_beyond_max_seq_len_is_flagged(pa):
    w = wl.make("gqa8b", device="cuda", lengths=[300, 700], seed=7)
    out = _decode(pa, w, True, partition_size=128, max_seq_len=256)
    assert pa.pa_device_errors(clear=True) & pa.DEVERR_SEQ_LEN
    assert torch.isfinite(out).all()


def test_out_of_range_slot_writes_nothing_and_is_flagged(pa):
    w = wl.make("tiny", device="cuda", seed=8)
    before = w.kv_cache.clone()
    sm = torch.full_like(w.slot_mapping, -1)
    sm[0] = w.num_blocks * w.block_size          # one past the pool
    pa.pa_reshape_and_cache(w.key, w.value, w.kv_cache, sm, w.block_size)
    assert pa.pa_device_errors(clear=True) & pa.DEVERR_SLOT
    assert torch.equal(w.kv_cache.view(torch.int16), before.view(torch.int16))


@pytest.mark.parametrize("split", [False, True])
def test_runs_on_a_side_stream(pa, split):
    w = wl.make("gqa8b", device="cuda", poison=True, num_seqs=16, seed=9)
    s = torch.cuda.Stream()
    with torch.cuda.stream(s):
        out = _decode(pa, w, split, partition_size=256, stream=s)
    s.synchronize()
    check_attention(out, oracle_decode(w), what="side stream")


def test_partition_size_invariance(pa):
    w = wl.make("gqa8b", device="cuda", poison=True, lengths=[1, 700, 1500, 4096, 64, 65],
                seed=10)
    ref = oracle_decode(w)
    one = _decode(pa, w, False)
    check_attention(one, ref, what="one-pass")
    for P in (64, 128, 192, 512, 1024, 4096):
        out = _decode(pa, w, True, partition_size=P)
        check_attention(out, ref, what=f"partition {P}")
        check_agree(out, one, what=f"partition {P} vs one-pass")


def test_split_runs_match_oracle(pa):
    """A sequence long enough that the split-K work list groups its full
    partitions into runs of four consecutive partitions (one work item and
    one partial state each; the partitions a run covers carry zero weight in
    the reduce), beside a shorter one: with 64-token partitions and two
    sequences, each keeps its last ceil(3 * 152 / 4) - 1 = 113 full
    partitions single, so the first sequence's 130 full partitions give 4
    runs.  Outputs and log-sum-exps match the oracle."""
    w = wl.make("gqa8b", device="cuda", poison=True, lengths=[64 * 130 + 5, 3000], seed=12)
    P = 64
    msl = int(w.seq_lens.max().item())
    ws = splitk_workspace(pa, w, msl, P)
    out = torch.empty_like(w.q)
    lse = torch.empty(w.num_seqs, w.num_heads, dtype=torch.float32, device="cuda")
    pa.pa_decode_splitk_lse(out, lse, w.q, w.kv_cache, w.block_tables, w.seq_lens, w.scale,
                            w.block_size, msl, ws, P)
    torch.cuda.synchronize()
    check_attention(out, oracle_decode(w), what="runs of partitions")
    check_lse(lse, oracle_decode_lse(w), what="runs of partitions")
    assert pa.pa_device_errors(clear=True) == 0


def test_reduce_many_partitions(pa):
    """More partitions per row than one shared-memory chunk of merge weights
    holds (625 and 514 of 64 tokens: the reduce walks two chunks, with thread
    groups splitting the partitions unevenly), beside a one-partition
    sequence and one that ends just past a partition boundary."""
    w = wl.make("gqa8b", device="cuda", poison=True,
                lengths=[40000, 64 * 513 + 7, 5, 33001], seed=12)
    ref = oracle_decode(w)
    out = _decode(pa, w, True, partition_size=64)
    check_attention(out, ref, what="hundreds of partitions")


@pytest.mark.parametrize("max_parts", [32, 33])
def test_reduce_partition_count_boundary(pa, max_parts):
    """Rows of up to 32 partitions are merged one warp per row, longer ones by
    the thread-group reduce: both sides of the switch, with rows of 1, 2, 31
    and the maximum number of 64-token partitions, a head count that is not a
    multiple of the heads one reduce CTA takes, and the log-sum-exp output."""
    P = 64
    lens = [P * max_parts, P * 30 + 1, P, P + 1, P * max_parts - 5]
    w = wl.make("gqa8b", device="cuda", poison=True, lengths=lens, num_heads=12,
                num_kv_heads=6, seed=40 + max_parts)
    msl = P * max_parts
    ws = splitk_workspace(pa, w, msl, P)
    out = torch.empty_like(w.q)
    lse = torch.empty((w.num_seqs, w.num_heads), dtype=torch.float32, device="cuda")
    pa.pa_decode_splitk_lse(out, lse, w.q, w.kv_cache, w.block_tables, w.seq_lens, w.scale,
                            w.block_size, msl, ws, P)
    check_attention(out, oracle_decode(w), what=f"max_parts={max_parts}")
    check_lse(lse, oracle_decode_lse(w), what=f"max_parts={max_parts}")
    assert pa.pa_device_errors(clear=True) == 0


@pytest.mark.parametrize("split", [False, True])
def test_deterministic_and_batch_invariant(pa, split):
    """Same inputs give identical bits; a sequence's output does not depend on
    which other sequences share the batch."""
    w = wl.make("gqa8b", device="cuda", num_seqs=32, seed=11)
    a = _decode(pa, w, split)
    b = _decode(pa, w, split)
    torch.cuda.synchronize()
    assert torch.equal(a.view(torch.int16), b.view(torch.int16))
    sub = [3, 17, 30]
    ws = wl.Workload(**{k: getattr(w, k) for k in w.__dataclass_fields__})
    ws.q = w.q[sub].contiguous()
    ws.block_tables = w.block_tables[sub].contiguous()
    ws.seq_lens = w.seq_lens[sub].contiguous()
    c = _decode(pa, ws, split, max_seq_len=int(w.seq_lens.max().item()))
    torch.cuda.synchronize()
    assert torch.equal(c.view(torch.int16), a[sub].view(torch.int16))


def test_bounded_wait_times_out_and_context_survives(pa):
    """A wait that nothing completes gives up, reports PA_DEVERR_TIMEOUT, and
    the context keeps working."""
    pa.pa_device_errors(clear=True)
    pa.pa_selftest_wait_timeout()
    assert pa.pa_device_errors(clear=True) & pa.DEVERR_TIMEOUT
    w = wl.make("tiny", device="cuda", poison=True)
    out = _decode(pa, w, False)
    torch.cuda.synchronize()
    check_attention(out, oracle_decode(w), what="after timeout self-test")
    assert pa.pa_device_errors(clear=True) == 0


@pytest.mark.parametrize("P", [64, 192, 320])
def test_tensor_core_one_head_per_cta_and_ragged_partitions(pa, P):
    """3 kv heads cannot be grouped, so the tensor-core kernel runs one kv
    head per CTA (128-token stages); partitions that are not a multiple of
    the stage end in partial stages."""
    w = wl.make("gqa8b", device="cuda", poison=True, lengths=[1, 100, 129, 700, 1031],
                num_heads=12, num_kv_heads=3, seed=40 + P)
    ref = oracle_decode(w)
    check_attention(_decode(pa, w, True, partition_size=P), ref, what=f"Hkv=3 split P={P}")
    check_attention(_decode(pa, w, False), ref, what="Hkv=3 one-pass")
    assert pa.pa_device_errors(clear=True) == 0


# ---------------------------------------------------------------------------
# Copy-on-write block copy
# ---------------------------------------------------------------------------

@pytest.mark.parametrize("name", ["mha7b", "gqa8b"])
def test_copy_blocks_bit_exact(pa, name):
    from oracle.oracle import get
    w = wl.make(name, device="cuda", poison=True, num_seqs=8, seed=50)
    rng = np.random.default_rng(51)
    ids = rng.permutation(w.num_blocks)
    n = min(300, w.num_blocks // 2)
    mapping = torch.from_numpy(np.stack([ids[:n], ids[n:2 * n]], 1).astype(np.int64)).cuda()
    assert pa.pa_validate_block_mapping(mapping, w.num_blocks) == 0
    ref = get().copy_blocks(wl.bits(w.kv_cache), mapping.cpu().numpy())
    pa.pa_copy_blocks(w.kv_cache, mapping, w.block_size)
    torch.cuda.synchronize()
    assert np.array_equal(wl.bits(w.kv_cache), ref)
    assert pa.pa_device_errors(clear=True) == 0


def test_copy_blocks_bad_id_is_skipped_and_flagged(pa):
    w = wl.make("tiny", device="cuda", seed=52)
    before = w.kv_cache.clone()
    mapping = torch.tensor([[w.num_blocks + 3, 0], [1, -1]], dtype=torch.int64, device="cuda")
    pa.pa_copy_blocks(w.kv_cache, mapping, w.block_size)
    assert pa.pa_device_errors(clear=True) & pa.DEVERR_BLOCK_ID
    assert torch.equal(w.kv_cache.view(torch.int16), before.view(torch.int16))


def test_copy_on_write_step_on_gpu(pa):
    """Fork, copy, repoint, write, decode: the GPU matches the oracle and the
    sequences that kept the shared block still read the original."""
    w = wl.make("gqa8b", device="cuda", poison=True, lengths=[40, 40, 40], seed=53)
    bs = w.block_size
    shared = w.block_tables[0].clone()
    tables = shared.repeat(3, 1).contiguous()            # three candidates share the prompt
    w.q[2].copy_(w.q[0])                                 # candidates 0 and 2 stay identical
    w.block_tables = tables
    free = int(w.num_blocks - 1)                         # a block no table uses
    used = set(tables.flatten().tolist())
    while free in used:
        free -= 1
    last = int(tables[1, (40 - 1) // bs].item())
    mapping = torch.tensor([[last, free]], dtype=torch.int64, device="cuda")
    pa.pa_copy_blocks(w.kv_cache, mapping, bs)
    tables[1, (40 - 1) // bs] = free
    w.seq_lens = torch.tensor([40, 41, 40], dtype=torch.int32, device="cuda")
    slot = torch.tensor([-1, free * bs + 40 % bs, -1], dtype=torch.int64, device="cuda")
    pa.pa_reshape_and_cache(w.key, w.value, w.kv_cache, slot, bs)
    out = _decode(pa, w, True, partition_size=64)
    torch.cuda.synchronize()
    check_attention(out, oracle_decode(w), what="copy-on-write step")
    assert torch.equal(out[0].view(torch.int16), out[2].view(torch.int16))


def test_stage_copy_bit_exact(pa):
    """Pinned host -> device, device -> pinned host and device -> device on the
    SMs, and the stream-copy fallback for a size that is not a multiple of 16
    and for a misaligned start, all bit-exact."""
    g = torch.Generator().manual_seed(21)
    n = 1606400
    src_h = torch.randint(0, 256, (n,), dtype=torch.uint8, generator=g).pin_memory()
    dev = torch.empty(n, dtype=torch.uint8, device="cuda")
    pa.pa_stage_copy(dev, src_h)
    back = torch.empty(n, dtype=torch.uint8).pin_memory()
    pa.pa_stage_copy(back, dev)
    dev2 = torch.empty(n, dtype=torch.uint8, device="cuda")
    pa.pa_stage_copy(dev2, dev)
    torch.cuda.synchronize()
    assert torch.equal(back, src_h)
    assert torch.equal(dev2.cpu(), src_h)
    # 1000 bytes (not a multiple of 16), and a start one byte past alignment
    odd = torch.empty(1000, dtype=torch.uint8, device="cuda")
    pa.pa_stage_copy(odd, src_h[:1000])
    mis = torch.empty(4096, dtype=torch.uint8, device="cuda")
    pa.pa_stage_copy(mis, src_h[1:4097])
    torch.cuda.synchronize()
    assert torch.equal(odd.cpu(), src_h[:1000])
    assert torch.equal(mis.cpu(), src_h[1:4097])
    assert pa.pa_device_errors(clear=True) == 0
