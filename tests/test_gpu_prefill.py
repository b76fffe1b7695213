"""Prefill / chunked prefill on the tensor cores vs the CPU oracle.

Every call goes through the C ABI.  Pools are NaN-poisoned wherever no
request owns a row, so a read past a request's end shows up in its output.
"""
import numpy as np
import pytest
import torch

import workload as wl
from tests._parity import check_attention, check_lse, oracle_prefill

pytestmark = pytest.mark.gpu


@pytest.fixture(scope="module")
def pa():
    from __graft_entry__ import build_library
    build_library()
    import paged_kv_cache_136_gb300 as pa
    pa.pa_device_errors(clear=True)
    return pa


def _run(pa, w, causal=True, with_lse=True, out=None, block_tables=None, seq_lens=None,
         max_query_len=None):
    out = torch.empty_like(w.q) if out is None else out
    lse = torch.empty(w.q.shape[:2], dtype=torch.float32, device=w.q.device) if with_lse else None
    mq = int(w.q_lens().max()) if max_query_len is None else max_query_len
    pa.pa_prefill(out, w.q, w.kv_cache, w.block_tables if block_tables is None else block_tables,
                  w.seq_lens if seq_lens is None else seq_lens, w.query_start_loc, w.scale,
                  w.block_size, mq, causal=causal, lse=lse)
    torch.cuda.synchronize()
    return out, lse


SHAPES = [
    # q_lens, ctx_lens, H, Hkv, D, bs, dtype
    ([1, 20, 37, 130], [0, 5, 0, 70], 4, 2, 128, 16, torch.float16),
    ([128, 256, 257, 1], [0, 128, 3, 500], 8, 8, 128, 32, torch.bfloat16),
    ([300, 17], [1000, 0], 4, 1, 128, 16, torch.bfloat16),
    ([1, 20, 37, 130], [0, 5, 0, 70], 4, 4, 64, 16, torch.float16),
    ([200, 511], [64, 0], 2, 2, 64, 32, torch.bfloat16),
    ([33, 190], [70, 0], 4, 2, 64, 16, torch.bfloat16),
    ([150, 3], [40, 260], 4, 2, 128, 32, torch.float16),
    # at most 128 query rows and an even group: a CTA's tiles are two heads
    ([100, 7, 128], [50, 300, 0], 8, 2, 128, 16, torch.bfloat16),
    ([1, 64], [10, 0], 16, 2, 64, 32, torch.float16),
]


@pytest.mark.parametrize("causal", [True, False])
@pytest.mark.parametrize("q_lens,ctx,H,Hkv,D,bs,dtype", SHAPES)
def test_prefill_matches_oracle(pa, q_lens, ctx, H, Hkv, D, bs, dtype, causal):
    w = wl.make_prefill("prefill_tiny", device="cuda", poison=True, q_lens=q_lens,
                        ctx_lens=ctx, num_heads=H, num_kv_heads=Hkv, head_size=D,
                        block_size=bs, dtype=dtype, seed=sum(q_lens) + D)
    out, lse = _run(pa, w, causal=causal)
    ref, ref_lse = oracle_prefill(w, causal=causal)
    check_attention(out, ref, what=f"prefill {q_lens} causal={causal}")
    check_lse(lse, ref_lse, what="prefill lse")
    assert pa.pa_device_errors(clear=True) == 0


def _sample_items(w, rng, n):
    """First and last rows of every request, rows around 128-row tile edges,
    and random rows; every query head."""
    qsl = w.query_start_loc.cpu().numpy()
    toks = set()
    for r in range(w.num_reqs):
        a, b = int(qsl[r]), int(qsl[r + 1])
        for t in (a, a + 127, a + 128, a + 255, a + 256, b - 1):
            if a <= t < b:
                toks.add(t)
    toks.update(rng.integers(0, w.num_tokens, size=n).tolist())
    toks = np.array(sorted(toks))
    heads = rng.integers(0, w.num_heads, size=toks.size)
    items = toks * w.num_heads + heads
    # every head at least once
    extra = (rng.integers(0, w.num_tokens, size=w.num_heads) * w.num_heads
             + np.arange(w.num_heads))
    return np.unique(np.concatenate([items, extra]))


@pytest.mark.parametrize("name", ["prefill_mha7b", "prefill_gqa8b"])
def test_prefill_full_size_sampled_rows(pa, name):
    w = wl.make_prefill(name, device="cuda", poison=True)
    out, lse = _run(pa, w)
    items = _sample_items(w, np.random.default_rng(7), 160)
    ref, ref_lse = oracle_prefill(w, items=items)
    check_attention(out, ref, items=items, what=name)
    check_lse(lse, ref_lse, items=items, what=name)
    assert pa.pa_device_errors(clear=True) == 0


def test_prefill_step_writes_then_attends(pa):
    """Cache write of the new tokens, then prefill: the new keys are read."""
    from oracle.oracle import get
    w = wl.make_prefill("prefill_tiny", device="cuda", poison=True)
    cache0 = wl.bits(w.kv_cache)
    pa.pa_reshape_and_cache(w.key, w.value, w.kv_cache, w.slot_mapping, w.block_size)
    out, lse = _run(pa, w)
    cb = get().reshape_and_cache(wl.bits(w.key), wl.bits(w.value), cache0,
                                 w.slot_mapping.cpu().numpy(), w.block_size)
    assert np.array_equal(wl.bits(w.kv_cache), cb)
    ref, ref_lse = oracle_prefill(w, cache_bits=cb)
    check_attention(out, ref, what="write then prefill")


def test_prefill_rescale_when_scores_grow(pa):
    """Keys whose scores climb by several units per key tile force the lazy
    rescale of O again and again."""
    w = wl.make_prefill("prefill_tiny", device="cuda", poison=True, q_lens=[200, 64],
                        ctx_lens=[900, 1200], seed=9)
    bs = w.block_size
    bt = w.block_tables.cpu().numpy()
    L = w.seq_lens.cpu().numpy()
    q = w.q.float()
    qdir = q / q.norm(dim=-1, keepdim=True)
    qsl = w.query_start_loc.cpu().numpy()
    for r in range(w.num_reqs):
        mean_q = qdir[qsl[r]:qsl[r + 1]].mean(0)          # [H, D]
        G = w.num_heads // w.num_kv_heads
        kdir = mean_q.view(w.num_kv_heads, G, -1).mean(1)  # [Hkv, D]
        for t in range(int(L[r])):
            b, o = int(bt[r, t // bs]), t % bs
            w.kv_cache[0, b, o] = (w.kv_cache[0, b, o].float() * 0.3 +
                                   kdir * (t / 32.0)).to(w.dtype)
    out, lse = _run(pa, w)
    ref, ref_lse = oracle_prefill(w)
    check_attention(out, ref, what="growing scores")
    check_lse(lse, ref_lse, what="growing scores lse")


def test_prefill_block_table_slice_with_row_stride(pa):
    """A column slice of the block table (the suffix pass of cascade
    attention) is read through its row stride."""
    w = wl.make_prefill("prefill_tiny", device="cuda", poison=True, q_lens=[5, 40, 1],
                        ctx_lens=[60, 40, 90], seed=10)
    pb = 2
    sl = (w.seq_lens - pb * w.block_size).contiguous()
    view = w.block_tables[:, pb:]
    out, lse = _run(pa, w, block_tables=view, seq_lens=sl)
    ref, ref_lse = oracle_prefill(w, block_tables=view.contiguous(), seq_lens=sl)
    check_attention(out, ref, what="sliced table")
    check_lse(lse, ref_lse, what="sliced table lse")


def test_prefill_rows_outside_requests_untouched(pa):
    w = wl.make_prefill("prefill_tiny", device="cuda", q_lens=[30, 10], ctx_lens=[0, 4],
                        seed=11)
    ref, _ = oracle_prefill(w)
    extra = torch.randn((7,) + tuple(w.q.shape[1:]), device="cuda").to(w.dtype)
    w.q = torch.cat([w.q, extra]).contiguous()
    out = torch.full_like(w.q, 3.0)
    _run(pa, w, out=out, with_lse=False)
    assert torch.all(out[40:] == 3.0)
    check_attention(out[:40], ref, what="packed rows")


def test_prefill_bad_metadata_is_flagged_and_skipped(pa):
    w = wl.make_prefill("prefill_tiny", device="cuda", q_lens=[30, 10], ctx_lens=[0, 4],
                        seed=12)
    sl = w.seq_lens.clone()
    sl[1] = 5                                       # shorter than its 10 query rows
    out = torch.full_like(w.q, 3.0)
    _run(pa, w, out=out, seq_lens=sl, with_lse=False)
    assert pa.pa_device_errors(clear=True) & pa.DEVERR_SEQ_LEN
    assert torch.all(out[30:] == 3.0)
    ref, _ = oracle_prefill(w, seq_lens=w.seq_lens)
    check_attention(out[:30], ref[:30], what="good request")
    bt = w.block_tables.clone()
    bt[0, 0] = w.num_blocks + 4                     # bad id: read as zeros, flagged
    _run(pa, w, out=out, block_tables=bt, with_lse=False)
    assert pa.pa_device_errors(clear=True) & pa.DEVERR_BLOCK_ID
    assert torch.isfinite(out.float()).all()


def test_prefill_deterministic(pa):
    w = wl.make_prefill("prefill_tiny", device="cuda", seed=13)
    a, la = _run(pa, w)
    b, lb = _run(pa, w)
    assert torch.equal(a.view(torch.int16), b.view(torch.int16)) and torch.equal(la, lb)
