"""CUDA library vs the CPU oracle on the five workloads and a shape sweep.

Every call goes through the C ABI (the ctypes binding).  Pools are
NaN-poisoned wherever no sequence owns a row, so a read past a sequence's end
shows up as a non-finite output.
"""
import numpy as np
import pytest
import torch

import workload as wl
from tests._parity import (check_attention, oracle_decode, oracle_reshape,
                           splitk_workspace)

pytestmark = pytest.mark.gpu


@pytest.fixture(scope="module")
def pa():
    from __graft_entry__ import build_library
    build_library()
    import paged_kv_cache_136_gb300 as pa
    assert pa.pa_device_errors(clear=True) >= 0
    return pa


def _no_device_errors(pa):
    assert pa.pa_device_errors(clear=True) == 0


# ---------------------------------------------------------------------------
# Cache write: bit-exact
# ---------------------------------------------------------------------------

@pytest.mark.parametrize("name", ["tiny", "mha7b", "gqa8b"])
def test_reshape_and_cache_bit_exact(pa, name):
    w = wl.make(name, device="cuda", poison=True)
    before = wl.bits(w.kv_cache)
    ref = oracle_reshape(w, before)
    pa.pa_reshape_and_cache(w.key, w.value, w.kv_cache, w.slot_mapping, w.block_size)
    torch.cuda.synchronize()
    got = wl.bits(w.kv_cache)
    assert np.array_equal(got, ref)
    _no_device_errors(pa)


def test_reshape_and_cache_strided_rows(pa):
    w = wl.make("tiny", device="cuda")
    T, hkv, d = w.key.shape
    big_k = torch.randn(T, hkv * d + 64, device="cuda").to(w.dtype)
    big_v = torch.randn(T, hkv * d + 64, device="cuda").to(w.dtype)
    k = big_k[:, : hkv * d].view(T, hkv, d)
    v = big_v[:, : hkv * d].view(T, hkv, d)
    assert k.stride(0) == hkv * d + 64
    before = wl.bits(w.kv_cache)
    from oracle.oracle import get
    ref = get().reshape_and_cache(wl.bits(big_k), wl.bits(big_v), before,
                                  w.slot_mapping.cpu().numpy(), w.block_size,
                                  key_stride=hkv * d + 64, value_stride=hkv * d + 64)
    pa.pa_reshape_and_cache(k, v, w.kv_cache, w.slot_mapping, w.block_size)
    torch.cuda.synchronize()
    assert np.array_equal(wl.bits(w.kv_cache), ref)


def test_reshape_and_cache_all_padding_writes_nothing(pa):
    w = wl.make("tiny", device="cuda")
    before = wl.bits(w.kv_cache)
    pa.pa_reshape_and_cache(w.key, w.value, w.kv_cache, torch.full_like(w.slot_mapping, -1),
                            w.block_size)
    torch.cuda.synchronize()
    assert np.array_equal(wl.bits(w.kv_cache), before)


# ---------------------------------------------------------------------------
# Decode: all five workloads at full size
# ---------------------------------------------------------------------------

def _step(pa, w, split: bool, partition_size: int = 512):
    """One hot-path step: write the new tokens, then decode."""
    pa.pa_reshape_and_cache(w.key, w.value, w.kv_cache, w.slot_mapping, w.block_size)
    out = torch.empty_like(w.q)
    if split:
        msl = int(w.seq_lens.max().item())
        ws = splitk_workspace(pa, w, msl, partition_size)
        pa.pa_decode_splitk(out, w.q, w.kv_cache, w.block_tables, w.seq_lens, w.scale,
                            w.block_size, msl, ws, partition_size)
    else:
        pa.pa_decode(out, w.q, w.kv_cache, w.block_tables, w.seq_lens, w.scale, w.block_size)
    torch.cuda.synchronize()
    return out


def _sample_items(w, n, seed=0):
    rng = np.random.default_rng(seed)
    total = w.num_seqs * w.num_heads
    return np.sort(rng.choice(total, min(n, total), replace=False)).astype(np.int32)


@pytest.mark.parametrize("name,split", [
    ("tiny", False), ("tiny", True), ("mha7b", False), ("mha7b", True),
    ("gqa8b", False), ("gqa8b", True), ("prefix", False), ("prefix", True),
])
def test_decode_matches_oracle(pa, name, split):
    w = wl.make(name, device="cuda", poison=True)
    out = _step(pa, w, split)
    ref = oracle_decode(w)        # oracle reads the pool after the cache write
    check_attention(out, ref, what=f"{name} split={split}")
    _no_device_errors(pa)


@pytest.mark.parametrize("split", [True, False])
def test_long_context_sampled(pa, split):
    """8 x 131072 tokens, 64/8 heads, bf16: sampled rows vs the oracle."""
    w = wl.make("long", device="cuda", poison=True)
    out = _step(pa, w, split)
    items = _sample_items(w, 48, seed=1)
    ref = oracle_decode(w, items=items)
    check_attention(out, ref, items=items, what=f"long split={split}")
    _no_device_errors(pa)


# ---------------------------------------------------------------------------
# Shape sweep: every built (head_size, block_size, group, dtype) combination,
# ragged lengths around block and stage boundaries.
# ---------------------------------------------------------------------------

SWEEP_LENS = [1, 15, 16, 17, 63, 64, 65, 200, 511, 512, 513, 1023]


@pytest.mark.parametrize("dtype", [torch.float16, torch.bfloat16])
@pytest.mark.parametrize("D", [64, 128])
@pytest.mark.parametrize("bs", [16, 32])
@pytest.mark.parametrize("G", [1, 2, 4, 8])
def test_shape_sweep(pa, dtype, D, bs, G):
    Hkv = 2
    w = wl.make("gqa8b", device="cuda", poison=True, lengths=SWEEP_LENS, num_heads=G * Hkv,
                num_kv_heads=Hkv, head_size=D, block_size=bs, dtype=dtype, seed=G * 1000 + D + bs)
    ref_cache = None
    for split in (False, True):
        if split:
            w.kv_cache.copy_(ref_cache)
        else:
            ref_cache = w.kv_cache.clone()
        out = _step(pa, w, split, partition_size=128)
        if not split:
            ref = oracle_decode(w)
        check_attention(out, ref, what=f"D={D} bs={bs} G={G} {dtype} split={split}")
    _no_device_errors(pa)
