"""Shared helpers of the GPU parity tests: run the CUDA library and the CPU
oracle on the same seeded inputs and compare.

Attention tolerance: the required bound is max-abs 2e-3 and max-rel 1e-2 on
fp16/bf16 inputs with fp32 accumulation.  It is applied element by element as
|gpu - ref| <= 2e-3 + 1e-2 * |ref|, with ref the oracle's fp64 result before
output rounding.  (A bf16 output of magnitude ~1 alone carries up to 2^-9 of
rounding error, so a pure 2e-3 absolute bound could not hold; the relative
term covers it.)  Tests also record the maximum absolute error and the
maximum relative error over |ref| >= 1e-2.
"""
from __future__ import annotations

import numpy as np
import torch

from oracle.oracle import get as get_oracle
from workload import ORACLE_DTYPE, Workload, bits

ATOL = 2e-3
RTOL = 1e-2


def oracle_decode(w: Workload, items=None, cache_bits=None) -> np.ndarray:
    orc = get_oracle()
    cb = cache_bits if cache_bits is not None else bits(w.kv_cache)
    return orc.decode(bits(w.q), cb, w.block_tables.cpu().numpy(), w.seq_lens.cpu().numpy(),
                      w.num_kv_heads, w.block_size, w.scale, ORACLE_DTYPE[w.dtype], items=items)


def oracle_prefill(w, items=None, cache_bits=None, causal=True, block_tables=None,
                   seq_lens=None):
    """fp64 (out, lse) of a prefill workload from the oracle."""
    orc = get_oracle()
    cb = cache_bits if cache_bits is not None else bits(w.kv_cache)
    bt = (w.block_tables if block_tables is None else block_tables).cpu().numpy()
    sl = (w.seq_lens if seq_lens is None else seq_lens).cpu().numpy()
    return orc.prefill(bits(w.q), cb, bt, sl, w.query_start_loc.cpu().numpy(), w.num_kv_heads,
                       w.block_size, w.scale, ORACLE_DTYPE[w.dtype], causal=causal,
                       items=items)


def oracle_decode_lse(w: Workload, items=None) -> np.ndarray:
    """Decode rows' natural-log softmax denominators from the oracle's
    prefill with one query row per request (the decode step is that case)."""
    B = w.num_seqs
    _, lse = get_oracle().prefill(bits(w.q), bits(w.kv_cache), w.block_tables.cpu().numpy(),
                                  w.seq_lens.cpu().numpy(), np.arange(B + 1, dtype=np.int32),
                                  w.num_kv_heads, w.block_size, w.scale, ORACLE_DTYPE[w.dtype],
                                  items=items)
    return lse


def check_lse(got: torch.Tensor, ref: np.ndarray, items=None, what: str = ""):
    """Log-sum-exps agree to 1e-3 absolute (the scores are fp32 dot products
    of 16-bit inputs; the log of the denominator is insensitive to P's
    16-bit rounding)."""
    g = got.detach().cpu().numpy().astype(np.float64).reshape(-1)
    r = np.asarray(ref).reshape(-1)
    if items is not None:
        g, r = g[np.asarray(items)], r[np.asarray(items)]
    assert np.isfinite(g).all() and np.isfinite(r).all(), f"{what}: non-finite lse"
    err = np.abs(g - r)
    assert (err <= 1e-3 + 1e-4 * np.abs(r)).all(), f"{what}: lse max err {err.max()}"


def oracle_reshape(w: Workload, cache_bits=None) -> np.ndarray:
    orc = get_oracle()
    cb = cache_bits if cache_bits is not None else bits(w.kv_cache)
    return orc.reshape_and_cache(bits(w.key), bits(w.value), cb, w.slot_mapping.cpu().numpy(),
                                 w.block_size)


def check_attention(got: torch.Tensor, ref: np.ndarray, items=None, what: str = "") -> dict:
    g = got.detach().float().cpu().numpy().astype(np.float64)
    if items is not None:
        B, H, D = g.shape
        g = g.reshape(B * H, D)[np.asarray(items)]
        ref = ref.reshape(B * H, D)[np.asarray(items)]
    assert np.isfinite(ref).all(), f"{what}: oracle produced non-finite values"
    assert np.isfinite(g).all(), f"{what}: GPU output has non-finite values"
    err = np.abs(g - ref)
    bound = ATOL + RTOL * np.abs(ref)
    big = np.abs(ref) >= 1e-2
    stats = {
        "max_abs": float(err.max()) if err.size else 0.0,
        "max_rel_ge_1e-2": float((err[big] / np.abs(ref[big])).max()) if big.any() else 0.0,
        "worst_ratio": float((err / bound).max()) if err.size else 0.0,
    }
    bad = err > bound
    if bad.any():
        idx = np.unravel_index(np.argmax(err / bound), err.shape)
        raise AssertionError(f"{what}: {int(bad.sum())} elements outside tolerance; worst at "
                             f"{idx}: gpu={g[idx]!r} ref={ref[idx]!r} stats={stats}")
    return stats


def splitk_workspace(pa, w: Workload, max_seq_len: int, partition_size: int,
                     pad: int = 0) -> torch.Tensor:
    n = pa.pa_decode_splitk_workspace_size(w.num_seqs, w.num_heads, w.head_size, max_seq_len,
                                           partition_size)
    # 256-byte aligned allocation (the caching allocator gives 512-aligned blocks)
    return torch.empty(n + pad, dtype=torch.uint8, device=w.q.device)
