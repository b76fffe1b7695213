"""Shared helpers of the GPU parity tests: run the CUDA library and the CPU
oracle on the same seeded inputs and compare.

Attention tolerance.  The required bound is max-abs error 2e-3 and max-rel
error 1e-2 for fp16/bf16 inputs with fp32 accumulation.  `ref` is the
oracle's fp64 result before output rounding.

- fp16 outputs: the bound as stated.  max |gpu - ref| <= 2e-3 over every
  element, and max |gpu - ref| / |ref| <= 1e-2 over the elements with
  |ref| >= 1e-2 (below that, relative error of a value that is mostly
  cancellation carries no information and the absolute bound governs).  An
  fp16 output below 4 carries at most 2^-10 of its own rounding, so the
  absolute bound leaves room for the fp32 arithmetic.
- bf16 outputs: the relative bound as stated.  The absolute bound is taken on
  the error beyond the output's own rounding: |gpu - ref| <= 2e-3 + half a
  bf16 ulp at max(|gpu|, |ref|).  A bf16 value in [1, 2) is a multiple of
  2^-7, so its correctly rounded form alone can be 3.9e-3 away from ref and
  the plain absolute bound could not hold for any bf16 kernel.

Every call records its error statistics; when the environment variable
PA_PARITY_LOG names a file, one JSON line per call is appended to it (test
id, output dtype, element count, max-abs, max-rel over |ref| >= 1e-2, the
worst error beyond output rounding).
"""
from __future__ import annotations

import json
import os

import numpy as np
import torch

from oracle.oracle import get as get_oracle
from workload import ORACLE_DTYPE, Workload, bits

ATOL = 2e-3          # max-abs bound
RTOL = 1e-2          # max-rel bound
REL_FLOOR = 1e-2     # max-rel is taken over |ref| >= REL_FLOOR

# significand bits after the leading one, and the smallest normal exponent
_FORMAT = {torch.float16: (10, -14), torch.bfloat16: (7, -126)}


def half_ulp(x: np.ndarray, dtype: torch.dtype) -> np.ndarray:
    """Half the spacing of `dtype` values at magnitude |x| (the largest
    rounding error of a correctly rounded result there)."""
    mant, emin = _FORMAT[dtype]
    a = np.abs(np.asarray(x, dtype=np.float64))
    e = np.floor(np.log2(np.where(a > 0, a, 1.0)))
    e = np.maximum(e, emin)
    return np.ldexp(0.5, (e - mant).astype(np.int64))


def _log(rec: dict) -> None:
    path = os.environ.get("PA_PARITY_LOG")
    if not path:
        return
    rec = dict(rec, test=os.environ.get("PYTEST_CURRENT_TEST", "").split(" ")[0])
    with open(path, "a") as f:
        f.write(json.dumps(rec) + "\n")


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
    """Log-sum-exps agree to 2e-5 absolute plus 1e-6 relative.  The kernels
    form the softmax denominator as an fp32 sum of fp32 exponentials of fp32
    scores (exact products of the 16-bit inputs): its relative error is a
    few fp32 ulps times the depth of the summation tree, about 1e-6 for the
    lengths tested, and the log turns that relative error into an absolute
    one.  The relative term covers the fp32 rounding of the running maximum
    added back (an fp32 ulp of lse is 1.2e-7 * |lse|)."""
    g = got.detach().cpu().numpy().astype(np.float64).reshape(-1)
    r = np.asarray(ref).reshape(-1)
    if items is not None:
        g, r = g[np.asarray(items)], r[np.asarray(items)]
    assert np.isfinite(g).all() and np.isfinite(r).all(), f"{what}: non-finite lse"
    err = np.abs(g - r)
    _log({"what": what + " [lse]", "dtype": "float32", "n": int(err.size),
          "max_abs": float(err.max()) if err.size else 0.0})
    assert (err <= 2e-5 + 1e-6 * np.abs(r)).all(), f"{what}: lse max err {err.max()}"


def oracle_reshape(w: Workload, cache_bits=None) -> np.ndarray:
    orc = get_oracle()
    cb = cache_bits if cache_bits is not None else bits(w.kv_cache)
    return orc.reshape_and_cache(bits(w.key), bits(w.value), cb, w.slot_mapping.cpu().numpy(),
                                 w.block_size)


def attention_stats(g: np.ndarray, ref: np.ndarray, dtype: torch.dtype) -> dict:
    """Error statistics of output `g` (fp64 copy of a `dtype` tensor) against
    the fp64 reference."""
    err = np.abs(g - ref)
    big = np.abs(ref) >= REL_FLOOR
    excess = err - half_ulp(np.maximum(np.abs(g), np.abs(ref)), dtype)
    return {
        "n": int(err.size),
        "max_abs": float(err.max()) if err.size else 0.0,
        "max_rel_ge_1e-2": float((err[big] / np.abs(ref[big])).max()) if big.any() else 0.0,
        "max_abs_beyond_rounding": float(excess.max()) if err.size else 0.0,
    }


def check_attention(got: torch.Tensor, ref: np.ndarray, items=None, what: str = "") -> dict:
    """Assert the attention tolerance (module docstring) element by element;
    return the error statistics."""
    dtype = got.dtype
    assert dtype in _FORMAT, f"{what}: unexpected output dtype {dtype}"
    g = got.detach().float().cpu().numpy().astype(np.float64)
    ref = np.asarray(ref, dtype=np.float64)
    if items is not None:
        B, H, D = g.shape
        g = g.reshape(B * H, D)[np.asarray(items)]
        ref = ref.reshape(B * H, D)[np.asarray(items)]
    assert np.isfinite(ref).all(), f"{what}: oracle produced non-finite values"
    assert np.isfinite(g).all(), f"{what}: GPU output has non-finite values"
    stats = attention_stats(g, ref, dtype)
    _log({"what": what, "dtype": str(dtype).replace("torch.", ""), **stats})
    err = np.abs(g - ref)
    abs_bound = np.full_like(err, ATOL)
    if dtype == torch.bfloat16:
        abs_bound += half_ulp(np.maximum(np.abs(g), np.abs(ref)), dtype)
    big = np.abs(ref) >= REL_FLOOR
    bad_abs = err > abs_bound
    bad_rel = big & (err > RTOL * np.abs(ref))
    bad = bad_abs | bad_rel
    if bad.any():
        score = np.maximum(err / abs_bound, np.where(big, err / (RTOL * np.abs(ref) + 1e-300), 0))
        idx = np.unravel_index(np.argmax(score), err.shape)
        raise AssertionError(
            f"{what}: {int(bad_abs.sum())} elements over the abs bound, {int(bad_rel.sum())} "
            f"over the rel bound; worst at {idx}: gpu={g[idx]!r} ref={ref[idx]!r} "
            f"stats={stats}")
    return stats


def check_agree(a: torch.Tensor, b: torch.Tensor, what: str = "") -> float:
    """Two GPU results of the same attention (different partitionings) agree
    within the abs bound plus one output ulp: each is a correctly rounded
    fp32 accumulation of the same sum, which may round to neighbouring
    values."""
    x = a.detach().float().cpu().numpy().astype(np.float64)
    y = b.detach().float().cpu().numpy().astype(np.float64)
    d = np.abs(x - y)
    bound = ATOL + 2.0 * half_ulp(np.maximum(np.abs(x), np.abs(y)), a.dtype)
    assert (d <= bound).all(), f"{what}: max diff {d.max()} (bound there {bound.flat[d.argmax()]})"
    return float(d.max()) if d.size else 0.0


def splitk_workspace(pa, w: Workload, max_seq_len: int, partition_size: int,
                     pad: int = 0) -> torch.Tensor:
    n = pa.pa_decode_splitk_workspace_size(w.num_seqs, w.num_heads, w.head_size, max_seq_len,
                                           partition_size)
    # 256-byte aligned allocation (the caching allocator gives 512-aligned blocks)
    return torch.empty(n + pad, dtype=torch.uint8, device=w.q.device)
