"""ctypes front end of the CPU oracle in ``pa_oracle.c``.

TEST INFRASTRUCTURE ONLY.  The oracle is the plain CPU statement of paged
decode attention that the CUDA library is checked against.  Only the tests,
``__graft_entry__.smoke()`` and the benchmark's CPU-baseline leg may import
this module; the library itself never does, and it shares no code with it.

Arrays of fp16/bf16 values travel as their uint16 bit patterns, so the oracle
sees exactly the bytes the GPU sees.
"""
from __future__ import annotations

import ctypes
import os
import subprocess
import threading

import numpy as np

FP16 = 0
BF16 = 1

_HERE = os.path.dirname(os.path.abspath(__file__))
SOURCE = os.path.join(_HERE, "pa_oracle.c")
_SO = os.path.join(_HERE, "_build", "liboracle.so")

_ERRORS = {
    -1: "invalid argument",
    -2: "block id out of range",
    -3: "seq_len out of range",
    -4: "slot out of range",
    -5: "out of memory",
}


class OracleError(RuntimeError):
    pass


def compile_source(src: str, so_path: str) -> str:
    """Compile one oracle C source into a shared object with plain gcc."""
    os.makedirs(os.path.dirname(so_path), exist_ok=True)
    tmp = so_path + f".{os.getpid()}.tmp"
    cmd = ["gcc", "-O2", "-std=c11", "-fPIC", "-shared", "-pthread",
           "-fno-fast-math", "-ffp-contract=off", src, "-o", tmp, "-lm"]
    subprocess.run(cmd, check=True)
    os.replace(tmp, so_path)
    return so_path


def build(force: bool = False) -> str:
    """Compile pa_oracle.c into oracle/_build/liboracle.so."""
    if force or not os.path.exists(_SO) or os.path.getmtime(_SO) < os.path.getmtime(SOURCE):
        compile_source(SOURCE, _SO)
    return _SO


def _ptr(a: np.ndarray):
    return a.ctypes.data_as(ctypes.c_void_p)


def _check(rc: int):
    if rc != 0:
        raise OracleError(_ERRORS.get(rc, f"oracle error {rc}"))


def _u16(a) -> np.ndarray:
    a = np.ascontiguousarray(a)
    if a.dtype != np.uint16:
        a = a.view(np.uint16)
    return a


class Oracle:
    """The oracle's entry points, bound to one compiled shared object."""

    def __init__(self, so_path: str):
        lib = ctypes.CDLL(so_path)
        P = ctypes.c_void_p
        i32, i64, dbl = ctypes.c_int, ctypes.c_int64, ctypes.c_double
        lib.or_half_to_double.restype = dbl
        lib.or_half_to_double.argtypes = [ctypes.c_uint16]
        lib.or_bf16_to_double.restype = dbl
        lib.or_bf16_to_double.argtypes = [ctypes.c_uint16]
        lib.or_double_to_half.restype = ctypes.c_uint16
        lib.or_double_to_half.argtypes = [dbl]
        lib.or_double_to_bf16.restype = ctypes.c_uint16
        lib.or_double_to_bf16.argtypes = [dbl]
        lib.or_round.restype = None
        lib.or_round.argtypes = [P, P, i64, i32]
        lib.or_widen.restype = None
        lib.or_widen.argtypes = [P, P, i64, i32]
        lib.or_translate.restype = None
        lib.or_translate.argtypes = [P, i32, i32, P, P]
        lib.or_slot_of_token.restype = i64
        lib.or_slot_of_token.argtypes = [P, i32, i32]
        lib.or_reshape_and_cache.restype = i32
        lib.or_reshape_and_cache.argtypes = [P, P, P, P, i32, i32, i32, i32, i32, i64, i64]
        lib.or_decode.restype = i32
        lib.or_decode.argtypes = [P, P, P, P, P, i32, i32, i32, i32, i32, i32, i32,
                                  dbl, i32, P, i64, i32]
        lib.or_online_softmax.restype = i32
        lib.or_online_softmax.argtypes = [P, P, P, P, P, i32, i32, i32]
        lib.or_merge_partials.restype = i32
        lib.or_merge_partials.argtypes = [P, P, P, P, i32, i32]
        lib.or_copy_blocks.restype = i32
        lib.or_copy_blocks.argtypes = [P, P, i32, i32, i32, i32, i32]
        lib.or_prefill.restype = i32
        lib.or_prefill.argtypes = [P, P, P, P, P, i64, P, P, i32, i32, i32, i32, i32, i32, i32,
                                   dbl, i32, i32, P, i64, i32]
        lib.or_merge_attn_states.restype = i32
        lib.or_merge_attn_states.argtypes = [P, P, P, P, P, P, i64, i32]
        lib.or_fp8e4m3_to_double.restype = dbl
        lib.or_fp8e4m3_to_double.argtypes = [ctypes.c_uint8]
        lib.or_double_to_fp8e4m3.restype = ctypes.c_uint8
        lib.or_double_to_fp8e4m3.argtypes = [dbl]
        lib.or_fp8_widen.restype = None
        lib.or_fp8_widen.argtypes = [P, P, i64]
        lib.or_fp8_quantize.restype = None
        lib.or_fp8_quantize.argtypes = [P, P, i64, ctypes.c_float]
        lib.or_reshape_and_cache_fp8.restype = i32
        lib.or_reshape_and_cache_fp8.argtypes = [P, P, P, P, i32, i32, i32, i32, i32, i64, i64,
                                                 i32, ctypes.c_float, ctypes.c_float]
        lib.or_decode_fp8.restype = i32
        lib.or_decode_fp8.argtypes = [P, P, P, P, P, i32, i32, i32, i32, i32, i32, i32, dbl,
                                      i32, dbl, dbl, P, i64]
        lib.or_check_tables.restype = i32
        lib.or_check_tables.argtypes = [P, P, i32, i32, i32, i32]
        self.lib = lib

    # -- number formats ------------------------------------------------------
    def widen(self, bits, dtype: int) -> np.ndarray:
        """fp16/bf16 bit patterns -> float64 values (IEEE definitions)."""
        b = _u16(bits)
        out = np.empty(b.shape, dtype=np.float64)
        self.lib.or_widen(_ptr(b), _ptr(out), b.size, dtype)
        return out

    def round_to(self, x, dtype: int) -> np.ndarray:
        """float64 values -> fp16/bf16 bit patterns, nearest, ties to even."""
        x = np.ascontiguousarray(x, dtype=np.float64)
        out = np.empty(x.shape, dtype=np.uint16)
        self.lib.or_round(_ptr(x), _ptr(out), x.size, dtype)
        return out

    # -- address translation -------------------------------------------------
    def translate(self, block_table_row, t: int, block_size: int):
        row = np.ascontiguousarray(block_table_row, dtype=np.int32)
        phys = np.zeros(1, np.int32)
        off = np.zeros(1, np.int32)
        self.lib.or_translate(_ptr(row), t, block_size, _ptr(phys), _ptr(off))
        return int(phys[0]), int(off[0])

    def slot_of_token(self, block_table_row, t: int, block_size: int) -> int:
        row = np.ascontiguousarray(block_table_row, dtype=np.int32)
        return int(self.lib.or_slot_of_token(_ptr(row), t, block_size))

    # -- cache write ---------------------------------------------------------
    def reshape_and_cache(self, key, value, cache, slot_mapping, block_size: int,
                          key_stride: int | None = None, value_stride: int | None = None):
        """Return a copy of ``cache`` (uint16 [2, NB, bs, Hkv, D]) with the new
        tokens written.  ``key``/``value`` are uint16 [T, ...] rows."""
        c = np.array(_u16(cache), copy=True)
        two, nb, bs, hkv, d = c.shape
        assert two == 2 and bs == block_size
        k = _u16(key)
        v = _u16(value)
        t = k.shape[0]
        ks = key_stride if key_stride is not None else int(np.prod(k.shape[1:]))
        vs = value_stride if value_stride is not None else int(np.prod(v.shape[1:]))
        sm = np.ascontiguousarray(slot_mapping, dtype=np.int64)
        _check(self.lib.or_reshape_and_cache(_ptr(k), _ptr(v), _ptr(c), _ptr(sm), t, hkv, d,
                                             bs, nb, ks, vs))
        return c

    # -- decode attention ----------------------------------------------------
    def decode(self, q, cache, block_tables, seq_lens, num_kv_heads: int, block_size: int,
               scale: float, dtype: int, items=None, nthreads: int | None = None):
        """fp64 attention output [B, H, D].  ``items`` (seq * H + head) limits
        the rows computed; the other rows are NaN."""
        qb = _u16(q)
        cb = _u16(cache)
        b, h, d = qb.shape
        nb = cb.shape[1]
        bt = np.ascontiguousarray(block_tables, dtype=np.int32)
        sl = np.ascontiguousarray(seq_lens, dtype=np.int32)
        mb = bt.shape[1]
        out = np.full((b, h, d), np.nan, dtype=np.float64)
        if items is not None:
            it = np.ascontiguousarray(items, dtype=np.int32)
            itp, nit = _ptr(it), it.size
        else:
            itp, nit = None, 0
        if nthreads is None:
            nthreads = os.cpu_count() or 1
        _check(self.lib.or_decode(_ptr(out), _ptr(qb), _ptr(cb), _ptr(bt), _ptr(sl), b, h,
                                  num_kv_heads, d, block_size, nb, mb, float(scale), dtype,
                                  itp, nit, int(nthreads)))
        return out

    def online_softmax(self, a, V, block: int):
        """The block-wise online softmax merge; returns (out[D], m, l)."""
        a = np.ascontiguousarray(a, dtype=np.float64)
        V = np.ascontiguousarray(V, dtype=np.float64)
        n, d = V.shape
        out = np.empty(d, np.float64)
        m = np.zeros(1, np.float64)
        l = np.zeros(1, np.float64)
        _check(self.lib.or_online_softmax(_ptr(out), _ptr(m), _ptr(l), _ptr(a), _ptr(V), n,
                                          d, block))
        return out, float(m[0]), float(l[0])

    def merge_partials(self, m, l, o) -> np.ndarray:
        m = np.ascontiguousarray(m, dtype=np.float64)
        l = np.ascontiguousarray(l, dtype=np.float64)
        o = np.ascontiguousarray(o, dtype=np.float64)
        parts, d = o.shape
        out = np.empty(d, np.float64)
        _check(self.lib.or_merge_partials(_ptr(out), _ptr(m), _ptr(l), _ptr(o), parts, d))
        return out

    def copy_blocks(self, cache, mapping):
        """Return a copy of ``cache`` (uint16 [2, NB, bs, Hkv, D]) after copying
        block src -> dst for each (src, dst) row of ``mapping`` in order."""
        c = np.array(_u16(cache), copy=True)
        _, nb, bs, hkv, d = c.shape
        mp = np.ascontiguousarray(mapping, dtype=np.int64).reshape(-1, 2)
        _check(self.lib.or_copy_blocks(_ptr(c), _ptr(mp), mp.shape[0], nb, bs, hkv, d))
        return c

    def prefill(self, q, cache, block_tables, seq_lens, query_start_loc, num_kv_heads: int,
                block_size: int, scale: float, dtype: int, causal: bool = True, items=None,
                nthreads: int | None = None, block_table_stride: int | None = None,
                max_blocks_per_seq: int | None = None):
        """fp64 attention of the packed query rows q [T, H, D] to each request's
        paged keys; returns (out [T, H, D], lse [T, H]).  ``items`` (token * H +
        head) limits the rows computed; the other rows are NaN.  The block table
        may be a 1-D buffer read with an explicit row stride."""
        qb = _u16(q)
        cb = _u16(cache)
        t, h, d = qb.shape
        nb = cb.shape[1]
        bt = np.ascontiguousarray(block_tables, dtype=np.int32)
        if block_table_stride is None:
            block_table_stride = bt.shape[1]
        if max_blocks_per_seq is None:
            max_blocks_per_seq = block_table_stride
        sl = np.ascontiguousarray(seq_lens, dtype=np.int32)
        qsl = np.ascontiguousarray(query_start_loc, dtype=np.int32)
        assert qsl.size == sl.size + 1 and int(qsl[-1]) == t
        out = np.full((t, h, d), np.nan, dtype=np.float64)
        lse = np.full((t, h), np.nan, dtype=np.float64)
        if items is not None:
            it = np.ascontiguousarray(items, dtype=np.int64)
            itp, nit = _ptr(it), it.size
        else:
            itp, nit = None, 0
        if nthreads is None:
            nthreads = os.cpu_count() or 1
        _check(self.lib.or_prefill(_ptr(out), _ptr(lse), _ptr(qb), _ptr(cb), _ptr(bt),
                                   int(block_table_stride), _ptr(sl), _ptr(qsl), sl.size, h,
                                   num_kv_heads, d, block_size, nb, int(max_blocks_per_seq),
                                   float(scale), 1 if causal else 0, dtype, itp, nit,
                                   int(nthreads)))
        return out, lse

    def merge_attn_states(self, o_a, lse_a, o_b, lse_b):
        """Merge two partial attention results given with their log-sum-exps:
        o_x [..., D], lse_x [...]; returns (out, lse)."""
        o_a = np.ascontiguousarray(o_a, dtype=np.float64)
        o_b = np.ascontiguousarray(o_b, dtype=np.float64)
        lse_a = np.ascontiguousarray(lse_a, dtype=np.float64)
        lse_b = np.ascontiguousarray(lse_b, dtype=np.float64)
        assert o_a.shape == o_b.shape and lse_a.shape == lse_b.shape == o_a.shape[:-1]
        d = o_a.shape[-1]
        out = np.empty_like(o_a)
        lse = np.empty_like(lse_a)
        _check(self.lib.or_merge_attn_states(_ptr(out), _ptr(lse), _ptr(o_a), _ptr(lse_a),
                                             _ptr(o_b), _ptr(lse_b), lse_a.size, d))
        return out, lse

    # -- FP8 (e4m3) KV cache ----------------------------------------------------
    def fp8_widen(self, codes) -> np.ndarray:
        """e4m3 codes (uint8) -> float64 values."""
        c = np.ascontiguousarray(codes, dtype=np.uint8)
        out = np.empty(c.shape, dtype=np.float64)
        self.lib.or_fp8_widen(_ptr(c), _ptr(out), c.size)
        return out

    def fp8_quantize(self, x, scale: float) -> np.ndarray:
        """float32 values -> e4m3 codes of fp32(x / scale)."""
        x = np.ascontiguousarray(x, dtype=np.float32)
        out = np.empty(x.shape, dtype=np.uint8)
        self.lib.or_fp8_quantize(_ptr(x), _ptr(out), x.size, float(scale))
        return out

    def fp8_encode(self, x: float) -> int:
        return int(self.lib.or_double_to_fp8e4m3(float(x)))

    def reshape_and_cache_fp8(self, key, value, cache, slot_mapping, block_size: int,
                              src_dtype: int, k_scale: float, v_scale: float):
        """Copy of the uint8 pool ``cache`` [2, NB, bs, Hkv, D] with the new
        tokens quantised and written."""
        c = np.array(np.ascontiguousarray(cache, dtype=np.uint8), copy=True)
        _, nb, bs, hkv, d = c.shape
        assert bs == block_size
        k = _u16(key)
        v = _u16(value)
        t = k.shape[0]
        sm = np.ascontiguousarray(slot_mapping, dtype=np.int64)
        _check(self.lib.or_reshape_and_cache_fp8(_ptr(k), _ptr(v), _ptr(c), _ptr(sm), t, hkv, d,
                                                 bs, nb, int(np.prod(k.shape[1:])),
                                                 int(np.prod(v.shape[1:])), src_dtype,
                                                 float(k_scale), float(v_scale)))
        return c

    def decode_fp8(self, q, cache, block_tables, seq_lens, num_kv_heads: int, block_size: int,
                   scale: float, q_dtype: int, k_scale: float, v_scale: float, items=None):
        """fp64 decode output [B, H, D] over a uint8 e4m3 pool."""
        qb = _u16(q)
        cb = np.ascontiguousarray(cache, dtype=np.uint8)
        b, h, d = qb.shape
        bt = np.ascontiguousarray(block_tables, dtype=np.int32)
        sl = np.ascontiguousarray(seq_lens, dtype=np.int32)
        out = np.full((b, h, d), np.nan, dtype=np.float64)
        if items is not None:
            it = np.ascontiguousarray(items, dtype=np.int32)
            itp, nit = _ptr(it), it.size
        else:
            itp, nit = None, 0
        _check(self.lib.or_decode_fp8(_ptr(out), _ptr(qb), _ptr(cb), _ptr(bt), _ptr(sl), b, h,
                                      num_kv_heads, d, block_size, cb.shape[1], bt.shape[1],
                                      float(scale), q_dtype, float(k_scale), float(v_scale),
                                      itp, nit))
        return out

    def check_tables(self, block_tables, seq_lens, block_size: int, num_blocks: int) -> int:
        bt = np.ascontiguousarray(block_tables, dtype=np.int32)
        sl = np.ascontiguousarray(seq_lens, dtype=np.int32)
        return int(self.lib.or_check_tables(_ptr(bt), _ptr(sl), sl.size, bt.shape[1],
                                            block_size, num_blocks))


_default = None
_lock = threading.Lock()


def get() -> Oracle:
    """The oracle built from oracle/pa_oracle.c (compiled on first use)."""
    global _default
    with _lock:
        if _default is None:
            _default = Oracle(build())
    return _default
