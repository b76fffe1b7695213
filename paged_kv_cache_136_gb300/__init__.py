"""Python binding of libpa.so: paged KV-cache decode attention on GB300.

Argument marshalling only.  Each function takes torch tensors, checks their
device/dtype/shape, and calls the C entry point of the same name
(``include/pa.h``) with raw device pointers and the current CUDA stream.  All
computation runs in the library's CUDA kernels; there is no fallback path.
Importing this package fails loudly if libpa.so has not been built.
"""
from __future__ import annotations

import ctypes
import os

import torch

_LIB_PATH = os.path.join(os.path.dirname(os.path.abspath(__file__)), "_lib", "libpa.so")

__all__ = [
    "PAError", "lib_path", "pa_reshape_and_cache", "pa_decode", "pa_decode_splitk",
    "pa_decode_splitk_workspace_size", "pa_decode_splitk_noalloc", "NOALLOC_SCRATCH_BYTES",
    "pa_validate_tables", "pa_validate_slots",
    "pa_device_errors", "pa_selftest_wait_timeout", "pa_copy_blocks", "pa_prefill",
    "pa_decode_splitk_lse", "pa_merge_attn_states", "pa_cascade_decode",
    "pa_cascade_decode_workspace_size", "pa_reshape_and_cache_fp8", "pa_decode_fp8",
    "pa_decode_splitk_fp8", "pa_decode_splitk_fp8_workspace_size",
    "pa_validate_block_mapping", "pa_status_string", "pa_version", "pa_profile_kernel_events",
    "DEVERR_BLOCK_ID",
    "DEVERR_SEQ_LEN", "DEVERR_SLOT", "DEVERR_TIMEOUT",
]

PA_OK = 0
DEVERR_BLOCK_ID = 0x1
DEVERR_SEQ_LEN = 0x2
DEVERR_SLOT = 0x4
DEVERR_TIMEOUT = 0x8
DEVERR_PREFIX = 0x10

_DTYPE = {torch.float16: 0, torch.bfloat16: 1}

if not os.path.exists(_LIB_PATH):
    raise ImportError(
        f"libpa.so not found at {_LIB_PATH}; build it first with "
        "`python paged_kv_cache_136_gb300/build.py` (nvcc, sm_103a)")

_lib = ctypes.CDLL(_LIB_PATH)
_P, _I, _I64, _F, _SZ, _U = (ctypes.c_void_p, ctypes.c_int, ctypes.c_int64, ctypes.c_float,
                             ctypes.c_size_t, ctypes.c_uint)
_lib.pa_reshape_and_cache.restype = _I
_lib.pa_reshape_and_cache.argtypes = [_P, _P, _P, _P, _I, _I, _I, _I, _I, _I64, _I64, _I, _P]
_lib.pa_decode.restype = _I
_lib.pa_decode.argtypes = [_P, _P, _P, _P, _P, _I, _I, _I, _I, _I, _I, _I, _F, _I, _P]
_lib.pa_decode_splitk_workspace_size.restype = _SZ
_lib.pa_decode_splitk_workspace_size.argtypes = [_I, _I, _I, _I, _I]
_lib.pa_decode_splitk.restype = _I
_lib.pa_decode_splitk.argtypes = [_P, _P, _P, _P, _P, _I, _I, _I, _I, _I, _I, _I, _F, _I,
                                  _I, _I, _P, _SZ, _P]
_lib.pa_decode_splitk_noalloc.restype = _I
_lib.pa_decode_splitk_noalloc.argtypes = [_P, _P, _P, _P, _P, _I, _I, _I, _I, _I, _I, _I, _F,
                                          _I, _I, _I, _P]
_lib.pa_validate_tables.restype = _I
_lib.pa_validate_tables.argtypes = [_P, _P, _I, _I, _I, _I]
_lib.pa_validate_slots.restype = _I
_lib.pa_validate_slots.argtypes = [_P, _I, _I, _I]
_lib.pa_device_errors.restype = _I
_lib.pa_device_errors.argtypes = [ctypes.POINTER(_U), _I]
_lib.pa_decode_splitk_lse.restype = _I
_lib.pa_decode_splitk_lse.argtypes = [_P, _P, _P, _P, _P, _P, _I, _I, _I, _I, _I, _I, _I, _F,
                                      _I, _I, _I, _P, _SZ, _P]
_lib.pa_stage_copy.restype = _I
_lib.pa_stage_copy.argtypes = [_P, _P, _SZ, _P]
_lib.pa_merge_attn_states.restype = _I
_lib.pa_merge_attn_states.argtypes = [_P, _P, _P, _P, _P, _P, _I, _I, _I, _I, _P]
_lib.pa_cascade_decode_workspace_size.restype = _SZ
_lib.pa_cascade_decode_workspace_size.argtypes = [_I, _I, _I, _I, _I, _I, _I, _I]
_lib.pa_cascade_decode.restype = _I
_lib.pa_cascade_decode.argtypes = [_P, _P, _P, _P, _P, _I, _I, _I, _I, _I, _I, _I, _I, _F, _I,
                                   _I, _I, _P, _SZ, _P]
_lib.pa_reshape_and_cache_fp8.restype = _I
_lib.pa_reshape_and_cache_fp8.argtypes = [_P, _P, _P, _P, _I, _I, _I, _I, _I, _I64, _I64, _I, _F,
                                          _F, _P]
_lib.pa_decode_fp8.restype = _I
_lib.pa_decode_fp8.argtypes = [_P, _P, _P, _P, _P, _I, _I, _I, _I, _I, _I, _I, _F, _F, _F, _I,
                               _P]
_lib.pa_decode_splitk_fp8_workspace_size.restype = _SZ
_lib.pa_decode_splitk_fp8_workspace_size.argtypes = [_I, _I, _I, _I, _I]
_lib.pa_decode_splitk_fp8.restype = _I
_lib.pa_decode_splitk_fp8.argtypes = [_P, _P, _P, _P, _P, _I, _I, _I, _I, _I, _I, _I, _F, _F,
                                      _F, _I, _I, _I, _P, _SZ, _P]
_lib.pa_prefill.restype = _I
_lib.pa_prefill.argtypes = [_P, _P, _P, _P, _P, _I64, _P, _P, _I, _I, _I, _I, _I, _I, _I, _I,
                            _I, _F, _I, _I, _P]
_lib.pa_copy_blocks.restype = _I
_lib.pa_copy_blocks.argtypes = [_P, _P, _I, _I, _I, _I, _I, _I, _P]
_lib.pa_validate_block_mapping.restype = _I
_lib.pa_validate_block_mapping.argtypes = [_P, _I, _I]
_lib.pa_selftest_wait_timeout.restype = _I
_lib.pa_selftest_wait_timeout.argtypes = [_P]
_lib.pa_profile_kernel_events.restype = _I
_lib.pa_profile_kernel_events.argtypes = [_P, _P]
_lib.pa_status_string.restype = ctypes.c_char_p
_lib.pa_status_string.argtypes = [_I]
_lib.pa_version.restype = _I
_lib.pa_version.argtypes = []


class PAError(RuntimeError):
    def __init__(self, status: int, where: str):
        super().__init__(f"{where}: {pa_status_string(status)} ({status})")
        self.status = status


def lib_path() -> str:
    return _LIB_PATH


def pa_status_string(status: int) -> str:
    return _lib.pa_status_string(status).decode()


def pa_version() -> int:
    return _lib.pa_version()


def _check(status: int, where: str):
    if status != PA_OK:
        raise PAError(status, where)


def _dev(t: torch.Tensor, name: str):
    if not isinstance(t, torch.Tensor) or not t.is_cuda:
        raise ValueError(f"{name} must be a CUDA tensor")
    return t.data_ptr()


# The current device's current CUDA stream as a raw handle.  torch's internal
# accessor skips building a torch.cuda.Stream object on every call (a few
# microseconds per call in a decode loop); the public API is the fallback.
_raw_current_stream = getattr(torch._C, "_cuda_getCurrentRawStream", None)
_current_device = getattr(torch._C, "_cuda_getDevice", None)


def _stream(stream):
    if stream is None:
        if _raw_current_stream is not None and _current_device is not None:
            return _raw_current_stream(_current_device())
        return torch.cuda.current_stream().cuda_stream
    if isinstance(stream, torch.cuda.Stream):
        return stream.cuda_stream
    return int(stream)


def _pool_dims(kv_cache: torch.Tensor, block_size: int):
    if kv_cache.dim() != 5 or kv_cache.shape[0] != 2 or kv_cache.shape[2] != block_size:
        raise ValueError("kv_cache must be [2, num_blocks, block_size, num_kv_heads, head_size]")
    if not kv_cache.is_contiguous():
        raise ValueError("kv_cache must be contiguous")
    _, nb, _, hkv, d = kv_cache.shape
    return int(nb), int(hkv), int(d)


def pa_reshape_and_cache(key: torch.Tensor, value: torch.Tensor, kv_cache: torch.Tensor,
                         slot_mapping: torch.Tensor, block_size: int, stream=None) -> None:
    """Scatter new tokens' K/V ([T, Hkv, D], rows may be strided) into the pool
    at slot_mapping (int64, negative = padding)."""
    nb, hkv, d = _pool_dims(kv_cache, block_size)
    T = int(key.shape[0])
    for name, t in (("key", key), ("value", value)):
        if t.dtype != kv_cache.dtype or t.shape[0] != T:
            raise ValueError(f"{name} must match kv_cache dtype and token count")
        if t.dim() != 3 or t.shape[1] != hkv or t.shape[2] != d or t.stride(2) != 1 or t.stride(1) != d:
            raise ValueError(f"{name} must be [T, num_kv_heads, head_size] with contiguous rows")
    if slot_mapping.dtype != torch.int64 or slot_mapping.numel() != T or not slot_mapping.is_contiguous():
        raise ValueError("slot_mapping must be contiguous int64 [T]")
    if kv_cache.dtype not in _DTYPE:
        raise ValueError("dtype must be float16 or bfloat16")
    if T == 0:
        return
    _check(_lib.pa_reshape_and_cache(_dev(key, "key"), _dev(value, "value"),
                                     _dev(kv_cache, "kv_cache"), _dev(slot_mapping, "slot_mapping"),
                                     T, hkv, d, block_size, nb, key.stride(0), value.stride(0),
                                     _DTYPE[kv_cache.dtype], _stream(stream)),
           "pa_reshape_and_cache")


def _decode_common(out, q, kv_cache, block_tables, seq_lens, block_size):
    nb, hkv, d = _pool_dims(kv_cache, block_size)
    if q.dim() != 3 or q.shape[2] != d or not q.is_contiguous():
        raise ValueError("q must be contiguous [B, H, head_size]")
    if out.shape != q.shape or out.dtype != q.dtype or not out.is_contiguous():
        raise ValueError("out must be contiguous and match q")
    if q.dtype != kv_cache.dtype or q.dtype not in _DTYPE:
        raise ValueError("q, kv_cache and out must share dtype float16 or bfloat16")
    B, H = int(q.shape[0]), int(q.shape[1])
    if block_tables.dtype != torch.int32 or block_tables.dim() != 2 or block_tables.shape[0] != B \
            or not block_tables.is_contiguous():
        raise ValueError("block_tables must be contiguous int32 [B, max_blocks_per_seq]")
    if seq_lens.dtype != torch.int32 or seq_lens.numel() != B or not seq_lens.is_contiguous():
        raise ValueError("seq_lens must be contiguous int32 [B]")
    return B, H, hkv, d, nb, int(block_tables.shape[1])


def pa_decode(out: torch.Tensor, q: torch.Tensor, kv_cache: torch.Tensor,
              block_tables: torch.Tensor, seq_lens: torch.Tensor, scale: float,
              block_size: int, stream=None) -> torch.Tensor:
    """One-pass paged decode attention; writes and returns ``out``."""
    B, H, hkv, d, nb, mb = _decode_common(out, q, kv_cache, block_tables, seq_lens, block_size)
    _check(_lib.pa_decode(_dev(out, "out"), _dev(q, "q"), _dev(kv_cache, "kv_cache"),
                          _dev(block_tables, "block_tables"), _dev(seq_lens, "seq_lens"),
                          B, H, hkv, d, block_size, nb, mb, float(scale), _DTYPE[q.dtype],
                          _stream(stream)), "pa_decode")
    return out


def pa_decode_splitk_workspace_size(num_seqs: int, num_heads: int, head_size: int,
                                    max_seq_len: int, partition_size: int = 512) -> int:
    return int(_lib.pa_decode_splitk_workspace_size(num_seqs, num_heads, head_size,
                                                    max_seq_len, partition_size))


def pa_decode_splitk(out: torch.Tensor, q: torch.Tensor, kv_cache: torch.Tensor,
                     block_tables: torch.Tensor, seq_lens: torch.Tensor, scale: float,
                     block_size: int, max_seq_len: int, workspace: torch.Tensor,
                     partition_size: int = 512, stream=None) -> torch.Tensor:
    """Partitioned paged decode attention with log-sum-exp reduce; ``workspace``
    is a CUDA byte tensor of at least pa_decode_splitk_workspace_size bytes."""
    B, H, hkv, d, nb, mb = _decode_common(out, q, kv_cache, block_tables, seq_lens, block_size)
    ws_bytes = workspace.numel() * workspace.element_size()
    _check(_lib.pa_decode_splitk(_dev(out, "out"), _dev(q, "q"), _dev(kv_cache, "kv_cache"),
                                 _dev(block_tables, "block_tables"), _dev(seq_lens, "seq_lens"),
                                 B, H, hkv, d, block_size, nb, mb, float(scale), _DTYPE[q.dtype],
                                 int(max_seq_len), int(partition_size),
                                 _dev(workspace, "workspace"), ws_bytes, _stream(stream)),
           "pa_decode_splitk")
    return out


def _lse_arg(lse, rows: int, cols: int, name: str = "lse"):
    if lse.dtype != torch.float32 or tuple(lse.shape) != (rows, cols) or not lse.is_contiguous():
        raise ValueError(f"{name} must be contiguous float32 [{rows}, {cols}]")
    return _dev(lse, name)


def pa_decode_splitk_lse(out: torch.Tensor, lse: torch.Tensor, q: torch.Tensor,
                         kv_cache: torch.Tensor, block_tables: torch.Tensor,
                         seq_lens: torch.Tensor, scale: float, block_size: int,
                         max_seq_len: int, workspace: torch.Tensor, partition_size: int = 512,
                         stream=None) -> torch.Tensor:
    """pa_decode_splitk that also writes the natural-log softmax denominators
    into ``lse`` (float32 [B, H])."""
    B, H, hkv, d, nb, mb = _decode_common(out, q, kv_cache, block_tables, seq_lens, block_size)
    lp = _lse_arg(lse, B, H)
    ws_bytes = workspace.numel() * workspace.element_size()
    _check(_lib.pa_decode_splitk_lse(_dev(out, "out"), lp, _dev(q, "q"),
                                     _dev(kv_cache, "kv_cache"), _dev(block_tables, "block_tables"),
                                     _dev(seq_lens, "seq_lens"), B, H, hkv, d, block_size, nb, mb,
                                     float(scale), _DTYPE[q.dtype], int(max_seq_len),
                                     int(partition_size), _dev(workspace, "workspace"), ws_bytes,
                                     _stream(stream)), "pa_decode_splitk_lse")
    return out


def pa_merge_attn_states(out: torch.Tensor, o_a: torch.Tensor, lse_a: torch.Tensor,
                         o_b: torch.Tensor, lse_b: torch.Tensor,
                         out_lse: torch.Tensor | None = None, stream=None) -> torch.Tensor:
    """Merge two partial attention results [T, H, D] given with their
    log-sum-exps [T, H]; writes and returns ``out``."""
    for name, t in (("out", out), ("o_a", o_a), ("o_b", o_b)):
        if t.dim() != 3 or t.shape != o_a.shape or t.dtype != o_a.dtype or not t.is_contiguous():
            raise ValueError(f"{name} must be contiguous [T, H, D] like o_a")
    if o_a.dtype not in _DTYPE:
        raise ValueError("dtype must be float16 or bfloat16")
    T, H, D = (int(x) for x in o_a.shape)
    la, lb = _lse_arg(lse_a, T, H, "lse_a"), _lse_arg(lse_b, T, H, "lse_b")
    lo = _lse_arg(out_lse, T, H, "out_lse") if out_lse is not None else ctypes.c_void_p(0)
    if T == 0:
        return out
    _check(_lib.pa_merge_attn_states(_dev(out, "out"), lo, _dev(o_a, "o_a"), la,
                                     _dev(o_b, "o_b"), lb, T, H, D, _DTYPE[o_a.dtype],
                                     _stream(stream)), "pa_merge_attn_states")
    return out


def pa_cascade_decode_workspace_size(num_seqs: int, num_heads: int, head_size: int,
                                     max_blocks_per_seq: int, prefix_blocks: int,
                                     max_seq_len: int, block_size: int,
                                     partition_size: int = 512) -> int:
    return int(_lib.pa_cascade_decode_workspace_size(num_seqs, num_heads, head_size,
                                                     max_blocks_per_seq, prefix_blocks,
                                                     max_seq_len, block_size, partition_size))


def pa_cascade_decode(out: torch.Tensor, q: torch.Tensor, kv_cache: torch.Tensor,
                      block_tables: torch.Tensor, seq_lens: torch.Tensor, scale: float,
                      block_size: int, prefix_blocks: int, max_seq_len: int,
                      workspace: torch.Tensor, partition_size: int = 512,
                      stream=None) -> torch.Tensor:
    """Decode attention for sequences whose tables share their first
    ``prefix_blocks`` blocks (cascade: prefix once, suffixes, merge)."""
    B, H, hkv, d, nb, mb = _decode_common(out, q, kv_cache, block_tables, seq_lens, block_size)
    ws_bytes = workspace.numel() * workspace.element_size()
    _check(_lib.pa_cascade_decode(_dev(out, "out"), _dev(q, "q"), _dev(kv_cache, "kv_cache"),
                                  _dev(block_tables, "block_tables"), _dev(seq_lens, "seq_lens"),
                                  B, H, hkv, d, block_size, nb, mb, int(prefix_blocks),
                                  float(scale), _DTYPE[q.dtype], int(max_seq_len),
                                  int(partition_size), _dev(workspace, "workspace"), ws_bytes,
                                  _stream(stream)), "pa_cascade_decode")
    return out


NOALLOC_SCRATCH_BYTES = 16 << 20   # PA_NOALLOC_SCRATCH_BYTES in pa.h


def pa_decode_splitk_noalloc(out: torch.Tensor, q: torch.Tensor, kv_cache: torch.Tensor,
                             block_tables: torch.Tensor, seq_lens: torch.Tensor, scale: float,
                             block_size: int, max_seq_len: int, partition_size: int = 512,
                             stream=None) -> torch.Tensor:
    """pa_decode_splitk for callers that cannot allocate device memory: the
    partial states go to a fixed scratch array inside the library
    (NOALLOC_SCRATCH_BYTES per device), so nothing is allocated per call.
    Calls that overlap on the GPU share that array and must be ordered."""
    B, H, hkv, d, nb, mb = _decode_common(out, q, kv_cache, block_tables, seq_lens, block_size)
    _check(_lib.pa_decode_splitk_noalloc(_dev(out, "out"), _dev(q, "q"),
                                         _dev(kv_cache, "kv_cache"),
                                         _dev(block_tables, "block_tables"),
                                         _dev(seq_lens, "seq_lens"), B, H, hkv, d, block_size,
                                         nb, mb, float(scale), _DTYPE[q.dtype],
                                         int(max_seq_len), int(partition_size),
                                         _stream(stream)),
           "pa_decode_splitk_noalloc")
    return out


def pa_validate_tables(block_tables: torch.Tensor, seq_lens: torch.Tensor, block_size: int,
                       num_blocks: int) -> int:
    """Host check of the decode preconditions on CPU copies; returns a status."""
    bt = block_tables.detach().to("cpu", torch.int32).contiguous()
    sl = seq_lens.detach().to("cpu", torch.int32).contiguous()
    return _lib.pa_validate_tables(ctypes.c_void_p(bt.data_ptr()), ctypes.c_void_p(sl.data_ptr()),
                                   int(sl.numel()), int(bt.shape[1]), block_size, num_blocks)


def pa_validate_slots(slot_mapping: torch.Tensor, block_size: int, num_blocks: int) -> int:
    sm = slot_mapping.detach().to("cpu", torch.int64).contiguous()
    return _lib.pa_validate_slots(ctypes.c_void_p(sm.data_ptr()), int(sm.numel()), block_size,
                                  num_blocks)


def pa_prefill(out: torch.Tensor, q: torch.Tensor, kv_cache: torch.Tensor,
               block_tables: torch.Tensor, seq_lens: torch.Tensor,
               query_start_loc: torch.Tensor, scale: float, block_size: int,
               max_query_len: int, causal: bool = True, lse: torch.Tensor | None = None,
               stream=None) -> torch.Tensor:
    """Prefill / chunked-prefill attention of the packed query rows q [T, H, D]
    to each request's paged keys; writes and returns ``out``.  ``block_tables``
    may be a column slice of a larger table (rows contiguous, any row stride).
    ``lse`` (float32 [T, H]) receives the natural-log softmax denominators."""
    nb, hkv, d = _pool_dims(kv_cache, block_size)
    if q.dim() != 3 or q.shape[2] != d or not q.is_contiguous():
        raise ValueError("q must be contiguous [num_tokens, H, head_size]")
    if out.shape != q.shape or out.dtype != q.dtype or not out.is_contiguous():
        raise ValueError("out must be contiguous and match q")
    if q.dtype != kv_cache.dtype or q.dtype not in _DTYPE:
        raise ValueError("q, kv_cache and out must share dtype float16 or bfloat16")
    T, H = int(q.shape[0]), int(q.shape[1])
    R = int(seq_lens.numel())
    if block_tables.dtype != torch.int32 or block_tables.dim() != 2 or \
            block_tables.shape[0] != R or block_tables.stride(1) != 1 or \
            block_tables.stride(0) < block_tables.shape[1]:
        raise ValueError("block_tables must be int32 [R, max_blocks] with contiguous rows")
    if seq_lens.dtype != torch.int32 or not seq_lens.is_contiguous():
        raise ValueError("seq_lens must be contiguous int32 [R]")
    if query_start_loc.dtype != torch.int32 or query_start_loc.numel() != R + 1 or \
            not query_start_loc.is_contiguous():
        raise ValueError("query_start_loc must be contiguous int32 [R + 1]")
    lse_ptr = ctypes.c_void_p(0)
    if lse is not None:
        if lse.dtype != torch.float32 or tuple(lse.shape) != (T, H) or not lse.is_contiguous():
            raise ValueError("lse must be contiguous float32 [num_tokens, H]")
        lse_ptr = _dev(lse, "lse")
    if R == 0 or T == 0:
        return out
    _check(_lib.pa_prefill(_dev(out, "out"), lse_ptr, _dev(q, "q"), _dev(kv_cache, "kv_cache"),
                           _dev(block_tables, "block_tables"), int(block_tables.stride(0)),
                           _dev(seq_lens, "seq_lens"), _dev(query_start_loc, "query_start_loc"),
                           R, T, int(max_query_len), H, hkv, d, block_size, nb,
                           max(1, int(block_tables.shape[1])), float(scale),
                           1 if causal else 0, _DTYPE[q.dtype], _stream(stream)), "pa_prefill")
    return out


def _fp8_pool(kv_cache: torch.Tensor, block_size: int):
    if kv_cache.dtype != torch.uint8:
        raise ValueError("an FP8 pool is a uint8 tensor of e4m3 codes")
    return _pool_dims(kv_cache, block_size)


def pa_reshape_and_cache_fp8(key: torch.Tensor, value: torch.Tensor, kv_cache: torch.Tensor,
                             slot_mapping: torch.Tensor, block_size: int, k_scale: float,
                             v_scale: float, stream=None) -> None:
    """Quantise new tokens' K/V ([T, Hkv, D] fp16/bf16) to e4m3 with the
    per-tensor scales and scatter them into the uint8 pool."""
    nb, hkv, d = _fp8_pool(kv_cache, block_size)
    T = int(key.shape[0])
    for name, t in (("key", key), ("value", value)):
        if t.dtype not in _DTYPE or t.dtype != key.dtype or t.shape[0] != T:
            raise ValueError(f"{name} must be fp16/bf16 [T, ...] like key")
        if t.dim() != 3 or t.shape[1] != hkv or t.shape[2] != d or t.stride(2) != 1 or \
                t.stride(1) != d:
            raise ValueError(f"{name} must be [T, num_kv_heads, head_size] with contiguous rows")
    if slot_mapping.dtype != torch.int64 or slot_mapping.numel() != T or \
            not slot_mapping.is_contiguous():
        raise ValueError("slot_mapping must be contiguous int64 [T]")
    if T == 0:
        return
    _check(_lib.pa_reshape_and_cache_fp8(_dev(key, "key"), _dev(value, "value"),
                                         _dev(kv_cache, "kv_cache"),
                                         _dev(slot_mapping, "slot_mapping"), T, hkv, d,
                                         block_size, nb, key.stride(0), value.stride(0),
                                         _DTYPE[key.dtype], float(k_scale), float(v_scale),
                                         _stream(stream)), "pa_reshape_and_cache_fp8")


def _fp8_decode_common(out, q, kv_cache, block_tables, seq_lens, block_size):
    nb, hkv, d = _fp8_pool(kv_cache, block_size)
    if q.dim() != 3 or q.shape[2] != d or not q.is_contiguous() or q.dtype not in _DTYPE:
        raise ValueError("q must be contiguous fp16/bf16 [B, H, head_size]")
    if out.shape != q.shape or out.dtype != q.dtype or not out.is_contiguous():
        raise ValueError("out must be contiguous and match q")
    B, H = int(q.shape[0]), int(q.shape[1])
    if block_tables.dtype != torch.int32 or block_tables.dim() != 2 or \
            block_tables.shape[0] != B or not block_tables.is_contiguous():
        raise ValueError("block_tables must be contiguous int32 [B, max_blocks_per_seq]")
    if seq_lens.dtype != torch.int32 or seq_lens.numel() != B or not seq_lens.is_contiguous():
        raise ValueError("seq_lens must be contiguous int32 [B]")
    return B, H, hkv, d, nb, int(block_tables.shape[1])


def pa_decode_fp8(out: torch.Tensor, q: torch.Tensor, kv_cache: torch.Tensor,
                  block_tables: torch.Tensor, seq_lens: torch.Tensor, scale: float,
                  block_size: int, k_scale: float, v_scale: float,
                  stream=None) -> torch.Tensor:
    """One-pass paged decode over an FP8 (e4m3) pool."""
    B, H, hkv, d, nb, mb = _fp8_decode_common(out, q, kv_cache, block_tables, seq_lens,
                                              block_size)
    _check(_lib.pa_decode_fp8(_dev(out, "out"), _dev(q, "q"), _dev(kv_cache, "kv_cache"),
                              _dev(block_tables, "block_tables"), _dev(seq_lens, "seq_lens"),
                              B, H, hkv, d, block_size, nb, mb, float(scale), float(k_scale),
                              float(v_scale), _DTYPE[q.dtype], _stream(stream)), "pa_decode_fp8")
    return out


def pa_decode_splitk_fp8_workspace_size(num_seqs: int, num_heads: int, head_size: int,
                                        max_seq_len: int, partition_size: int = 512) -> int:
    return int(_lib.pa_decode_splitk_fp8_workspace_size(num_seqs, num_heads, head_size,
                                                        max_seq_len, partition_size))


def pa_decode_splitk_fp8(out: torch.Tensor, q: torch.Tensor, kv_cache: torch.Tensor,
                         block_tables: torch.Tensor, seq_lens: torch.Tensor, scale: float,
                         block_size: int, k_scale: float, v_scale: float, max_seq_len: int,
                         workspace: torch.Tensor, partition_size: int = 512,
                         stream=None) -> torch.Tensor:
    """Split-K paged decode over an FP8 (e4m3) pool on the tensor cores;
    ``workspace`` holds pa_decode_splitk_fp8_workspace_size bytes."""
    B, H, hkv, d, nb, mb = _fp8_decode_common(out, q, kv_cache, block_tables, seq_lens,
                                              block_size)
    ws_bytes = workspace.numel() * workspace.element_size()
    _check(_lib.pa_decode_splitk_fp8(_dev(out, "out"), _dev(q, "q"), _dev(kv_cache, "kv_cache"),
                                     _dev(block_tables, "block_tables"),
                                     _dev(seq_lens, "seq_lens"), B, H, hkv, d, block_size, nb, mb,
                                     float(scale), float(k_scale), float(v_scale),
                                     _DTYPE[q.dtype], int(max_seq_len), int(partition_size),
                                     _dev(workspace, "workspace"), ws_bytes, _stream(stream)),
           "pa_decode_splitk_fp8")
    return out


def pa_copy_blocks(kv_cache: torch.Tensor, block_mapping: torch.Tensor, block_size: int,
                   stream=None) -> None:
    """Copy the K and V rows of block src into block dst for every (src, dst)
    row of ``block_mapping`` (CUDA int64 [n, 2]), the device half of
    copy-on-write."""
    nb, hkv, d = _pool_dims(kv_cache, block_size)
    if kv_cache.dtype not in _DTYPE:
        raise ValueError("dtype must be float16 or bfloat16")
    if block_mapping.dtype != torch.int64 or block_mapping.dim() != 2 or \
            block_mapping.shape[1] != 2 or not block_mapping.is_contiguous():
        raise ValueError("block_mapping must be contiguous int64 [n, 2]")
    n = int(block_mapping.shape[0])
    if n == 0:
        return
    _check(_lib.pa_copy_blocks(_dev(kv_cache, "kv_cache"), _dev(block_mapping, "block_mapping"),
                               n, nb, block_size, hkv, d, _DTYPE[kv_cache.dtype],
                               _stream(stream)), "pa_copy_blocks")


def pa_stage_copy(dst: torch.Tensor, src: torch.Tensor, stream=None) -> None:
    """Copy ``src`` into ``dst`` (same byte count, both contiguous) on the
    GPU's SMs, stream-ordered.  Each side is a CUDA tensor or a pinned host
    tensor, which the SMs read or write directly through its device mapping."""
    for t, name in ((dst, "dst"), (src, "src")):
        if not t.is_contiguous():
            raise ValueError(f"{name} must be contiguous")
        if not t.is_cuda and not t.is_pinned():
            raise ValueError(f"{name} must be a CUDA tensor or pinned host memory")
    nbytes = dst.numel() * dst.element_size()
    if src.numel() * src.element_size() != nbytes:
        raise ValueError("dst and src must hold the same number of bytes")
    _check(_lib.pa_stage_copy(dst.data_ptr(), src.data_ptr(),
                              nbytes, _stream(stream)), "pa_stage_copy")


def pa_validate_block_mapping(block_mapping: torch.Tensor, num_blocks: int) -> int:
    m = block_mapping.detach().to("cpu", torch.int64).contiguous()
    return _lib.pa_validate_block_mapping(ctypes.c_void_p(m.data_ptr()), int(m.shape[0]),
                                          num_blocks)


def pa_selftest_wait_timeout(stream=None) -> None:
    """Run the bounded-wait self-test kernel (a wait nothing completes); it
    sets DEVERR_TIMEOUT after ~2 s and returns."""
    _check(_lib.pa_selftest_wait_timeout(_stream(stream)), "pa_selftest_wait_timeout")


def pa_profile_kernel_events(before, after) -> None:
    """Record CUDA events ``before``/``after`` (torch.cuda.Event, already
    recorded once so that they exist, or None to stop) around the main
    attention kernel of this thread's later decode calls."""
    def raw(ev):
        if ev is None:
            return ctypes.c_void_p(0)
        if not ev.cuda_event:
            raise ValueError("record the event once before passing it (it is created lazily)")
        return ctypes.c_void_p(ev.cuda_event)
    _check(_lib.pa_profile_kernel_events(raw(before), raw(after)), "pa_profile_kernel_events")


def pa_device_errors(clear: bool = True) -> int:
    """Sticky device error bits (DEVERR_*) of the current device; synchronises."""
    flags = ctypes.c_uint(0)
    _check(_lib.pa_device_errors(ctypes.byref(flags), 1 if clear else 0), "pa_device_errors")
    return int(flags.value)
