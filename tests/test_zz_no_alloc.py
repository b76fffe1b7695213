"""pa_decode_splitk_noalloc: split-K decode for callers that cannot allocate
device memory (code hosted in a framework that owns all device memory and
exposes no allocator to it, or a latency-critical loop where an allocation,
which may synchronise the device, is not allowed).  The entry point keeps its
partial states in a fixed scratch array inside the library instead of a
caller-provided workspace.

Each call goes through the C ABI and is compared with the existing
pa_decode_splitk (given a torch-allocated workspace), on two calls in a row
with different inputs, so stale scratch contents from the first call cannot
hide in the second.  This file is named to be collected last.
"""
import ctypes

import pytest
import torch

import workload as wl
from tests._parity import check_attention, splitk_workspace

pytestmark = pytest.mark.gpu


@pytest.fixture(scope="module")
def pa():
    from __graft_entry__ import build_library
    build_library()
    import paged_kv_cache_136_gb300 as pa
    pa.pa_device_errors(clear=True)
    return pa


def _raw_noalloc(pa, w, out, max_seq_len, partition_size):
    """Call the C entry point directly with raw device pointers."""
    lib = ctypes.CDLL(pa.lib_path())
    f = lib.pa_decode_splitk_noalloc
    f.restype = ctypes.c_int
    f.argtypes = ([ctypes.c_void_p] * 5 + [ctypes.c_int] * 7 +
                  [ctypes.c_float, ctypes.c_int, ctypes.c_int, ctypes.c_int, ctypes.c_void_p])
    return f(out.data_ptr(), w.q.data_ptr(), w.kv_cache.data_ptr(), w.block_tables.data_ptr(),
             w.seq_lens.data_ptr(), w.num_seqs, w.num_heads, w.num_kv_heads, w.head_size,
             w.block_size, w.num_blocks, int(w.block_tables.shape[1]), w.scale,
             0 if w.dtype == torch.float16 else 1, max_seq_len, partition_size,
             torch.cuda.current_stream().cuda_stream)


def _reference(pa, w, max_seq_len, partition_size):
    out = torch.empty_like(w.q)
    ws = splitk_workspace(pa, w, max_seq_len, partition_size)
    pa.pa_decode_splitk(out, w.q, w.kv_cache, w.block_tables, w.seq_lens, w.scale,
                        w.block_size, max_seq_len, ws, partition_size)
    return out


def test_noalloc_matches_workspace_entry_point_twice(pa):
    cases = [
        (wl.make("mha7b", device="cuda", poison=True, num_seqs=24, seed=21), 512),
        (wl.make("gqa8b", device="cuda", poison=True, num_seqs=48, seed=22), 256),
    ]
    for w, P in cases:
        msl = int(w.seq_lens.max().item())
        need = pa.pa_decode_splitk_workspace_size(w.num_seqs, w.num_heads, w.head_size, msl, P)
        assert need <= pa.NOALLOC_SCRATCH_BYTES
        out = torch.full_like(w.q, float("nan"))
        assert _raw_noalloc(pa, w, out, msl, P) == 0
        ref = _reference(pa, w, msl, P)
        torch.cuda.synchronize()
        check_attention(out, ref.double().cpu().numpy(), what=f"noalloc {w.name}")
    assert pa.pa_device_errors(clear=True) == 0


def test_noalloc_binding_and_size_limit(pa):
    w = wl.make("gqa8b", device="cuda", num_seqs=8, seed=23)
    msl = int(w.seq_lens.max().item())
    out = torch.empty_like(w.q)
    pa.pa_decode_splitk_noalloc(out, w.q, w.kv_cache, w.block_tables, w.seq_lens, w.scale,
                                w.block_size, msl, 128)
    ref = _reference(pa, w, msl, 128)
    torch.cuda.synchronize()
    check_attention(out, ref.double().cpu().numpy(), what="noalloc binding")
    # A max_seq_len whose partial states exceed the fixed scratch is refused
    # before any launch.
    too_long = 1 << 24
    assert pa.pa_decode_splitk_workspace_size(w.num_seqs, w.num_heads, w.head_size, too_long,
                                              128) > pa.NOALLOC_SCRATCH_BYTES
    assert _raw_noalloc(pa, w, out, too_long, 128) == 3   # PA_ERR_WORKSPACE
