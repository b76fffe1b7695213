"""pa_decode_splitk_noalloc: split-K decode for callers that cannot allocate
device memory (code hosted in a framework that owns all device memory and
exposes no allocator to it, or a latency-critical loop where an allocation,
which may synchronise the device, is not allowed).  The entry point keeps its
partial states in a fixed scratch array inside the library instead of a
caller-provided workspace.

Each call goes through the C ABI.  Its output must equal, bit for bit, that
of the existing pa_decode_splitk given a torch-allocated workspace (the same
kernels run on the same inputs, only the scratch address differs), and must
match the CPU oracle on sampled rows.  Two calls are enqueued back to back on
one stream with no synchronisation between them and different inputs, so the
second call reuses the shared array while the first call's kernels may still
be in flight: stream order alone must keep them apart, and stale contents
from the first call must not leak into the second.  This file is named to be
collected last.
"""
import ctypes

import numpy as np
import pytest
import torch

import workload as wl
from tests._parity import check_attention, oracle_decode, splitk_workspace

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


def _with_workspace(pa, w, max_seq_len, partition_size):
    out = torch.empty_like(w.q)
    ws = splitk_workspace(pa, w, max_seq_len, partition_size)
    pa.pa_decode_splitk(out, w.q, w.kv_cache, w.block_tables, w.seq_lens, w.scale,
                        w.block_size, max_seq_len, ws, partition_size)
    return out


def _sample_rows(w, n, seed):
    rows = w.num_seqs * w.num_heads
    return np.sort(np.random.default_rng(seed).choice(rows, size=min(n, rows), replace=False))


def _check(out, ref_ws, w, what, seed):
    assert torch.equal(out.view(torch.int16), ref_ws.view(torch.int16)), \
        f"{what}: differs from pa_decode_splitk with a workspace"
    items = _sample_rows(w, 96, seed)
    check_attention(out, oracle_decode(w, items=items), items=items, what=what)


def test_noalloc_two_calls_queued_back_to_back(pa):
    cases = [
        (wl.make("mha7b", device="cuda", poison=True, num_seqs=24, seed=21), 512),
        (wl.make("gqa8b", device="cuda", poison=True, num_seqs=48, seed=22), 256),
    ]
    outs = []
    torch.cuda.synchronize()
    for w, P in cases:                    # no synchronisation between the two calls
        msl = int(w.seq_lens.max().item())
        need = pa.pa_decode_splitk_workspace_size(w.num_seqs, w.num_heads, w.head_size, msl, P)
        assert need <= pa.NOALLOC_SCRATCH_BYTES
        out = torch.full_like(w.q, float("nan"))
        assert _raw_noalloc(pa, w, out, msl, P) == 0
        outs.append(out)
    torch.cuda.synchronize()
    for (w, P), out in zip(cases, outs):
        msl = int(w.seq_lens.max().item())
        ref_ws = _with_workspace(pa, w, msl, P)
        torch.cuda.synchronize()
        _check(out, ref_ws, w, f"noalloc {w.name} P={P}", seed=P)
    assert pa.pa_device_errors(clear=True) == 0


def test_noalloc_binding_and_size_limit(pa):
    w = wl.make("gqa8b", device="cuda", num_seqs=8, seed=23)
    msl = int(w.seq_lens.max().item())
    out = torch.empty_like(w.q)
    pa.pa_decode_splitk_noalloc(out, w.q, w.kv_cache, w.block_tables, w.seq_lens, w.scale,
                                w.block_size, msl, 128)
    ref_ws = _with_workspace(pa, w, msl, 128)
    torch.cuda.synchronize()
    _check(out, ref_ws, w, "noalloc binding", seed=1)
    # A max_seq_len whose partial states exceed the fixed scratch is refused
    # before any launch.
    too_long = 1 << 24
    assert pa.pa_decode_splitk_workspace_size(w.num_seqs, w.num_heads, w.head_size, too_long,
                                              128) > pa.NOALLOC_SCRATCH_BYTES
    assert _raw_noalloc(pa, w, out, too_long, 128) == 3   # PA_ERR_WORKSPACE
