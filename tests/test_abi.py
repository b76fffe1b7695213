"""The C ABI on the host: libpa.so loads, exports every entry point pa.h
declares, and its host-side logic (argument checks, workspace sizing, table
and slot validation) behaves as documented.  No call here reaches CUDA: every
compute call below is rejected by the host checks before any launch."""
import ctypes
import os
import re

import numpy as np
import pytest

ROOT = os.path.dirname(os.path.dirname(os.path.abspath(__file__)))


@pytest.fixture(scope="module")
def pa():
    from __graft_entry__ import build_library
    build_library()
    import paged_kv_cache_136_gb300 as pa
    return pa


def declared_functions():
    text = open(os.path.join(ROOT, "include", "pa.h")).read()
    text = re.sub(r"/\*.*?\*/", "", text, flags=re.S)
    return sorted(set(re.findall(r"\b(pa_[a-z_0-9]+)\s*\(", text)))


def test_header_declares_the_entry_points():
    names = declared_functions()
    for n in ("pa_reshape_and_cache", "pa_decode", "pa_decode_splitk",
              "pa_decode_splitk_workspace_size", "pa_validate_tables", "pa_validate_slots",
              "pa_device_errors", "pa_status_string", "pa_version", "pa_copy_blocks",
              "pa_validate_block_mapping", "pa_selftest_wait_timeout", "pa_prefill",
              "pa_decode_splitk_lse", "pa_merge_attn_states", "pa_cascade_decode",
              "pa_cascade_decode_workspace_size", "pa_reshape_and_cache_fp8", "pa_decode_fp8",
              "pa_decode_splitk_fp8", "pa_decode_splitk_fp8_workspace_size"):
        assert n in names


def test_library_exports_every_declared_symbol(pa):
    lib = ctypes.CDLL(pa.lib_path())
    missing = [n for n in declared_functions() if not hasattr(lib, n)]
    assert not missing, missing


def test_profile_hook_arguments(pa):
    lib = ctypes.CDLL(pa.lib_path())
    f = lib.pa_profile_kernel_events
    f.restype = ctypes.c_int
    f.argtypes = [ctypes.c_void_p, ctypes.c_void_p]
    assert f(ctypes.c_void_p(FAKE), None) == 1      # one event alone: PA_ERR_INVALID_ARG
    assert f(None, ctypes.c_void_p(FAKE)) == 1
    assert f(None, None) == 0                       # off


def test_status_strings(pa):
    assert pa.pa_status_string(0) == "PA_OK"
    assert pa.pa_status_string(3) == "PA_ERR_WORKSPACE"
    assert pa.pa_status_string(99) == "PA_ERR_UNKNOWN"
    assert pa.pa_version() >= 10000


def _expected_ws(B, H, D, L, P):
    """Header 256 B, then the unit list (B*parts) and the partial o (fp32 D)
    and (m, l) per (sequence, head, partition), each region rounded up to 256
    bytes."""
    r = lambda x: -(-x // 256) * 256
    parts = max(1, -(-L // P))
    rows = B * H * parts
    return 256 + r(B * parts * 4) + r(rows * D * 4) + r(rows * 2 * 4)


def test_workspace_size(pa):
    for B, H, D, L, P in [(8, 64, 128, 131072, 512), (8, 64, 128, 513, 512), (3, 4, 64, 0, 64),
                          (64, 32, 128, 2048, 512)]:
        assert pa.pa_decode_splitk_workspace_size(B, H, D, L, P) == _expected_ws(B, H, D, L, P)
    assert pa.pa_decode_splitk_workspace_size(-1, 8, 128, 100, 512) == 0
    assert pa.pa_decode_splitk_workspace_size(8, 8, 128, 100, 0) == 0


def _raw(pa):
    return ctypes.CDLL(pa.lib_path())


FAKE = 1 << 20  # a 16-byte aligned non-null value; never dereferenced here


def _decode(lib, **kw):
    a = dict(out=FAKE, q=FAKE, cache=FAKE, bt=FAKE, sl=FAKE, B=4, H=8, Hkv=2, D=128, bs=16,
             NB=100, MB=10, scale=0.1, dtype=0)
    a.update(kw)
    f = lib.pa_decode
    f.restype = ctypes.c_int
    f.argtypes = [ctypes.c_void_p] * 5 + [ctypes.c_int] * 7 + [ctypes.c_float, ctypes.c_int,
                                                               ctypes.c_void_p]
    return f(a["out"], a["q"], a["cache"], a["bt"], a["sl"], a["B"], a["H"], a["Hkv"], a["D"],
             a["bs"], a["NB"], a["MB"], a["scale"], a["dtype"], None)


@pytest.mark.parametrize("kw,status", [
    (dict(out=0), 1), (dict(q=0), 1), (dict(bt=0), 1), (dict(H=7), 1), (dict(Hkv=0), 1),
    (dict(scale=float("nan")), 1), (dict(q=FAKE + 8), 1), (dict(B=-1), 1), (dict(NB=0), 1),
    (dict(D=96), 2), (dict(bs=8), 2), (dict(H=48, Hkv=3), 2), (dict(dtype=5), 2),
    (dict(NB=1 << 27, bs=32), 2),
])
def test_decode_rejects_bad_arguments_before_any_launch(pa, kw, status):
    assert _decode(_raw(pa), **kw) == status


def test_splitk_checks_workspace_and_partition(pa):
    lib = _raw(pa)
    f = lib.pa_decode_splitk
    f.restype = ctypes.c_int
    f.argtypes = ([ctypes.c_void_p] * 5 + [ctypes.c_int] * 7 +
                  [ctypes.c_float, ctypes.c_int, ctypes.c_int, ctypes.c_int, ctypes.c_void_p,
                   ctypes.c_size_t, ctypes.c_void_p])
    need = pa.pa_decode_splitk_workspace_size(4, 8, 128, 2048, 512)
    args = [FAKE] * 5 + [4, 8, 2, 128, 16, 100, 10, 0.1, 0]
    assert f(*args, 2048, 500, FAKE, need, None) == 1          # partition not a multiple of 64
    assert f(*args, 2048, 512, FAKE, need - 1, None) == 3      # workspace too small
    assert f(*args, 2048, 512, 0, need, None) == 3             # no workspace
    assert f(*args, 2048, 512, FAKE + 16, need, None) == 3     # workspace not 256-aligned
    assert f(*args[:5], 0, *args[6:], 2048, 512, FAKE, need, None) == 0  # no sequences: no-op


def test_reshape_rejects_bad_strides(pa):
    lib = _raw(pa)
    f = lib.pa_reshape_and_cache
    f.restype = ctypes.c_int
    f.argtypes = [ctypes.c_void_p] * 4 + [ctypes.c_int] * 5 + [ctypes.c_int64] * 2 + \
                 [ctypes.c_int, ctypes.c_void_p]
    assert f(FAKE, FAKE, FAKE, FAKE, 4, 2, 64, 16, 10, 127, 128, 0, None) == 1
    assert f(FAKE, FAKE, FAKE, FAKE, 4, 2, 64, 16, 10, 132, 128, 0, None) == 1
    assert f(FAKE, FAKE, FAKE, FAKE, 4, 2, 64, 16, 10, 128, 128, 3, None) == 2
    assert f(FAKE, FAKE, FAKE, FAKE, 0, 2, 64, 16, 10, 128, 128, 0, None) == 0  # no tokens


def test_validate_tables(pa):
    import torch
    bt = torch.tensor([[3, 1, -1], [0, 2, 4]], dtype=torch.int32)
    sl = torch.tensor([20, 48], dtype=torch.int32)
    assert pa.pa_validate_tables(bt, sl, 16, 5) == 0
    assert pa.pa_validate_tables(bt, sl, 16, 4) == 5          # id 4 out of range
    assert pa.pa_validate_tables(bt, torch.tensor([33, 48], dtype=torch.int32), 16, 5) == 5
    assert pa.pa_validate_tables(bt, torch.tensor([20, 49], dtype=torch.int32), 16, 5) == 5
    assert pa.pa_validate_tables(bt, torch.tensor([-1, 48], dtype=torch.int32), 16, 5) == 5


def test_validate_tables_agrees_with_oracle(pa):
    import torch
    from oracle.oracle import get
    orc = get()
    rng = np.random.default_rng(0)
    for _ in range(200):
        B, MB, bs, NB = 3, 4, 16, 10
        bt = rng.integers(-2, NB + 2, (B, MB)).astype(np.int32)
        sl = rng.integers(-2, MB * bs + 3, B).astype(np.int32)
        a = pa.pa_validate_tables(torch.from_numpy(bt), torch.from_numpy(sl), bs, NB)
        b = orc.check_tables(bt, sl, bs, NB)
        assert (a == 0) == (b == 0)


def test_validate_slots(pa):
    import torch
    assert pa.pa_validate_slots(torch.tensor([0, 5, -1, 31]), 16, 2) == 0
    assert pa.pa_validate_slots(torch.tensor([0, 5, 5]), 16, 2) == 5       # duplicate
    assert pa.pa_validate_slots(torch.tensor([32]), 16, 2) == 5            # past the pool
    assert pa.pa_validate_slots(torch.tensor([-1, -1]), 16, 2) == 0        # padding may repeat


def test_import_fails_loudly_without_library(tmp_path):
    """The binding refuses to import when libpa.so is missing (no fallback)."""
    import shutil
    import subprocess
    import sys
    pkg = tmp_path / "paged_kv_cache_136_gb300"
    pkg.mkdir()
    shutil.copy(os.path.join(ROOT, "paged_kv_cache_136_gb300", "__init__.py"), pkg)
    code = "import paged_kv_cache_136_gb300"
    r = subprocess.run([sys.executable, "-c", code], capture_output=True, text=True,
                       cwd=str(tmp_path))
    assert r.returncode != 0 and "ImportError" in r.stderr and "libpa.so" in r.stderr


def test_validate_block_mapping(pa):
    import torch
    ok = torch.tensor([[2, 9], [6, 11]])
    assert pa.pa_validate_block_mapping(ok, 12) == 0
    assert pa.pa_validate_block_mapping(torch.tensor([[2, 9], [6, 9]]), 12) == 5   # dst twice
    assert pa.pa_validate_block_mapping(torch.tensor([[2, 9], [9, 11]]), 12) == 5  # dst is a src
    assert pa.pa_validate_block_mapping(torch.tensor([[2, 12]]), 12) == 5          # out of range
    assert pa.pa_validate_block_mapping(torch.tensor([[3, 4], [3, 5]]), 12) == 0   # fork: src twice


def test_copy_blocks_rejects_bad_arguments(pa):
    lib = _raw(pa)
    f = lib.pa_copy_blocks
    f.restype = ctypes.c_int
    f.argtypes = [ctypes.c_void_p] * 2 + [ctypes.c_int] * 6 + [ctypes.c_void_p]
    assert f(FAKE, FAKE, 3, 10, 16, 2, 64, 7, None) == 2      # dtype
    assert f(0, FAKE, 3, 10, 16, 2, 64, 0, None) == 1         # null pool
    assert f(FAKE, FAKE, 0, 10, 16, 2, 64, 0, None) == 0      # nothing to copy


def test_prefill_rejects_bad_arguments(pa):
    lib = _raw(pa)
    f = lib.pa_prefill
    f.restype = ctypes.c_int
    f.argtypes = ([ctypes.c_void_p] * 5 + [ctypes.c_int64] + [ctypes.c_void_p] * 2 +
                  [ctypes.c_int] * 9 + [ctypes.c_float, ctypes.c_int, ctypes.c_int,
                                        ctypes.c_void_p])
    P = [FAKE, 0, FAKE, FAKE, FAKE, 8, FAKE, FAKE]
    ok = dict(R=2, T=10, mq=8, H=4, Hkv=2, D=128, bs=16, NB=10, MB=8)

    def call(P=P, scale=0.1, causal=1, dtype=0, **kw):
        a = {**ok, **kw}
        return f(*P, a["R"], a["T"], a["mq"], a["H"], a["Hkv"], a["D"], a["bs"], a["NB"],
                 a["MB"], scale, causal, dtype, None)
    assert call(D=96) == 2                                    # head_size
    assert call(bs=8) == 2                                    # block_size
    assert call(dtype=5) == 2
    assert call(Hkv=3) == 1                                   # H % Hkv
    assert call(MB=9) == 1                                    # stride < max blocks
    assert call(scale=float("nan")) == 1
    assert call(T=0) == 0                                     # nothing to do
    assert call(R=0) == 0
    assert call(P=[FAKE + 2] + P[1:]) == 1                    # misaligned out
    assert call(P=[0] + P[1:]) == 1                           # null out


def test_cascade_workspace_size_covers_its_parts(pa):
    B, H, D, MB, pb, bs, P = 128, 32, 128, 157, 125, 16, 512
    n = pa.pa_cascade_decode_workspace_size(B, H, D, MB, pb, 2500, bs, P)
    split = pa.pa_decode_splitk_workspace_size(B, H, D, 2500 - pb * bs, P)
    parts = B * H * D * 4 * 2 + B * H * 4 * 2 + B * 4 + B * (MB - pb) * 4   # float32 parts
    assert n >= split + parts and n % 256 == 0
    assert pa.pa_cascade_decode_workspace_size(B, H, D, MB, MB + 1, 2500, bs, P) == 0


def test_merge_and_cascade_reject_bad_arguments(pa):
    lib = _raw(pa)
    f = lib.pa_merge_attn_states
    f.restype = ctypes.c_int
    f.argtypes = [ctypes.c_void_p] * 6 + [ctypes.c_int] * 4 + [ctypes.c_void_p]
    assert f(FAKE, 0, FAKE, FAKE, FAKE, FAKE, 4, 2, 96, 0, None) == 2     # head_size
    assert f(FAKE, 0, FAKE, FAKE, FAKE, FAKE, 4, 2, 128, 9, None) == 2    # dtype
    assert f(FAKE, 0, FAKE, FAKE, FAKE, FAKE, 0, 2, 128, 0, None) == 0    # nothing to do
    assert f(FAKE + 8, 0, FAKE, FAKE, FAKE, FAKE, 4, 2, 128, 0, None) == 1
    g = lib.pa_decode_splitk_lse
    g.restype = ctypes.c_int
    g.argtypes = ([ctypes.c_void_p] * 6 + [ctypes.c_int] * 7 + [ctypes.c_float] +
                  [ctypes.c_int] * 3 + [ctypes.c_void_p, ctypes.c_size_t, ctypes.c_void_p])
    assert g(FAKE, 0, FAKE, FAKE, FAKE, FAKE, 2, 4, 4, 128, 16, 8, 4, 0.1, 0, 64, 512, FAKE,
             1 << 20, None) == 1                                           # lse missing


def test_fp8_calls_reject_bad_arguments(pa):
    lib = _raw(pa)
    f = lib.pa_reshape_and_cache_fp8
    f.restype = ctypes.c_int
    f.argtypes = ([ctypes.c_void_p] * 4 + [ctypes.c_int] * 5 + [ctypes.c_int64] * 2 +
                  [ctypes.c_int, ctypes.c_float, ctypes.c_float, ctypes.c_void_p])
    assert f(FAKE, FAKE, FAKE, FAKE, 4, 2, 64, 16, 8, 128, 128, 0, 1.0, 1.0, None) == 2   # D 64
    assert f(FAKE, FAKE, FAKE, FAKE, 4, 2, 128, 16, 8, 256, 256, 0, 0.0, 1.0, None) == 1  # scale
    assert f(FAKE, FAKE, FAKE, FAKE, 4, 2, 128, 16, 8, 256, 256, 0, 1.0, -1.0, None) == 1
    assert f(FAKE, FAKE, FAKE, FAKE, 0, 2, 128, 16, 8, 256, 256, 0, 1.0, 1.0, None) == 0
    g = lib.pa_decode_fp8
    g.restype = ctypes.c_int
    g.argtypes = ([ctypes.c_void_p] * 5 + [ctypes.c_int] * 7 + [ctypes.c_float] * 3 +
                  [ctypes.c_int, ctypes.c_void_p])
    assert g(FAKE, FAKE, FAKE, FAKE, FAKE, 2, 4, 2, 64, 16, 8, 4, 0.1, 1.0, 1.0, 0, None) == 2
    assert g(FAKE, FAKE, FAKE, FAKE, FAKE, 2, 4, 2, 128, 16, 8, 4, 0.1, 0.0, 1.0, 0, None) == 1


def test_stage_copy_rejects_bad_arguments(pa):
    """A zero-byte copy is a no-op whatever the pointers; a null pointer with
    bytes to move is rejected before any CUDA call.  The binding refuses
    pageable host tensors (the SMs cannot reach them) and strided views."""
    import torch
    lib = _raw(pa)
    f = lib.pa_stage_copy
    f.restype = ctypes.c_int
    f.argtypes = [ctypes.c_void_p, ctypes.c_void_p, ctypes.c_size_t, ctypes.c_void_p]
    assert f(None, None, 0, None) == 0
    assert f(None, FAKE, 16, None) == 1
    assert f(FAKE, None, 16, None) == 1
    host = torch.zeros(64, dtype=torch.uint8)
    with pytest.raises(ValueError, match="CUDA tensor or pinned"):
        pa.pa_stage_copy(host, host)
    with pytest.raises(ValueError, match="contiguous"):
        pa.pa_stage_copy(torch.zeros(128, dtype=torch.uint8)[::2], host)
