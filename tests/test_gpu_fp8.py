"""FP8 (e4m3) KV cache: the quantising cache write (bit-exact) and decode
over the FP8 pool vs the CPU oracle, through the C ABI."""
import numpy as np
import pytest
import torch

import workload as wl
from tests._parity import check_attention

pytestmark = pytest.mark.gpu


@pytest.fixture(scope="module")
def pa():
    from __graft_entry__ import build_library
    build_library()
    import paged_kv_cache_136_gb300 as pa
    pa.pa_device_errors(clear=True)
    return pa


def _ws(pa, w, msl, part):
    n = pa.pa_decode_splitk_fp8_workspace_size(w.num_seqs, w.num_heads, w.head_size, msl, part)
    return torch.empty(n, dtype=torch.uint8, device=w.q.device)


def _oracle_decode_fp8(w, items=None, cache=None):
    from oracle.oracle import get
    c = w.kv_cache.cpu().numpy() if cache is None else cache
    return get().decode_fp8(wl.bits(w.q), c, w.block_tables.cpu().numpy(),
                            w.seq_lens.cpu().numpy(), w.num_kv_heads, w.block_size, w.scale,
                            wl.ORACLE_DTYPE[w.dtype], w.meta["k_scale"], w.meta["v_scale"],
                            items=items)


@pytest.mark.parametrize("name", ["mha7b", "gqa8b"])
def test_reshape_fp8_bit_exact(pa, name):
    from oracle.oracle import get
    w = wl.make_fp8(name, device="cuda", poison=True, k_scale=0.37, v_scale=1.9)
    sm = w.slot_mapping.clone()
    sm[1] = -1                                       # padding
    before = w.kv_cache.cpu().numpy()
    # a few new values beyond the saturation point
    key = w.key.clone()
    key[0, 0, :4] = torch.tensor([500.0, -500.0, 1e4, 0.0], dtype=key.dtype)
    pa.pa_reshape_and_cache_fp8(key, w.value, w.kv_cache, sm, w.block_size, 0.37, 1.9)
    torch.cuda.synchronize()
    ref = get().reshape_and_cache_fp8(wl.bits(key), wl.bits(w.value), before, sm.cpu().numpy(),
                                      w.block_size, wl.ORACLE_DTYPE[w.dtype], 0.37, 1.9)
    assert np.array_equal(w.kv_cache.cpu().numpy(), ref)
    assert pa.pa_device_errors(clear=True) == 0


CASES = [
    # name, num_seqs, block_size override, heads override (H, Hkv)
    ("mha7b", 12, 16, None),          # G 1
    ("gqa8b", 24, 16, None),          # G 4
    ("gqa8b", 16, 32, (16, 8)),       # G 2, block 32
    ("long", 2, 32, None),            # G 8, long (made short below)
    ("gqa8b", 10, 16, (12, 3)),       # G 4, 3 kv heads: one kv head per CTA
]


@pytest.mark.parametrize("split", [False, True])
@pytest.mark.parametrize("name,B,bs,heads", CASES)
def test_decode_fp8_matches_oracle(pa, name, B, bs, heads, split):
    kw = {"num_seqs": B, "block_size": bs}
    if heads:
        kw.update(num_heads=heads[0], num_kv_heads=heads[1])
    if name == "long":
        kw["lengths"] = [3000, 777]
    w = wl.make_fp8(name, device="cuda", poison=True, k_scale=0.45, v_scale=0.6, seed=60, **kw)
    out = torch.empty_like(w.q)
    if split:
        msl = int(w.seq_lens.max())
        ws = _ws(pa, w, msl, 256)
        pa.pa_decode_splitk_fp8(out, w.q, w.kv_cache, w.block_tables, w.seq_lens, w.scale,
                                w.block_size, 0.45, 0.6, msl, ws, 256)
    else:
        pa.pa_decode_fp8(out, w.q, w.kv_cache, w.block_tables, w.seq_lens, w.scale,
                         w.block_size, 0.45, 0.6)
    torch.cuda.synchronize()
    assert pa.pa_device_errors(clear=True) == 0
    check_attention(out, _oracle_decode_fp8(w), what=f"fp8 {name} split={split}")


def test_fp8_step_write_then_decode(pa):
    """Quantising cache write of the new tokens, then split-K decode."""
    from oracle.oracle import get
    w = wl.make_fp8("gqa8b", device="cuda", poison=True, num_seqs=32, seed=61)
    before = w.kv_cache.cpu().numpy()
    ks, vs = w.meta["k_scale"], w.meta["v_scale"]
    pa.pa_reshape_and_cache_fp8(w.key, w.value, w.kv_cache, w.slot_mapping, w.block_size, ks, vs)
    msl = int(w.seq_lens.max())
    ws = _ws(pa, w, msl, 512)
    out = torch.empty_like(w.q)
    pa.pa_decode_splitk_fp8(out, w.q, w.kv_cache, w.block_tables, w.seq_lens, w.scale,
                            w.block_size, ks, vs, msl, ws, 512)
    torch.cuda.synchronize()
    cb = get().reshape_and_cache_fp8(wl.bits(w.key), wl.bits(w.value), before,
                                     w.slot_mapping.cpu().numpy(), w.block_size,
                                     wl.ORACLE_DTYPE[w.dtype], ks, vs)
    assert np.array_equal(w.kv_cache.cpu().numpy(), cb)
    check_attention(out, _oracle_decode_fp8(w, cache=cb), what="fp8 step")


def test_fp8_full_size_sampled(pa):
    w = wl.make_fp8("mha7b", device="cuda", poison=True, seed=62)
    msl = int(w.seq_lens.max())
    ws = _ws(pa, w, msl, 512)
    out = torch.empty_like(w.q)
    pa.pa_decode_splitk_fp8(out, w.q, w.kv_cache, w.block_tables, w.seq_lens, w.scale,
                            w.block_size, w.meta["k_scale"], w.meta["v_scale"], msl, ws, 512)
    torch.cuda.synchronize()
    items = np.unique(np.random.default_rng(63).integers(0, w.num_seqs * w.num_heads, 200))
    check_attention(out, _oracle_decode_fp8(w, items=items), items=items, what="fp8 full")


def test_fp8_bad_block_id_and_empty_sequence(pa):
    w = wl.make_fp8("gqa8b", device="cuda", num_seqs=6, seed=64)
    bt = w.block_tables.clone()
    bt[2, 0] = w.num_blocks + 9
    sl = w.seq_lens.clone()
    sl[4] = 0
    out = torch.empty_like(w.q)
    pa.pa_decode_fp8(out, w.q, w.kv_cache, bt, sl, w.scale, w.block_size, 0.5, 0.5)
    torch.cuda.synchronize()
    assert pa.pa_device_errors(clear=True) & pa.DEVERR_BLOCK_ID
    assert torch.count_nonzero(out[4]) == 0
    assert torch.isfinite(out.float()).all()


def test_fp8_split_cuda_core_family(pa):
    """The CUDA-core split-K path (forced) stays checked too."""
    import os
    import subprocess
    import sys
    root = os.path.dirname(os.path.dirname(os.path.abspath(__file__)))
    code = (
        "import torch, workload as wl\n"
        "import paged_kv_cache_136_gb300 as pa\n"
        "from tests._parity import check_attention\n"
        "from tests.test_gpu_fp8 import _oracle_decode_fp8, _ws\n"
        "for name, kw in [('gqa8b', dict(num_seqs=12)), ('mha7b', dict(num_seqs=6))]:\n"
        "    w = wl.make_fp8(name, device='cuda', poison=True, seed=65, **kw)\n"
        "    msl = int(w.seq_lens.max()); ws = _ws(pa, w, msl, 128)\n"
        "    out = torch.empty_like(w.q)\n"
        "    pa.pa_decode_splitk_fp8(out, w.q, w.kv_cache, w.block_tables, w.seq_lens,\n"
        "                            w.scale, w.block_size, 0.5, 0.5, msl, ws, 128)\n"
        "    torch.cuda.synchronize()\n"
        "    check_attention(out, _oracle_decode_fp8(w), what='simt fp8 ' + name)\n"
        "assert pa.pa_device_errors(clear=True) == 0\n"
        "print('ok')\n")
    env = dict(os.environ, PA_DECODE_KERNEL="simt")
    r = subprocess.run([sys.executable, "-c", code], cwd=root, env=env, capture_output=True,
                       text=True, timeout=600)
    assert r.returncode == 0 and "ok" in r.stdout, r.stdout[-2000:] + r.stderr[-3000:]
