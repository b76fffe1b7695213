"""Log-sum-exp output of the decode, merge of attention states and cascade
(shared-prefix) decode vs the CPU oracle, through the C ABI."""
import os
import subprocess
import sys

import numpy as np
import pytest
import torch

import workload as wl
from tests._parity import (check_attention, check_lse, oracle_decode, oracle_decode_lse,
                           splitk_workspace)

pytestmark = pytest.mark.gpu
ROOT = os.path.dirname(os.path.dirname(os.path.abspath(__file__)))


@pytest.fixture(scope="module")
def pa():
    from __graft_entry__ import build_library
    build_library()
    import paged_kv_cache_136_gb300 as pa
    pa.pa_device_errors(clear=True)
    return pa


# ---------------------------------------------------------------------------
# merge_attn_states
# ---------------------------------------------------------------------------

@pytest.mark.parametrize("dtype", [torch.float16, torch.bfloat16])
@pytest.mark.parametrize("D", [64, 128])
def test_merge_attn_states_matches_oracle(pa, dtype, D):
    from oracle.oracle import get
    g = torch.Generator(device="cuda").manual_seed(D)
    T, H = 300, 8
    o_a = torch.randn((T, H, D), generator=g, device="cuda").to(dtype)
    o_b = torch.randn((T, H, D), generator=g, device="cuda").to(dtype)
    lse_a = torch.randn((T, H), generator=g, device="cuda") * 4
    lse_b = torch.randn((T, H), generator=g, device="cuda") * 4
    lse_a[0, :] = -float("inf")                   # empty first part
    lse_b[1, :] = -float("inf")                   # empty second part
    lse_a[2, :] = lse_b[2, :] = -float("inf")     # both empty
    lse_a[3, :] = lse_b[3, :] + 60                # one part dominates
    o_a[0, 1, :] = float("nan")                   # an empty part's rows are not read
    o_b[1, 2, :] = float("nan")
    out = torch.empty_like(o_a)
    out_lse = torch.empty_like(lse_a)
    pa.pa_merge_attn_states(out, o_a, lse_a, o_b, lse_b, out_lse=out_lse)
    torch.cuda.synchronize()
    orc = get()
    wa = orc.widen(wl.bits(o_a), wl.ORACLE_DTYPE[dtype])
    wb = orc.widen(wl.bits(o_b), wl.ORACLE_DTYPE[dtype])
    wa[0], wb[1] = 0.0, 0.0                       # the oracle's empty parts hold zeros
    ref, ref_lse = orc.merge_attn_states(wa, lse_a.double().cpu().numpy(), wb,
                                         lse_b.double().cpu().numpy())
    check_attention(out, ref, what="merge")
    got_lse = out_lse.double().cpu().numpy()
    assert np.all(got_lse[2] == -np.inf) and np.all(ref_lse[2] == -np.inf)
    fin = np.isfinite(ref_lse)
    np.testing.assert_allclose(got_lse[fin], ref_lse[fin], rtol=1e-6, atol=1e-5)
    # the merge may write over one of its inputs
    pa.pa_merge_attn_states(o_a, o_a, lse_a, o_b, lse_b)
    torch.cuda.synchronize()
    assert torch.equal(o_a.view(torch.int16), out.view(torch.int16))


# ---------------------------------------------------------------------------
# decode with log-sum-exp
# ---------------------------------------------------------------------------

@pytest.mark.parametrize("name,part", [("gqa8b", 64), ("mha7b", 512), ("tiny", 64)])
def test_decode_splitk_lse(pa, name, part):
    w = wl.make(name, device="cuda", poison=True, num_seqs=24 if name != "tiny" else None,
                seed=31)
    if name != "tiny":
        sl = w.seq_lens.clone()
        sl[3] = 0                                     # an empty sequence
        w.seq_lens = sl
    msl = int(w.seq_lens.max())
    ws = splitk_workspace(pa, w, msl, part)
    out = torch.empty_like(w.q)
    lse = torch.empty(w.q.shape[:2], dtype=torch.float32, device="cuda")
    pa.pa_decode_splitk_lse(out, lse, w.q, w.kv_cache, w.block_tables, w.seq_lens, w.scale,
                            w.block_size, msl, ws, part)
    torch.cuda.synchronize()
    assert pa.pa_device_errors(clear=True) == 0
    check_attention(out, oracle_decode(w), what=f"{name} out")
    L = w.seq_lens.cpu().numpy()
    keep = np.repeat(L > 0, w.num_heads)
    items = np.nonzero(keep)[0]
    ref = oracle_decode_lse(w, items=items)
    check_lse(lse, ref, items=items, what=f"{name} lse")
    if name != "tiny":
        assert torch.all(lse[3] == -float("inf"))


def test_decode_splitk_lse_simt_family(pa):
    """The CUDA-core family (forced) writes the same log-sum-exps."""
    code = (
        "import torch, numpy as np, workload as wl\n"
        "import paged_kv_cache_136_gb300 as pa\n"
        "from tests._parity import splitk_workspace\n"
        "from tests._parity import check_lse, oracle_decode_lse\n"
        "w = wl.make('gqa8b', device='cuda', poison=True, num_seqs=12, seed=33)\n"
        "msl = int(w.seq_lens.max()); ws = splitk_workspace(pa, w, msl, 128)\n"
        "out = torch.empty_like(w.q)\n"
        "lse = torch.empty(w.q.shape[:2], dtype=torch.float32, device='cuda')\n"
        "pa.pa_decode_splitk_lse(out, lse, w.q, w.kv_cache, w.block_tables, w.seq_lens,\n"
        "                        w.scale, w.block_size, msl, ws, 128)\n"
        "torch.cuda.synchronize()\n"
        "check_lse(lse, oracle_decode_lse(w), what='simt lse')\n"
        "print('ok')\n")
    env = dict(os.environ, PA_DECODE_KERNEL="simt")
    r = subprocess.run([sys.executable, "-c", code], cwd=ROOT, env=env, capture_output=True,
                       text=True, timeout=600)
    assert r.returncode == 0 and "ok" in r.stdout, r.stdout[-2000:] + r.stderr[-3000:]


# ---------------------------------------------------------------------------
# cascade decode
# ---------------------------------------------------------------------------

def _cascade(pa, w, prefix_blocks, part=512, max_seq_len=None):
    msl = int(w.seq_lens.max()) if max_seq_len is None else max_seq_len
    n = pa.pa_cascade_decode_workspace_size(w.num_seqs, w.num_heads, w.head_size,
                                            w.block_tables.shape[1], prefix_blocks, msl,
                                            w.block_size, part)
    ws = torch.empty(n, dtype=torch.uint8, device="cuda")
    out = torch.empty_like(w.q)
    pa.pa_cascade_decode(out, w.q, w.kv_cache, w.block_tables, w.seq_lens, w.scale,
                         w.block_size, prefix_blocks, msl, ws, part)
    torch.cuda.synchronize()
    return out


def test_cascade_equals_plain_decode_small(pa):
    w = wl.make("prefix", device="cuda", poison=True, num_seqs=16, seed=40)
    pb = w.meta["shared_blocks"]
    out = _cascade(pa, w, pb, part=128)
    assert pa.pa_device_errors(clear=True) == 0
    check_attention(out, oracle_decode(w), what="cascade")


def test_cascade_full_size_sampled(pa):
    w = wl.make("prefix", device="cuda", poison=True)
    pb = w.meta["shared_blocks"]
    out = _cascade(pa, w, pb)
    assert pa.pa_device_errors(clear=True) == 0
    rng = np.random.default_rng(41)
    items = np.unique(rng.integers(0, w.num_seqs * w.num_heads, size=300))
    check_attention(out, oracle_decode(w, items=items), items=items, what="cascade full")


def test_cascade_suffix_empty_and_partial_prefix(pa):
    """A sequence that is exactly the prefix (empty suffix); a prefix split
    that is not the whole shared part (fewer prefix blocks than shared)."""
    w = wl.make("prefix", device="cuda", poison=True, num_seqs=8, seed=42)
    pb = w.meta["shared_blocks"]
    sl = w.seq_lens.clone()
    sl[2] = pb * w.block_size
    w.seq_lens = sl
    out = _cascade(pa, w, pb, part=64)
    assert pa.pa_device_errors(clear=True) == 0
    ref = oracle_decode(w)
    check_attention(out, ref, what="empty suffix")
    out2 = _cascade(pa, w, pb - 7, part=64)
    check_attention(out2, ref, what="partial prefix")
    out3 = _cascade(pa, w, 0, part=64)
    check_attention(out3, ref, what="no prefix")


def test_cascade_flags_a_table_without_the_prefix(pa):
    w = wl.make("prefix", device="cuda", num_seqs=4, seed=43)
    pb = w.meta["shared_blocks"]
    bt = w.block_tables.clone()
    bt[1, 5] = bt[1, pb]                 # row 1 leaves the shared prefix
    w.block_tables = bt
    _cascade(pa, w, pb, part=64)
    assert pa.pa_device_errors(clear=True) & pa.DEVERR_PREFIX


def test_cascade_in_a_graph_and_in_stream_order(pa):
    """The prefix pass runs on the library's side stream, forked from and
    joined back into the caller's: a graph captured on the caller's stream
    replays the same result, and work queued after the call on that stream
    sees the finished output."""
    w = wl.make("prefix", device="cuda", poison=True, num_seqs=24, seed=44)
    pb = w.meta["shared_blocks"]
    eager = _cascade(pa, w, pb, part=128)
    msl = int(w.seq_lens.max())
    n = pa.pa_cascade_decode_workspace_size(w.num_seqs, w.num_heads, w.head_size,
                                            w.block_tables.shape[1], pb, msl, w.block_size, 128)
    ws = torch.empty(n, dtype=torch.uint8, device="cuda")
    out = torch.full_like(w.q, float("nan"))
    s = torch.cuda.Stream()
    with torch.cuda.stream(s):
        pa.pa_cascade_decode(out, w.q, w.kv_cache, w.block_tables, w.seq_lens, w.scale,
                             w.block_size, pb, msl, ws, 128)
        after = out.clone()
    s.synchronize()
    assert torch.equal(after.view(torch.int16), eager.view(torch.int16))
    g = torch.cuda.CUDAGraph()
    out.fill_(float("nan"))
    torch.cuda.synchronize()
    with torch.cuda.graph(g, stream=s):
        pa.pa_cascade_decode(out, w.q, w.kv_cache, w.block_tables, w.seq_lens, w.scale,
                             w.block_size, pb, msl, ws, 128)
    for _ in range(2):
        out.fill_(float("nan"))
        g.replay()
        torch.cuda.synchronize()
        assert torch.equal(out.view(torch.int16), eager.view(torch.int16))
    assert pa.pa_device_errors(clear=True) == 0


def test_cascade_first_call_inside_a_capture(pa):
    """A host thread whose first cascade call comes inside a graph capture
    gets no side stream (nothing is created during a capture): every step
    runs on the caller's stream, with the same result."""
    import threading
    w = wl.make("prefix", device="cuda", poison=True, num_seqs=12, seed=45)
    pb = w.meta["shared_blocks"]
    eager = _cascade(pa, w, pb, part=64)
    msl = int(w.seq_lens.max())
    n = pa.pa_cascade_decode_workspace_size(w.num_seqs, w.num_heads, w.head_size,
                                            w.block_tables.shape[1], pb, msl, w.block_size, 64)
    ws = torch.empty(n, dtype=torch.uint8, device="cuda")
    out = torch.full_like(w.q, float("nan"))
    errors = []

    def capture_and_replay():
        try:
            torch.cuda.set_device(out.device)
            s = torch.cuda.Stream()
            g = torch.cuda.CUDAGraph()
            with torch.cuda.graph(g, stream=s):
                pa.pa_cascade_decode(out, w.q, w.kv_cache, w.block_tables, w.seq_lens,
                                     w.scale, w.block_size, pb, msl, ws, 64)
            g.replay()
            torch.cuda.synchronize()
        except Exception as e:  # reported in the main thread
            errors.append(e)

    t = threading.Thread(target=capture_and_replay)
    t.start()
    t.join()
    assert not errors, errors
    assert torch.equal(out.view(torch.int16), eager.view(torch.int16))
    assert pa.pa_device_errors(clear=True) == 0


def test_cascade_from_two_host_threads(pa):
    """Two host threads, each with its own stream and workspace, run the
    cascade at the same time: each thread's calls fork onto that thread's
    own side stream, and both results match the single-thread result."""
    import threading
    w = wl.make("prefix", device="cuda", poison=True, num_seqs=16, seed=46)
    pb = w.meta["shared_blocks"]
    eager = _cascade(pa, w, pb, part=128)
    msl = int(w.seq_lens.max())
    n = pa.pa_cascade_decode_workspace_size(w.num_seqs, w.num_heads, w.head_size,
                                            w.block_tables.shape[1], pb, msl, w.block_size, 128)
    outs = [torch.full_like(w.q, float("nan")) for _ in range(2)]
    wss = [torch.empty(n, dtype=torch.uint8, device="cuda") for _ in range(2)]
    errors = []
    start = threading.Barrier(2)

    def run(i):
        try:
            torch.cuda.set_device(w.q.device)
            s = torch.cuda.Stream()
            start.wait()
            with torch.cuda.stream(s):
                for _ in range(20):
                    pa.pa_cascade_decode(outs[i], w.q, w.kv_cache, w.block_tables, w.seq_lens,
                                         w.scale, w.block_size, pb, msl, wss[i], 128)
            s.synchronize()
        except Exception as e:  # reported in the main thread
            errors.append(e)

    ts = [threading.Thread(target=run, args=(i,)) for i in range(2)]
    for t in ts:
        t.start()
    for t in ts:
        t.join()
    assert not errors, errors
    for o in outs:
        assert torch.equal(o.view(torch.int16), eager.view(torch.int16))
    assert pa.pa_device_errors(clear=True) == 0
