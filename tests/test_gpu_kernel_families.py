"""Both decode kernel families against the oracle.

For head_size 128 the library has a CUDA-core kernel and a tensor-core
(tcgen05) kernel; PA_DECODE_KERNEL=simt|tcgen05 forces one per process.  Each
case runs in a child process with the variable set, so every family stays
checked whichever one the automatic choice prefers."""
import json
import os
import subprocess
import sys

import pytest

pytestmark = pytest.mark.gpu

ROOT = os.path.dirname(os.path.dirname(os.path.abspath(__file__)))

CHILD = r"""
import json, sys
sys.path.insert(0, {root!r})
import torch
import workload as wl
from tests._parity import check_attention, oracle_decode, splitk_workspace
from __graft_entry__ import build_library
build_library()
import paged_kv_cache_136_gb300 as pa
res = {{}}
for name, kw in {cases!r}:
    w = wl.make(name, device="cuda", poison=True, **kw)
    ref = oracle_decode(w)
    out = torch.empty_like(w.q)
    pa.pa_decode(out, w.q, w.kv_cache, w.block_tables, w.seq_lens, w.scale, w.block_size)
    res[name + "/onepass"] = check_attention(out, ref, what=name + " onepass")
    for P in (128, 512):
        msl = int(w.seq_lens.max().item())
        ws = splitk_workspace(pa, w, msl, P)
        out = torch.full_like(w.q, float("nan"))
        pa.pa_decode_splitk(out, w.q, w.kv_cache, w.block_tables, w.seq_lens, w.scale,
                            w.block_size, msl, ws, P)
        res[name + f"/split{{P}}"] = check_attention(out, ref, what=name + f" split {{P}}")
assert pa.pa_device_errors(clear=True) == 0
print("RESULT " + json.dumps(res))
"""

CASES = [
    ("mha7b", dict(num_seqs=12, seed=31)),
    ("gqa8b", dict(num_seqs=40, seed=32)),
    ("gqa8b", dict(lengths=[1, 127, 128, 129, 255, 256, 257, 1000, 2047], seed=33)),
    ("long", dict(lengths=[3000, 4097], seed=34)),
    ("prefix", dict(num_seqs=6, seed=35)),
    ("gqa8b", dict(lengths=[0, 300, 0, 17], seed=36)),
    ("gqa8b", dict(lengths=[200, 600], num_heads=16, num_kv_heads=8, seed=37)),
    ("gqa8b", dict(lengths=[200, 600], num_heads=8, num_kv_heads=8, dtype=__import__("torch").float16,
                   seed=38)),
    ("long", dict(lengths=[700, 1500], num_heads=64, num_kv_heads=8, block_size=16, seed=39)),
]


@pytest.mark.parametrize("family", ["simt", "tcgen05"])
def test_family_matches_oracle(family):
    code = CHILD.format(root=ROOT, cases=CASES)
    env = dict(os.environ, PA_DECODE_KERNEL=family)
    r = subprocess.run([sys.executable, "-c", code], cwd=ROOT, env=env, capture_output=True,
                       text=True, timeout=900)
    assert r.returncode == 0, r.stdout[-3000:] + r.stderr[-3000:]
    line = [l for l in r.stdout.splitlines() if l.startswith("RESULT ")]
    assert line, r.stdout
    stats = json.loads(line[0][7:])
    assert stats
