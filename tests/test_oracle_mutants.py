"""Each plausible slip planted in a copy of the oracle fails at least one pin.

The mutants are made on the CPU from a temporary copy of oracle/pa_oracle.c;
the oracle source itself is never changed.  Every pin run happens in a child
process, so a mutant that crashes cannot take the test session down (a crash
also counts as caught).
"""
import os
import subprocess
import sys

import pytest

from oracle.oracle import SOURCE, compile_source

ROOT = os.path.dirname(os.path.dirname(os.path.abspath(__file__)))

# (name, text in pa_oracle.c, replacement)
MUTANTS = [
    ("softmax_sign", "a[t] = exp(a[t] - m);", "a[t] = exp(m - a[t]);"),
    ("scale_dropped", "a[t] = A->scale * acc;", "a[t] = acc;"),
    ("gqa_head_map", "const int kvh = h / G;", "const int kvh = h % A->num_kv_heads;"),
    ("query_row_uses_kv_head", "const size_t qrow = ((size_t)s * A->num_heads + h) * D;",
     "const size_t qrow = ((size_t)s * A->num_heads + kvh) * D;"),
    ("offset_shifted", "*offset = t % block_size;", "*offset = (t + 1) % block_size;"),
    ("block_index", "*physical_block = block_table_row[t / block_size];",
     "*physical_block = block_table_row[t / (block_size * 2)];"),
    ("head_major_layout",
     "return ((((size_t)plane * num_blocks + phys) * block_size + off) * num_kv_heads + kvh) *\n               head_size + d;",
     "return ((((size_t)plane * num_blocks + phys) * num_kv_heads + kvh) * block_size + off) *\n               head_size + d;"),
    ("value_into_key_plane",
     "cache[or_pool_index(1, blk, off, h, d, num_blocks, block_size, num_kv_heads,",
     "cache[or_pool_index(0, blk, off, h, d, num_blocks, block_size, num_kv_heads,"),
    ("normaliser_drops_term", "    for (int t = 0; t < L; t++) {\n        a[t] = exp(a[t] - m);\n        l += a[t];\n    }",
     "    for (int t = 0; t < L; t++) {\n        a[t] = exp(a[t] - m);\n        if (t) l += a[t];\n    }"),
    ("no_normalisation", "o[d] = acc / l;", "o[d] = acc;"),
    ("half_subnormal_exponent", "v = ldexp((double)f, -24);", "v = ldexp((double)f, -25);"),
    ("ties_away_from_zero", "double n = nearbyint(a / quantum);", "double n = round(a / quantum);"),
    ("online_merge_skips_rescale", "l = c_old * l + c_new * lj;", "l = l + c_new * lj;"),
    ("partials_unweighted_denominator", "denom += exp(m[p] - M) * l[p];", "denom += l[p];"),
    ("copy_wrong_plane", "const size_t base = (size_t)plane * num_blocks * block_elems;",
     "const size_t base = 0;"),
    ("max_misses_first_score", "double m = a[0];\n    for (int t = 1; t < L; t++)",
     "double m = a[L - 1] - 50.0;\n    for (int t = 1; t < L; t++)"),
]


@pytest.mark.parametrize("name,old,new", MUTANTS, ids=[m[0] for m in MUTANTS])
def test_planted_mistake_is_caught(tmp_path, name, old, new):
    src = open(SOURCE).read()
    assert src.count(old) == 1, f"mutant {name}: anchor text not found exactly once"
    mutant_c = tmp_path / f"{name}.c"
    mutant_c.write_text(src.replace(old, new))
    so = compile_source(str(mutant_c), str(tmp_path / f"lib{name}.so"))
    env = dict(os.environ, PA_ORACLE_SO=so)
    r = subprocess.run([sys.executable, "-m", "pytest", "-x", "-q", "-p", "no:cacheprovider",
                        os.path.join(ROOT, "tests", "test_oracle_pins.py")],
                       cwd=ROOT, env=env, capture_output=True, text=True, timeout=600)
    assert r.returncode != 0, f"mutant {name} passed every pin:\n{r.stdout[-2000:]}"
