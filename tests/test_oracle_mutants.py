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

# (name, text in pa_oracle.c, replacement[, which occurrence]).  Text that
# occurs more than once (the decode, prefill and FP8 decode routines state the
# same softmax steps) names the occurrence to change, in file order:
# 0 = decode, 1 = prefill, 2 = FP8 decode.
MUTANTS = [
    ("softmax_sign", "a[t] = exp(a[t] - m);", "a[t] = exp(m - a[t]);", 0),
    ("prefill_softmax_sign", "a[t] = exp(a[t] - m);", "a[t] = exp(m - a[t]);", 1),
    ("fp8_softmax_sign", "a[t] = exp(a[t] - m);", "a[t] = exp(m - a[t]);", 2),
    ("scale_dropped", "a[t] = A->scale * acc;", "a[t] = acc;", 0),
    ("prefill_scale_dropped", "a[t] = A->scale * acc;", "a[t] = acc;", 1),
    ("gqa_head_map", "const int kvh = h / G;", "const int kvh = h % A->num_kv_heads;", 0),
    ("fp8_gqa_head_map", "const int kvh = h / G;", "const int kvh = h % num_kv_heads;", 1),
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
     "cache[or_pool_index(0, blk, off, h, d, num_blocks, block_size, num_kv_heads,", 0),
    ("fp8_value_into_key_plane",
     "cache[or_pool_index(1, blk, off, h, d, num_blocks, block_size, num_kv_heads,",
     "cache[or_pool_index(0, blk, off, h, d, num_blocks, block_size, num_kv_heads,", 1),
    ("normaliser_drops_term", "    for (int t = 0; t < L; t++) {\n        a[t] = exp(a[t] - m);\n        l += a[t];\n    }",
     "    for (int t = 0; t < L; t++) {\n        a[t] = exp(a[t] - m);\n        if (t) l += a[t];\n    }"),
    ("no_normalisation", "o[d] = acc / l;", "o[d] = acc;", 0),
    ("prefill_no_normalisation", "o[d] = acc / l;", "o[d] = acc;", 1),
    ("fp8_no_normalisation", "o[d] = acc / l;", "o[d] = acc;", 2),
    ("half_subnormal_exponent", "v = ldexp((double)f, -24);", "v = ldexp((double)f, -25);"),
    ("ties_away_from_zero", "double n = nearbyint(a / quantum);", "double n = round(a / quantum);", 0),
    ("fp8_ties_away_from_zero", "double n = nearbyint(a / quantum);",
     "double n = round(a / quantum);", 1),
    ("online_merge_skips_rescale", "l = c_old * l + c_new * lj;", "l = l + c_new * lj;"),
    ("partials_unweighted_denominator", "denom += exp(m[p] - M) * l[p];", "denom += l[p];"),
    ("copy_wrong_plane", "const size_t base = (size_t)plane * num_blocks * block_elems;",
     "const size_t base = 0;"),
    ("prefill_causal_off_by_one", "const int n_keys = A->causal ? pos + 1 : L;",
     "const int n_keys = A->causal ? pos + 2 : L;"),
    ("prefill_top_left_causal",
     "const int pos = L - q_len + (int)(tok - A->query_start_loc[r]);",
     "const int pos = (int)(tok - A->query_start_loc[r]);"),
    ("prefill_ignores_query_start_loc",
     "const int pos = L - q_len + (int)(tok - A->query_start_loc[r]);",
     "const int pos = L - q_len + (int)tok;"),
    ("prefill_lse_in_log2", "A->lse[(size_t)tok * A->num_heads + h] = m + log(l);",
     "A->lse[(size_t)tok * A->num_heads + h] = m + log2(l);"),
    ("prefill_query_head_for_kv_head", "const size_t qrow = ((size_t)tok * A->num_heads + h) * D;",
     "const size_t qrow = ((size_t)tok * A->num_heads + kvh) * D;"),
    ("merge_lse_drops_max", "lse_out[i] = M + log(wa + wb);", "lse_out[i] = log(wa + wb);"),
    ("merge_unnormalised", "o[d] = (wa * o_a[(size_t)i * D + d] + wb * o_b[(size_t)i * D + d]) / (wa + wb);",
     "o[d] = wa * o_a[(size_t)i * D + d] + wb * o_b[(size_t)i * D + d];"),
    ("fp8_exponent_bias", "v = ldexp(8.0 + m, e - 10);         /* (1 + m/8) * 2^(e-7) */",
     "v = ldexp(8.0 + m, e - 11);         /* (1 + m/8) * 2^(e-7) */"),
    ("fp8_no_saturation", "        return sign | 0x7E;                 /* saturate to 448 */",
     "        return sign | 0x7F;                 /* saturate to 448 */"),
    ("fp8_subnormal_quantum", "    const double quantum = ldexp(1.0, e - 3);",
     "    const double quantum = ldexp(1.0, e - 2);"),
    ("fp8_value_scale_on_keys",
     "                Vc[(size_t)t * D + d] = v_scale * or_fp8e4m3_to_double(cache[or_pool_index(",
     "                Vc[(size_t)t * D + d] = k_scale * or_fp8e4m3_to_double(cache[or_pool_index("),
    ("fp8_write_divides_by_value_scale",
     "head_size)] = or_double_to_fp8e4m3((double)(kx / k_scale));",
     "head_size)] = or_double_to_fp8e4m3((double)(kx / v_scale));"),
    ("max_misses_first_score", "double m = a[0];\n    for (int t = 1; t < L; t++)",
     "double m = a[L - 1] - 50.0;\n    for (int t = 1; t < L; t++)"),
]


def _plant(src: str, old: str, new: str, which):
    if which is None:
        assert src.count(old) == 1, "anchor text not found exactly once"
        return src.replace(old, new)
    assert src.count(old) > which and src.count(old) >= 2, "anchor occurrence missing"
    at = -1
    for _ in range(which + 1):
        at = src.index(old, at + 1)
    return src[:at] + new + src[at + len(old):]


@pytest.mark.parametrize("mutant", MUTANTS, ids=[m[0] for m in MUTANTS])
def test_planted_mistake_is_caught(tmp_path, mutant):
    name, old, new = mutant[:3]
    which = mutant[3] if len(mutant) > 3 else None
    src = open(SOURCE).read()
    mutant_c = tmp_path / f"{name}.c"
    mutant_c.write_text(_plant(src, old, new, which))
    so = compile_source(str(mutant_c), str(tmp_path / f"lib{name}.so"))
    env = dict(os.environ, PA_ORACLE_SO=so)
    r = subprocess.run([sys.executable, "-m", "pytest", "-x", "-q", "-p", "no:cacheprovider",
                        os.path.join(ROOT, "tests", "test_oracle_pins.py")],
                       cwd=ROOT, env=env, capture_output=True, text=True, timeout=600)
    assert r.returncode != 0, f"mutant {name} passed every pin:\n{r.stdout[-2000:]}"
