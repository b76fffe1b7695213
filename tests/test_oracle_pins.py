"""Pins of the CPU oracle to facts that do not come from the oracle itself.

Each test checks the oracle against something independent: the pages' worked
example, another implementation of a number format (numpy, torch), a library
attention routine (torch's scaled_dot_product_attention in fp64), brute force,
closed forms, or invariants the pages state.  Together they are chosen so that
a plausible slip anywhere in the oracle (a dropped term, a wrong sign, index or
head mapping, a transposed operand, a wrong rounding) fails at least one.
"""
import json
import math
import os

import numpy as np
import pytest
import torch

from oracle.oracle import BF16, FP16, Oracle, OracleError, get

GOLDEN = os.path.join(os.path.dirname(__file__), "golden")


@pytest.fixture(scope="module")
def orc():
    # PA_ORACLE_SO points the pins at another build of the oracle source (the
    # mutation test uses it to show that planted mistakes are caught).
    so = os.environ.get("PA_ORACLE_SO")
    return Oracle(so) if so else get()


ALL_BITS = np.arange(65536, dtype=np.uint32).astype(np.uint16)


# ---------------------------------------------------------------------------
# Number formats
# ---------------------------------------------------------------------------

def test_half_decode_matches_numpy(orc):
    got = orc.widen(ALL_BITS, FP16)
    ref = ALL_BITS.view(np.float16).astype(np.float64)
    assert np.array_equal(np.isnan(got), np.isnan(ref))
    ok = ~np.isnan(ref)
    assert np.array_equal(got[ok], ref[ok])
    assert np.array_equal(np.signbit(got[ok]), np.signbit(ref[ok]))


def test_bf16_decode_matches_torch(orc):
    got = orc.widen(ALL_BITS, BF16)
    ref = torch.from_numpy(ALL_BITS.view(np.int16).copy()).view(torch.bfloat16).to(torch.float64).numpy()
    assert np.array_equal(np.isnan(got), np.isnan(ref))
    ok = ~np.isnan(ref)
    assert np.array_equal(got[ok], ref[ok])


def _finite_table(orc, dtype):
    vals = orc.widen(ALL_BITS, dtype)
    fin = np.isfinite(vals)
    return ALL_BITS[fin], vals[fin]


def _brute_round(x, bits_tab, vals_tab, maxval, dtype_bits):
    """Nearest finite value, ties to the even significand; beyond the
    overflow threshold the result is infinity."""
    out = []
    for v in x:
        a = abs(v)
        if a >= maxval:
            out.append(None)
            continue
        d = np.abs(vals_tab - v)
        best = d.min()
        cand = bits_tab[d == best]
        cand = [c for c in cand if (int(c) >> 15) == (1 if v < 0 or (v == 0 and math.copysign(1, v) < 0) else 0)] or list(cand)
        if len(cand) > 1:
            cand = [c for c in cand if int(c) & 1 == 0] or cand
        out.append(int(cand[0]))
    return out


@pytest.mark.parametrize("dtype", [FP16, BF16])
def test_encode_matches_brute_force(orc, dtype):
    rng = np.random.default_rng(7)
    bits_tab, vals_tab = _finite_table(orc, dtype)
    # Random values over the whole range, exact ties between neighbours, and
    # subnormals.
    if dtype == FP16:
        mags = np.exp(rng.uniform(np.log(1e-8), np.log(6e4), 400))
    else:
        mags = np.exp(rng.uniform(np.log(1e-39), np.log(3e38), 400))
    x = mags * rng.choice([-1.0, 1.0], mags.size)
    pos = np.sort(vals_tab[vals_tab > 0])
    idx = rng.integers(0, pos.size - 1, 200)
    ties = (pos[idx] + pos[idx + 1]) / 2.0      # exact in double
    x = np.concatenate([x, ties, -ties[:50], [0.0, -0.0]])
    got = orc.round_to(x, dtype)
    # Overflow threshold: halfway between the largest finite value and the
    # next power of two (which is where a wider exponent would put it).
    maxfin = pos[-1]
    step = maxfin - pos[-2]
    thresh = maxfin + step / 2.0
    ref = _brute_round(x, bits_tab, vals_tab, thresh, dtype)
    for xi, g, r in zip(x, got, ref):
        if r is None:
            assert (int(g) & 0x7fff) == (0x7c00 if dtype == FP16 else 0x7f80), xi
        else:
            assert int(g) == r, (xi, hex(int(g)), hex(r))


def test_half_encode_matches_numpy(orc):
    rng = np.random.default_rng(3)
    x = np.concatenate([rng.standard_normal(20000) * 4.0,
                        rng.standard_normal(2000) * 1e-6,      # subnormal range
                        rng.standard_normal(200) * 7e4])       # overflow range
    got = orc.round_to(x, FP16)
    ref = x.astype(np.float16).view(np.uint16)
    assert np.array_equal(got, ref)


def test_bf16_encode_matches_torch_for_float32_inputs(orc):
    rng = np.random.default_rng(4)
    x = (rng.standard_normal(20000) * 3.0).astype(np.float32).astype(np.float64)
    got = orc.round_to(x, BF16)
    ref = torch.from_numpy(x.astype(np.float32)).to(torch.bfloat16).view(torch.int16).numpy().view(np.uint16)
    assert np.array_equal(got, ref)


# ---------------------------------------------------------------------------
# Address translation: the pages' worked example
# ---------------------------------------------------------------------------

def test_38_token_example(orc):
    g = json.load(open(os.path.join(GOLDEN, "block_table_38_tokens.json")))
    bs, n, bt = g["block_size"], g["num_tokens"], g["block_table"]
    counts = {}
    offsets = {}
    order = []
    for t in range(n):
        phys, off = orc.translate(bt, t, bs)
        counts[phys] = counts.get(phys, 0) + 1
        offsets.setdefault(phys, []).append(off)
        if not order or order[-1] != phys:
            order.append(phys)
    assert order == [b["physical"] for b in g["blocks"]]
    for b in g["blocks"]:
        assert counts[b["physical"]] == b["tokens"]
        assert offsets[b["physical"]] == list(range(b["tokens"]))
    assert orc.slot_of_token(bt, g["derived"]["last_token"], bs) == g["derived"]["last_token_slot"]


# ---------------------------------------------------------------------------
# Cache write
# ---------------------------------------------------------------------------

def _rand_bits(rng, shape, dtype):
    x = rng.standard_normal(shape)
    if dtype == FP16:
        return x.astype(np.float16).view(np.uint16)
    return torch.from_numpy(x.astype(np.float32)).to(torch.bfloat16).view(torch.int16).numpy().view(np.uint16)


@pytest.mark.parametrize("stride_pad", [0, 24])
def test_reshape_matches_flat_slot_indexing(orc, stride_pad):
    rng = np.random.default_rng(11)
    T, Hkv, D, bs, NB = 9, 3, 32, 16, 7
    sentinel = np.uint16(0xABCD)
    cache = np.full((2, NB, bs, Hkv, D), sentinel, dtype=np.uint16)
    row = Hkv * D + stride_pad
    key = _rand_bits(rng, (T, row), FP16)
    value = _rand_bits(rng, (T, row), FP16)
    slots = rng.choice(NB * bs, T, replace=False).astype(np.int64)
    slots[[1, 5]] = -1
    got = orc.reshape_and_cache(key, value, cache, slots, bs, key_stride=row, value_stride=row)
    # The page's statement with the pool viewed as [2, num_slots, Hkv*D]:
    # key_cache[slot] = key[token], value_cache[slot] = value[token].
    ref = cache.reshape(2, NB * bs, Hkv * D).copy()
    ok = slots >= 0
    ref[0, slots[ok]] = key[ok, :Hkv * D]
    ref[1, slots[ok]] = value[ok, :Hkv * D]
    assert np.array_equal(got.reshape(2, NB * bs, Hkv * D), ref)
    # Padding tokens wrote nothing: exactly the valid slots changed.
    changed = np.any(got.reshape(2, NB * bs, -1) != sentinel, axis=2)
    assert set(np.nonzero(changed[0])[0]) <= set(slots[ok])


def test_reshape_rejects_out_of_range_slot(orc):
    cache = np.zeros((2, 2, 16, 1, 8), np.uint16)
    k = np.zeros((1, 8), np.uint16)
    with pytest.raises(OracleError):
        orc.reshape_and_cache(k, k, cache, np.array([32], np.int64), 16)


# ---------------------------------------------------------------------------
# Decode attention against a library attention routine
# ---------------------------------------------------------------------------

def _case(rng, lens, H, Hkv, D, bs, dtype, contiguous=True, extra_blocks=3):
    B = len(lens)
    nblk = [-(-L // bs) for L in lens]
    MB = max(max(nblk), 1)
    NB = sum(nblk) + extra_blocks
    cache = _rand_bits(rng, (2, NB, bs, Hkv, D), dtype)
    q = _rand_bits(rng, (B, H, D), dtype)
    bt = np.full((B, MB), -1, np.int32)
    ids = np.arange(NB, dtype=np.int32) if contiguous else rng.permutation(NB).astype(np.int32)
    c = 0
    starts = []
    for s in range(B):
        bt[s, :nblk[s]] = ids[c:c + nblk[s]]
        starts.append(c)
        c += nblk[s]
    return q, cache, bt, np.array(lens, np.int32), NB, starts


def _sdpa_contiguous(orc, q, cache, lens, starts, H, Hkv, D, bs, scale, dtype):
    """torch SDPA in fp64 over each sequence's rows, read as a flat slice of
    the pool (the blocks of a sequence are consecutive here)."""
    B = len(lens)
    qd = torch.from_numpy(orc.widen(q, dtype))
    kd = torch.from_numpy(orc.widen(cache[0], dtype)).reshape(-1, Hkv, D)
    vd = torch.from_numpy(orc.widen(cache[1], dtype)).reshape(-1, Hkv, D)
    out = np.zeros((B, H, D))
    G = H // Hkv
    for s in range(B):
        L = int(lens[s])
        if L == 0:
            continue
        k = kd[starts[s] * bs: starts[s] * bs + L].permute(1, 0, 2)      # [Hkv, L, D]
        v = vd[starts[s] * bs: starts[s] * bs + L].permute(1, 0, 2)
        k = k.repeat_interleave(G, dim=0)                                  # q head h -> kv head h // G
        v = v.repeat_interleave(G, dim=0)
        o = torch.nn.functional.scaled_dot_product_attention(
            qd[s][:, None, :], k, v, scale=scale)
        out[s] = o[:, 0, :].numpy()
    return out


CASES = [
    # lens, H, Hkv, D, bs, dtype
    ([1, 17, 33, 64], 4, 4, 64, 16, FP16),
    ([15, 16, 17, 100], 8, 2, 64, 16, BF16),
    ([31, 32, 33, 511, 513], 8, 1, 128, 32, BF16),
    ([200, 7], 16, 2, 128, 16, FP16),
]


@pytest.mark.parametrize("lens,H,Hkv,D,bs,dtype", CASES)
def test_decode_matches_sdpa(orc, lens, H, Hkv, D, bs, dtype):
    rng = np.random.default_rng(sum(lens) + H)
    q, cache, bt, sl, NB, starts = _case(rng, lens, H, Hkv, D, bs, dtype)
    scale = 1.0 / math.sqrt(D)
    got = orc.decode(q, cache, bt, sl, Hkv, bs, scale, dtype, nthreads=2)
    ref = _sdpa_contiguous(orc, q, cache, sl, starts, H, Hkv, D, bs, scale, dtype)
    np.testing.assert_allclose(got, ref, rtol=1e-11, atol=1e-12)


def test_decode_scale_is_applied(orc):
    rng = np.random.default_rng(21)
    lens = [40, 9]
    q, cache, bt, sl, NB, starts = _case(rng, lens, 4, 2, 64, 16, FP16)
    for scale in (0.05, 1.0, 0.3):
        got = orc.decode(q, cache, bt, sl, 2, 16, scale, FP16)
        ref = _sdpa_contiguous(orc, q, cache, sl, starts, 4, 2, 64, 16, scale, FP16)
        np.testing.assert_allclose(got, ref, rtol=1e-11, atol=1e-12)


# ---------------------------------------------------------------------------
# Invariants the pages state
# ---------------------------------------------------------------------------

def test_permutation_of_physical_blocks_is_invisible(orc):
    """The block table only relabels storage ("KV cache 不需要物理连续，只需要可寻址")."""
    rng = np.random.default_rng(5)
    lens = [50, 3, 129, 64]
    q, cache, bt, sl, NB, _ = _case(rng, lens, 8, 4, 64, 16, BF16, contiguous=False)
    ref = orc.decode(q, cache, bt, sl, 4, 16, 0.125, BF16)
    pi = rng.permutation(NB).astype(np.int32)
    cache2 = np.empty_like(cache)
    cache2[:, pi] = cache                       # block b moves to pi[b]
    bt2 = np.where(bt >= 0, pi[np.maximum(bt, 0)], -1).astype(np.int32)
    got = orc.decode(q, cache2, bt2, sl, 4, 16, 0.125, BF16)
    assert np.array_equal(got, ref)


def test_shared_blocks_equal_copied_blocks(orc):
    """Prefix blocks shared by reference give the same result as private copies."""
    rng = np.random.default_rng(6)
    bs, Hkv, D, H = 16, 2, 64, 4
    prefix_blocks, B = 3, 4
    suffix = [5, 16, 17, 1]
    MB = prefix_blocks + 2
    NB = prefix_blocks * (B + 1) + 2 * B
    cache = _rand_bits(rng, (2, NB, bs, Hkv, D), FP16)
    q = _rand_bits(rng, (B, H, D), FP16)
    shared = np.arange(prefix_blocks, dtype=np.int32)
    bt_ref = np.full((B, MB), -1, np.int32)
    bt_cpy = np.full((B, MB), -1, np.int32)
    cache_cpy = cache.copy()
    nxt = prefix_blocks
    for s in range(B):
        bt_ref[s, :prefix_blocks] = shared
        copies = np.arange(nxt, nxt + prefix_blocks, dtype=np.int32)
        nxt += prefix_blocks
        cache_cpy[:, copies] = cache[:, shared]
        bt_cpy[s, :prefix_blocks] = copies
        k = -(-suffix[s] // bs)
        own = np.arange(nxt, nxt + k, dtype=np.int32)
        nxt += k
        bt_ref[s, prefix_blocks:prefix_blocks + k] = own
        bt_cpy[s, prefix_blocks:prefix_blocks + k] = own
    sl = np.array([prefix_blocks * bs + x for x in suffix], np.int32)
    a = orc.decode(q, cache, bt_ref, sl, Hkv, bs, 0.125, FP16)
    b = orc.decode(q, cache_cpy, bt_cpy, sl, Hkv, bs, 0.125, FP16)
    assert np.array_equal(a, b)


def test_tail_of_last_block_is_ignored(orc):
    """Rows past seq_len in the last block never reach the output."""
    rng = np.random.default_rng(8)
    q, cache, bt, sl, NB, _ = _case(rng, [20, 33], 4, 4, 64, 16, FP16, contiguous=False)
    ref = orc.decode(q, cache, bt, sl, 4, 16, 0.125, FP16)
    poisoned = cache.copy()
    for s, L in enumerate(sl):
        last = bt[s, (L - 1) // 16]
        poisoned[:, last, (L - 1) % 16 + 1:] = 0x7E00        # fp16 NaN
    got = orc.decode(q, poisoned, bt, sl, 4, 16, 0.125, FP16)
    assert np.array_equal(got, ref)


# ---------------------------------------------------------------------------
# Closed forms
# ---------------------------------------------------------------------------

def _gathered_v(orc, cache, bt, L, kvh, bs, dtype):
    rows = [cache[1, bt[t // bs], t % bs, kvh] for t in range(L)]
    return orc.widen(np.stack(rows), dtype)


def test_zero_query_gives_mean_of_values(orc):
    rng = np.random.default_rng(9)
    lens = [1, 16, 45]
    q, cache, bt, sl, NB, _ = _case(rng, lens, 4, 2, 64, 16, BF16, contiguous=False)
    q[:] = 0
    got = orc.decode(q, cache, bt, sl, 2, 16, 0.125, BF16)
    for s, L in enumerate(lens):
        for h in range(4):
            v = _gathered_v(orc, cache, bt[s], L, h // 2, 16, BF16)
            np.testing.assert_allclose(got[s, h], v.mean(axis=0), rtol=1e-12, atol=1e-13)


def test_zero_scale_gives_mean_of_values(orc):
    rng = np.random.default_rng(10)
    q, cache, bt, sl, NB, _ = _case(rng, [30], 2, 1, 64, 16, FP16, contiguous=False)
    got = orc.decode(q, cache, bt, sl, 1, 16, 0.0, FP16)
    v = _gathered_v(orc, cache, bt[0], 30, 0, 16, FP16)
    np.testing.assert_allclose(got[0, 0], v.mean(axis=0), rtol=1e-12, atol=1e-13)
    np.testing.assert_allclose(got[0, 1], v.mean(axis=0), rtol=1e-12, atol=1e-13)


def test_single_token_returns_its_value(orc):
    rng = np.random.default_rng(12)
    q, cache, bt, sl, NB, _ = _case(rng, [1, 1], 4, 2, 64, 16, FP16, contiguous=False)
    got = orc.decode(q, cache, bt, sl, 2, 16, 0.125, FP16)
    for s in range(2):
        for h in range(4):
            v = orc.widen(cache[1, bt[s, 0], 0, h // 2], FP16)
            assert np.array_equal(got[s, h], v)


def test_one_hot_score_selects_one_value(orc):
    rng = np.random.default_rng(13)
    L, D, bs, jstar = 40, 64, 16, 27
    q, cache, bt, sl, NB, _ = _case(rng, [L], 1, 1, D, bs, FP16, contiguous=False)
    q[:] = 0
    q[0, 0, 5] = np.float16(1.0).view(np.uint16)
    for t in range(L):
        cache[0, bt[0, t // bs], t % bs, 0, :] = 0
    cache[0, bt[0, jstar // bs], jstar % bs, 0, 5] = np.float16(64.0).view(np.uint16)
    got = orc.decode(q, cache, bt, sl, 1, bs, 1.0, FP16)
    v = _gathered_v(orc, cache, bt[0], L, 0, bs, FP16)
    # weight of every other token is e^-64 relative to token j*.
    bound = (L - 1) * math.exp(-64) * np.abs(v).max() * 2
    assert np.abs(got[0, 0] - v[jstar]).max() <= bound


def test_empty_sequence_gives_zero_row(orc):
    rng = np.random.default_rng(14)
    q, cache, bt, sl, NB, _ = _case(rng, [5, 9], 2, 2, 64, 16, FP16)
    sl = np.array([0, 9], np.int32)
    got = orc.decode(q, cache, bt, sl, 2, 16, 0.125, FP16)
    assert np.array_equal(got[0], np.zeros((2, 64)))


# ---------------------------------------------------------------------------
# Online softmax: the pages' identity, and the partition merge
# ---------------------------------------------------------------------------

def test_online_softmax_equals_two_pass(orc):
    rng = np.random.default_rng(15)
    n, D = 1000, 32
    a = rng.standard_normal(n) * 6.0
    V = rng.standard_normal((n, D))
    w = np.exp(a - a.max())
    ref = (w[:, None] * V).sum(0) / w.sum()
    for block in (1, 3, 16, 512, n):
        out, m, l = orc.online_softmax(a, V, block)
        np.testing.assert_allclose(out, ref, rtol=1e-12, atol=1e-13)
        assert m == a.max()
        np.testing.assert_allclose(l, w.sum(), rtol=1e-12)


def test_merge_of_partition_states_equals_whole(orc):
    rng = np.random.default_rng(16)
    n, D, P = 1300, 16, 512
    a = rng.standard_normal(n) * 5.0
    V = rng.standard_normal((n, D))
    ms, ls, os_ = [], [], []
    for p0 in range(0, n, P):
        aa = a[p0:p0 + P]
        m = aa.max()
        w = np.exp(aa - m)
        ms.append(m)
        ls.append(w.sum())
        os_.append((w[:, None] * V[p0:p0 + P]).sum(0))
    got = orc.merge_partials(np.array(ms), np.array(ls), np.array(os_))
    w = np.exp(a - a.max())
    ref = (w[:, None] * V).sum(0) / w.sum()
    np.testing.assert_allclose(got, ref, rtol=1e-12, atol=1e-13)


def test_decode_equals_online_merge_over_blocks(orc):
    """Two-pass decode == online merge over the gathered blocks."""
    rng = np.random.default_rng(17)
    L, D, bs = 77, 64, 16
    q, cache, bt, sl, NB, _ = _case(rng, [L], 1, 1, D, bs, BF16, contiguous=False)
    got = orc.decode(q, cache, bt, sl, 1, bs, 0.125, BF16)[0, 0]
    qd = orc.widen(q[0, 0], BF16)
    K = np.stack([orc.widen(cache[0, bt[0, t // bs], t % bs, 0], BF16) for t in range(L)])
    V = _gathered_v(orc, cache, bt[0], L, 0, bs, BF16)
    out, _, _ = orc.online_softmax(0.125 * (K @ qd), V, bs)
    np.testing.assert_allclose(got, out, rtol=1e-12, atol=1e-13)


# ---------------------------------------------------------------------------
# Preconditions
# ---------------------------------------------------------------------------

def test_bad_block_id_is_rejected(orc):
    rng = np.random.default_rng(18)
    q, cache, bt, sl, NB, _ = _case(rng, [20], 2, 2, 64, 16, FP16)
    bt[0, 1] = NB
    with pytest.raises(OracleError):
        orc.decode(q, cache, bt, sl, 2, 16, 0.125, FP16)
    assert orc.check_tables(bt, sl, 16, NB) != 0


def test_seq_len_beyond_table_is_rejected(orc):
    rng = np.random.default_rng(19)
    q, cache, bt, sl, NB, _ = _case(rng, [20], 2, 2, 64, 16, FP16)
    sl[0] = bt.shape[1] * 16 + 1
    with pytest.raises(OracleError):
        orc.decode(q, cache, bt, sl, 2, 16, 0.125, FP16)


def test_output_rounding_matches_numpy_half(orc):
    rng = np.random.default_rng(20)
    q, cache, bt, sl, NB, _ = _case(rng, [33, 64], 4, 4, 64, 16, FP16, contiguous=False)
    out = orc.decode(q, cache, bt, sl, 4, 16, 0.125, FP16)
    assert np.array_equal(orc.round_to(out, FP16), out.astype(np.float16).view(np.uint16))


# ---------------------------------------------------------------------------
# Copy-on-write block copy
# ---------------------------------------------------------------------------

def test_copy_blocks_matches_array_assignment(orc):
    rng = np.random.default_rng(30)
    cache = _rand_bits(rng, (2, 12, 16, 3, 32), BF16)
    mapping = np.array([[2, 9], [6, 11], [0, 4]], np.int64)
    got = orc.copy_blocks(cache, mapping)
    ref = cache.copy()
    for src, dst in mapping:
        ref[:, dst] = ref[:, src]
    assert np.array_equal(got, ref)
    untouched = [b for b in range(12) if b not in (9, 11, 4)]
    assert np.array_equal(got[:, untouched], cache[:, untouched])


def test_copy_on_write_keeps_the_other_candidates_unchanged(orc):
    """The page's parallel-sampling example: prompt blocks 2 and 6 shared by
    three candidates (ref count 3); candidate 2 must write into block 6, so
    block 6 is copied to a fresh block 11, candidate 2's table is repointed
    and the token written there.  Candidates 1 and 3 read what they read
    before; candidate 2 reads the copy plus its token."""
    rng = np.random.default_rng(31)
    bs, hkv, d, NB = 16, 2, 64, 16
    cache = _rand_bits(rng, (2, NB, bs, hkv, d), FP16)
    q = _rand_bits(rng, (3, 4, d), FP16)
    tables = np.array([[2, 6], [2, 6], [2, 6]], np.int32)
    lens = np.array([26, 26, 26], np.int32)               # block 6 holds 10 tokens
    before = orc.decode(q, cache, tables, lens, hkv, bs, 0.125, FP16)
    cow = orc.copy_blocks(cache, np.array([[6, 11]], np.int64))
    tables2 = tables.copy()
    tables2[1, 1] = 11
    new_k = _rand_bits(rng, (1, hkv, d), FP16)
    new_v = _rand_bits(rng, (1, hkv, d), FP16)
    slot = orc.slot_of_token(tables2[1], 26, bs)          # token 26 -> block 11, offset 10
    assert slot == 11 * bs + 10
    cow = orc.reshape_and_cache(new_k, new_v, cow, np.array([slot], np.int64), bs)
    lens2 = np.array([26, 27, 26], np.int32)
    after = orc.decode(q, cow, tables2, lens2, hkv, bs, 0.125, FP16)
    assert np.array_equal(after[[0, 2]], before[[0, 2]])
    # candidate 2 = its private copy of the prompt + the new token
    private = cache.copy()
    private[:, 11] = cache[:, 6]
    private = orc.reshape_and_cache(new_k, new_v, private, np.array([slot], np.int64), bs)
    assert np.array_equal(after[1], orc.decode(q, private, tables2, lens2, hkv, bs, 0.125,
                                               FP16)[1])
    assert not np.array_equal(after[1], before[1])


def test_copy_blocks_rejects_bad_ids(orc):
    cache = np.zeros((2, 4, 16, 1, 8), np.uint16)
    with pytest.raises(OracleError):
        orc.copy_blocks(cache, np.array([[0, 4]], np.int64))


# ---------------------------------------------------------------------------
# Prefill / chunked prefill and the merge of attention states
# ---------------------------------------------------------------------------

def _prefill_case(rng, q_lens, ctx_lens, H, Hkv, D, bs, dtype, extra_blocks=4):
    """Scattered tables: the pool's blocks are dealt from a permutation."""
    q_lens = np.asarray(q_lens, np.int64)
    L = q_lens + np.asarray(ctx_lens, np.int64)
    nblk = -(-L // bs)
    R = len(q_lens)
    NB = int(nblk.sum()) + extra_blocks
    ids = rng.permutation(NB).astype(np.int32)
    bt = np.full((R, int(nblk.max())), -1, np.int32)
    c = 0
    for r in range(R):
        bt[r, :nblk[r]] = ids[c:c + nblk[r]]
        c += int(nblk[r])
    qsl = np.concatenate([[0], np.cumsum(q_lens)]).astype(np.int32)
    cache = _rand_bits(rng, (2, NB, bs, Hkv, D), dtype)
    q = _rand_bits(rng, (int(qsl[-1]), H, D), dtype)
    return q, cache, bt, L.astype(np.int32), qsl


def _sdpa_prefill(orc, q, cache, bt, L, qsl, H, Hkv, D, bs, scale, dtype, causal=True):
    """torch SDPA in fp64 with an explicit mask, keys gathered by numpy fancy
    indexing of the 5-D pool; also the log-sum-exp of the masked scores."""
    qd = torch.from_numpy(orc.widen(q, dtype))
    kd = torch.from_numpy(orc.widen(cache[0], dtype))
    vd = torch.from_numpy(orc.widen(cache[1], dtype))
    T = q.shape[0]
    out = np.zeros((T, H, D))
    lse = np.zeros((T, H))
    G = H // Hkv
    for r in range(len(L)):
        n, ql = int(L[r]), int(qsl[r + 1] - qsl[r])
        if ql == 0:
            continue
        t = np.arange(n)
        k = kd[bt[r, t // bs], t % bs].permute(1, 0, 2).repeat_interleave(G, dim=0)
        v = vd[bt[r, t // bs], t % bs].permute(1, 0, 2).repeat_interleave(G, dim=0)
        qq = qd[qsl[r]:qsl[r + 1]].permute(1, 0, 2)                       # [H, ql, D]
        pos = (n - ql) + np.arange(ql)
        allowed = torch.from_numpy(t[None, :] <= pos[:, None]) if causal else \
            torch.ones((ql, n), dtype=torch.bool)
        o = torch.nn.functional.scaled_dot_product_attention(qq, k, v, attn_mask=allowed,
                                                             scale=scale)
        out[qsl[r]:qsl[r + 1]] = o.permute(1, 0, 2).numpy()
        s = scale * (qq @ k.transpose(1, 2))
        s = s.masked_fill(~allowed, float("-inf"))
        lse[qsl[r]:qsl[r + 1]] = torch.logsumexp(s, dim=-1).T.numpy()
    return out, lse


PREFILL_CASES = [
    # q_lens, ctx_lens, H, Hkv, D, bs, dtype
    ([1, 20, 37], [0, 5, 0], 4, 2, 64, 16, FP16),
    ([16, 3, 40], [16, 30, 1], 4, 4, 64, 16, BF16),
    ([70, 1], [33, 64], 8, 1, 128, 32, BF16),
]


@pytest.mark.parametrize("causal", [True, False])
@pytest.mark.parametrize("q_lens,ctx,H,Hkv,D,bs,dtype", PREFILL_CASES)
def test_prefill_matches_masked_sdpa(orc, q_lens, ctx, H, Hkv, D, bs, dtype, causal):
    rng = np.random.default_rng(sum(q_lens) * 7 + sum(ctx) + H)
    q, cache, bt, L, qsl = _prefill_case(rng, q_lens, ctx, H, Hkv, D, bs, dtype)
    scale = 1.0 / math.sqrt(D)
    got, lse = orc.prefill(q, cache, bt, L, qsl, Hkv, bs, scale, dtype, causal=causal,
                           nthreads=2)
    ref, ref_lse = _sdpa_prefill(orc, q, cache, bt, L, qsl, H, Hkv, D, bs, scale, dtype,
                                 causal)
    np.testing.assert_allclose(got, ref, rtol=1e-11, atol=1e-12)
    np.testing.assert_allclose(lse, ref_lse, rtol=1e-12, atol=1e-12)


def test_prefill_first_row_of_a_fresh_prompt_is_its_value(orc):
    """A fresh prompt's first token sees only itself: its output is v_0."""
    rng = np.random.default_rng(61)
    q, cache, bt, L, qsl = _prefill_case(rng, [5, 9], [0, 0], 4, 2, 64, 16, BF16)
    out, lse = orc.prefill(q, cache, bt, L, qsl, 2, 16, 0.125, BF16)
    v = orc.widen(cache[1], BF16)
    for r in range(2):
        for h in range(4):
            assert np.array_equal(out[qsl[r], h], v[bt[r, 0], 0, h // 2])
            s = 0.125 * float(orc.widen(q[qsl[r], h], BF16) @ orc.widen(cache[0][bt[r, 0], 0, h // 2], BF16))
            assert lse[qsl[r], h] == pytest.approx(s, abs=1e-12)


def test_prefill_zero_query_gives_running_means(orc):
    """q = 0 makes every allowed score equal: row i of a request averages the
    values of positions 0..ctx+i (causal) and lse = log(ctx + i + 1)."""
    rng = np.random.default_rng(62)
    q, cache, bt, L, qsl = _prefill_case(rng, [12], [7], 2, 2, 64, 16, FP16)
    q[:] = 0
    out, lse = orc.prefill(q, cache, bt, L, qsl, 2, 16, 0.3, FP16)
    v = orc.widen(cache[1], FP16)
    rows = np.stack([v[bt[0, t // 16], t % 16] for t in range(19)])      # [19, Hkv, D]
    for i in range(12):
        n = 7 + i + 1
        np.testing.assert_allclose(out[i], rows[:n].mean(axis=0), rtol=1e-13, atol=1e-14)
        np.testing.assert_allclose(lse[i], math.log(n), rtol=0, atol=1e-13)


def test_prefill_with_one_query_row_equals_decode(orc):
    """q_len = 1 is the decode step: the two routines, written apart, agree."""
    rng = np.random.default_rng(63)
    lens = [1, 17, 40, 129]
    q, cache, bt, L, qsl = _prefill_case(rng, [1] * 4, [x - 1 for x in lens], 8, 2, 128, 16, BF16)
    got, _ = orc.prefill(q, cache, bt, L, qsl, 2, 16, 0.09, BF16)
    ref = orc.decode(q, cache, bt, L, 2, 16, 0.09, BF16)
    np.testing.assert_allclose(got, ref, rtol=1e-13, atol=1e-14)


def test_chunked_prefill_equals_one_pass(orc):
    """Prefilling a prompt in two chunks (the first with seq_len = its own
    end) gives the same rows as one pass over the whole prompt."""
    rng = np.random.default_rng(64)
    q, cache, bt, L, qsl = _prefill_case(rng, [45], [0], 4, 2, 64, 16, FP16)
    whole, whole_lse = orc.prefill(q, cache, bt, L, qsl, 2, 16, 0.125, FP16)
    a = 19
    c1, l1 = orc.prefill(q[:a], cache, bt, [a], [0, a], 2, 16, 0.125, FP16)
    c2, l2 = orc.prefill(q[a:], cache, bt, [45], [0, 45 - a], 2, 16, 0.125, FP16)
    np.testing.assert_allclose(np.concatenate([c1, c2]), whole, rtol=1e-14, atol=0)
    np.testing.assert_allclose(np.concatenate([l1, l2]), whole_lse, rtol=1e-14, atol=0)


def test_non_causal_last_row_equals_causal(orc):
    rng = np.random.default_rng(65)
    q, cache, bt, L, qsl = _prefill_case(rng, [10, 6], [3, 20], 4, 2, 64, 16, BF16)
    c, cl = orc.prefill(q, cache, bt, L, qsl, 2, 16, 0.125, BF16, causal=True)
    n, nl = orc.prefill(q, cache, bt, L, qsl, 2, 16, 0.125, BF16, causal=False)
    last = qsl[1:] - 1
    np.testing.assert_array_equal(c[last], n[last])
    np.testing.assert_array_equal(cl[last], nl[last])
    assert not np.allclose(c[0], n[0])


def test_cascade_prefix_then_suffix_merge_equals_whole(orc):
    """The shared-prefix split: a non-causal pass over the first P keys and a
    causal pass over the rest, merged with their log-sum-exps, reproduce one
    causal pass over all keys (output and lse)."""
    rng = np.random.default_rng(66)
    bs, P = 16, 32
    q, cache, bt, L, qsl = _prefill_case(rng, [1, 5, 20], [60, 40, P], 4, 2, 64, bs, BF16)
    whole, whole_lse = orc.prefill(q, cache, bt, L, qsl, 2, bs, 0.125, BF16)
    pb = P // bs
    # Each request's first P keys play the prefix: the prefix pass reads only
    # them (every query row sees all of them); the suffix pass reads the rest,
    # whose positions start at P.
    pre, pre_lse = orc.prefill(q, cache, bt[:, :pb].copy(), np.full(3, P, np.int32),
                               qsl, 2, bs, 0.125, BF16, causal=False)
    suf, suf_lse = orc.prefill(q, cache, bt[:, pb:].copy(), L - P, qsl, 2, bs, 0.125, BF16)
    got, got_lse = orc.merge_attn_states(pre, pre_lse, suf, suf_lse)
    np.testing.assert_allclose(got, whole, rtol=1e-12, atol=1e-13)
    np.testing.assert_allclose(got_lse, whole_lse, rtol=1e-13, atol=1e-13)


def test_merge_attn_states_closed_forms(orc):
    o_a = np.array([[1.0, 2.0], [3.0, -1.0], [0.5, 0.5], [7.0, 7.0]])
    o_b = np.array([[3.0, 0.0], [9.0, 9.0], [-2.0, 4.0], [1.0, 1.0]])
    inf = float("inf")
    lse_a = np.array([0.7, 2.0, -inf, -inf])
    lse_b = np.array([0.7, -inf, 5.0, -inf])
    out, lse = orc.merge_attn_states(o_a, lse_a, o_b, lse_b)
    np.testing.assert_allclose(out[0], [2.0, 1.0], rtol=1e-15)            # equal weights
    assert lse[0] == pytest.approx(0.7 + math.log(2.0), abs=1e-15)
    np.testing.assert_array_equal(out[1], o_a[1])                          # b empty
    assert lse[1] == 2.0
    np.testing.assert_array_equal(out[2], o_b[2])                          # a empty
    assert lse[2] == 5.0
    np.testing.assert_array_equal(out[3], [0.0, 0.0])                      # both empty
    assert lse[3] == -inf
    # weights e^1 : e^0 for lse (1 + c, c)
    out, lse = orc.merge_attn_states(o_a[:1], np.array([4.0]), o_b[:1], np.array([3.0]))
    w = math.e / (math.e + 1.0)
    np.testing.assert_allclose(out[0], w * o_a[0] + (1 - w) * o_b[0], rtol=1e-14)
    assert lse[0] == pytest.approx(3.0 + math.log(math.e + 1.0), abs=1e-14)


def test_prefill_rejects_bad_metadata(orc):
    rng = np.random.default_rng(67)
    q, cache, bt, L, qsl = _prefill_case(rng, [4, 4], [0, 0], 2, 2, 64, 16, FP16)
    with pytest.raises(OracleError):            # seq_len shorter than the query rows
        orc.prefill(q, cache, bt, np.array([3, 4], np.int32), qsl, 2, 16, 0.1, FP16)
    bad = bt.copy()
    bad[1, 0] = cache.shape[1] + 5
    with pytest.raises(OracleError):
        orc.prefill(q, cache, bad, L, qsl, 2, 16, 0.1, FP16)


# ---------------------------------------------------------------------------
# FP8 (e4m3) KV cache
# ---------------------------------------------------------------------------

ALL_FP8 = np.arange(256, dtype=np.uint8)


def _torch_fp8_values(codes):
    return torch.from_numpy(np.ascontiguousarray(codes, dtype=np.uint8)).view(
        torch.float8_e4m3fn).to(torch.float64).numpy()


def test_fp8_decode_matches_torch(orc):
    got = orc.fp8_widen(ALL_FP8)
    ref = _torch_fp8_values(ALL_FP8)
    assert np.array_equal(np.isnan(got), np.isnan(ref))
    ok = ~np.isnan(ref)
    assert np.array_equal(got[ok], ref[ok])
    assert np.nanmax(got) == 448.0 and np.isnan(got[0x7F]) and np.isnan(got[0xFF])


def test_fp8_every_finite_code_round_trips(orc):
    vals = orc.fp8_widen(ALL_FP8)
    for c in ALL_FP8:
        if not np.isnan(vals[c]):
            assert orc.fp8_encode(vals[c]) == c


def test_fp8_encode_is_nearest_even_by_brute_force(orc):
    vals = orc.fp8_widen(ALL_FP8)
    fin = ~np.isnan(vals)
    codes, cv = ALL_FP8[fin], vals[fin]
    rng = np.random.default_rng(81)
    xs = np.concatenate([rng.uniform(-460, 460, 3000), rng.normal(0, 0.01, 2000),
                         (cv[:-1] + np.roll(cv, -1)[:-1]) / 2])       # include midpoints
    for x in xs:
        got = orc.fp8_encode(x)
        if abs(x) >= 448:
            assert got == (0xFE if x < 0 else 0x7E)
            continue
        d = np.abs(cv - x)
        best = np.nonzero(d == d.min())[0]
        cand = [c for c in codes[best]]
        if len(cand) > 1:                     # a tie: the even code (fraction LSB 0)
            cand = [c for c in cand if (c & 1) == 0]
        if x == 0:
            cand = [0x80 if np.signbit(x) else 0x00]
        assert got in cand, (x, got, cand)


def test_fp8_encode_matches_torch_in_range(orc):
    rng = np.random.default_rng(82)
    x = np.concatenate([rng.normal(0, 3, 20000), rng.uniform(-440, 440, 5000)]).astype(np.float32)
    got = orc.fp8_quantize(x, 1.0)
    ref = torch.from_numpy(x).to(torch.float8_e4m3fn).view(torch.uint8).numpy()
    assert np.array_equal(got, ref)


def test_fp8_saturates_and_keeps_nan(orc):
    assert orc.fp8_encode(449.0) == 0x7E and orc.fp8_encode(1e30) == 0x7E
    assert orc.fp8_encode(-464.0) == 0xFE
    assert orc.fp8_encode(float("nan")) & 0x7F == 0x7F
    # below half the smallest subnormal (2^-10) rounds to zero
    assert orc.fp8_encode(2.0 ** -11) == 0x00 and orc.fp8_encode(-(2.0 ** -11)) == 0x80


def test_reshape_fp8_matches_torch_quantisation(orc):
    rng = np.random.default_rng(83)
    NB, bs, Hkv, D, T = 6, 16, 2, 64, 9
    key = _rand_bits(rng, (T, Hkv, D), BF16)
    value = _rand_bits(rng, (T, Hkv, D), BF16)
    cache = rng.integers(0, 256, size=(2, NB, bs, Hkv, D), dtype=np.uint8)
    slots = rng.permutation(NB * bs)[:T].astype(np.int64)
    slots[3] = -1
    ks, vs = 0.037, 0.11
    got = orc.reshape_and_cache_fp8(key, value, cache, slots, bs, BF16, ks, vs)
    ref = cache.copy()
    flat = ref.reshape(2, NB * bs, Hkv, D)
    kf = torch.from_numpy(orc.widen(key, BF16).astype(np.float32))
    vf = torch.from_numpy(orc.widen(value, BF16).astype(np.float32))
    kq = (kf / torch.tensor(ks, dtype=torch.float32)).to(torch.float8_e4m3fn).view(torch.uint8).numpy()
    vq = (vf / torch.tensor(vs, dtype=torch.float32)).to(torch.float8_e4m3fn).view(torch.uint8).numpy()
    for i, sl in enumerate(slots):
        if sl >= 0:
            flat[0, sl] = kq[i]
            flat[1, sl] = vq[i]
    assert np.array_equal(got, ref)


def _fp8_case(rng, lens, H, Hkv, D, bs, q_dtype):
    q, cache16, bt, sl, NB, starts = _case(rng, lens, H, Hkv, D, bs, q_dtype)
    x = rng.normal(0, 2, size=(2, NB, bs, Hkv, D)).astype(np.float32)
    cache8 = torch.from_numpy(x).to(torch.float8_e4m3fn).view(torch.uint8).numpy()
    return q, cache8, bt, sl, NB, starts


@pytest.mark.parametrize("lens,H,Hkv,bs", [([1, 17, 40], 4, 4, 16), ([100, 33], 8, 2, 32)])
def test_decode_fp8_matches_sdpa(orc, lens, H, Hkv, bs):
    rng = np.random.default_rng(84 + H)
    D = 128
    q, cache8, bt, sl, NB, starts = _fp8_case(rng, lens, H, Hkv, D, bs, FP16)
    ks, vs = 0.3, 0.7
    got = orc.decode_fp8(q, cache8, bt, sl, Hkv, bs, 1 / math.sqrt(D), FP16, ks, vs)
    # SDPA on torch's own dequantisation of the same pool
    kd = torch.from_numpy(_torch_fp8_values(cache8[0]).reshape(-1, Hkv, D) * ks)
    vd = torch.from_numpy(_torch_fp8_values(cache8[1]).reshape(-1, Hkv, D) * vs)
    qd = torch.from_numpy(orc.widen(q, FP16))
    G = H // Hkv
    for s in range(len(lens)):
        L = int(sl[s])
        k = kd[starts[s] * bs: starts[s] * bs + L].permute(1, 0, 2).repeat_interleave(G, dim=0)
        v = vd[starts[s] * bs: starts[s] * bs + L].permute(1, 0, 2).repeat_interleave(G, dim=0)
        o = torch.nn.functional.scaled_dot_product_attention(qd[s][:, None, :], k, v,
                                                             scale=1 / math.sqrt(D))
        np.testing.assert_allclose(got[s], o[:, 0, :].numpy(), rtol=1e-11, atol=1e-12)


def test_decode_fp8_equals_decode_on_the_dequantised_pool(orc):
    """With power-of-two scales every dequantised value is exact in fp16:
    the FP8 decode equals the fp16 decode of the dequantised pool."""
    rng = np.random.default_rng(85)
    lens = [5, 70, 129]
    q, cache8, bt, sl, NB, starts = _fp8_case(rng, lens, 4, 2, 128, 16, FP16)
    ks, vs = 0.25, 2.0
    got = orc.decode_fp8(q, cache8, bt, sl, 2, 16, 0.1, FP16, ks, vs)
    deq = np.stack([orc.fp8_widen(cache8[0]) * ks, orc.fp8_widen(cache8[1]) * vs])
    cache16 = deq.astype(np.float16).view(np.uint16)
    assert np.array_equal(cache16.view(np.float16).astype(np.float64), deq)
    ref = orc.decode(q, cache16, bt, sl, 2, 16, 0.1, FP16)
    np.testing.assert_allclose(got, ref, rtol=1e-14, atol=1e-15)
