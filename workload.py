"""Seeded synthetic inputs for paged decode attention.

This module only draws inputs: sequence lengths, a shuffled pool of physical
blocks dealt out to block tables, N(0,1) queries/keys/values, NaN poison for
memory no sequence owns, and the per-token write targets of the cache-write
step.  It computes nothing that the attention path computes.  Both the CUDA
library's tests/benchmark and the CPU oracle receive the same tensors from it;
neither side imports the other.

The write target of a new token is stated the way a serving engine's metadata
builder hands it to the cache-write kernel: the flat slot index
``block_number * block_size + block_offset`` ("PagedAttention 在 vLLM 中的实现
分析", section 3.2 "Slot Mapping").  Each new token lands at its sequence's last
position ``seq_len - 1``, so the decode step that follows reads it.

Workloads (seed = the config index unless given):

- ``tiny``: 4 sequences of lengths {1, 17, 33, 64}, block_size 16, 4 q / 4 kv
  heads, head_size 64, fp16, pool of 32 blocks, tables taken from a random
  permutation of the pool, scale 1/8, 4 new tokens of which token 2 is padding
  (slot -1).
- ``mha7b``: 64 sequences, lengths uniform on [128, 2048], 32/32 heads,
  head_size 128, block_size 16, fp16, pool 1.25x the blocks in use, blocks
  scattered at random, 64 new tokens.
- ``gqa8b``: 256 sequences, lengths round(exp(ln 500 + z)), z ~ N(0,1),
  clipped to [16, 4096], 32 q / 8 kv heads, head_size 128, block_size 16, bf16.
- ``long``: 8 sequences of 131072 tokens, 64 q / 8 kv heads, head_size 128,
  block_size 32, bf16; 1% of the (token, kv head) key rows are scaled by 8.
- ``prefix``: 128 sequences sharing one 2000-token prefix (the same 125
  physical blocks in every table) followed by a private suffix of uniform
  [50, 500] tokens starting at a block boundary, 32 q / 8 kv heads,
  head_size 128, block_size 16, bf16.

Prefill workloads (``make_prefill``; the pages give no prefill shapes, so these
are a stated recipe): the batch's new query tokens are packed row after row
and ``query_start_loc`` holds each request's first row.  Request r has
``ctx_r`` tokens already cached and ``q_r`` new tokens, ``seq_len = ctx_r +
q_r``; the new tokens' keys/values are written at positions ctx_r..seq_len-1
by the cache-write step before the attention reads them.

- ``prefill_tiny``: q_len {1, 20, 37, 130}, ctx {0, 5, 0, 70}, 4 q / 2 kv
  heads, head_size 128, block_size 16, fp16.
- ``prefill_mha7b``: 16 requests, q_len uniform on [256, 2048]; even requests
  are fresh prompts (ctx 0), odd ones continue a chunked prefill with ctx
  uniform on [0, 4096]; 32/32 heads, head_size 128, block_size 16, fp16.
- ``prefill_gqa8b``: the same lengths recipe with 32 q / 8 kv heads, bf16.

FP8 pools (``make_fp8``): the same structure, tables, queries and new tokens
as the named decode workload, with the pool drawn as e4m3 codes of N(0, 2)
values (torch's float8_e4m3fn conversion of the draws) and the per-tensor
scales k_scale = v_scale = 0.5, so the dequantised keys and values are about
N(0, 1).  The poison code is 0x7F (NaN).

Q, K and V are N(0,1) draws rounded to the cache dtype.  With ``poison=True``
every pool row that no sequence owns (unused blocks and the tail of each
sequence's last block) holds NaN, so a read past a sequence's end shows up in
its output.
"""
from __future__ import annotations

import math
from dataclasses import dataclass, field

import numpy as np
import torch

CONFIG_NAMES = ("tiny", "mha7b", "gqa8b", "long", "prefix")


@dataclass
class Workload:
    name: str
    q: torch.Tensor                 # [B, H, D]
    kv_cache: torch.Tensor          # [2, NB, bs, Hkv, D]
    block_tables: torch.Tensor      # [B, MB] int32, unused entries -1
    seq_lens: torch.Tensor          # [B] int32
    key: torch.Tensor               # [T, Hkv, D] new tokens
    value: torch.Tensor             # [T, Hkv, D]
    slot_mapping: torch.Tensor      # [T] int64, -1 = padding
    block_size: int
    scale: float
    num_heads: int
    num_kv_heads: int
    head_size: int
    partition_size: int = 512
    meta: dict = field(default_factory=dict)

    @property
    def num_seqs(self) -> int:
        return int(self.q.shape[0])

    @property
    def num_blocks(self) -> int:
        return int(self.kv_cache.shape[1])

    @property
    def dtype(self) -> torch.dtype:
        return self.q.dtype

    def kv_bytes(self) -> int:
        """Bytes of K and V the decode must read: one row per
        (sequence, token, kv head) for K and for V."""
        el = self.kv_cache.element_size()
        tokens = int(self.seq_lens.to(torch.int64).sum().item())
        return tokens * self.num_kv_heads * self.head_size * el * 2

    def unique_kv_bytes(self) -> int:
        """Bytes of distinct pool rows in use (shared blocks counted once)."""
        el = self.kv_cache.element_size()
        bt = self.block_tables.cpu().numpy()
        sl = self.seq_lens.cpu().numpy()
        rows = set()
        for s in range(bt.shape[0]):
            L = int(sl[s])
            nb = -(-L // self.block_size)
            for j in range(nb):
                n = min(self.block_size, L - j * self.block_size)
                rows.add((int(bt[s, j]), n))
        used = {}
        for b, n in rows:
            used[b] = max(used.get(b, 0), n)
        tokens = sum(used.values())
        return tokens * self.num_kv_heads * self.head_size * el * 2

    def to(self, device) -> "Workload":
        w = Workload(**{k: getattr(self, k) for k in self.__dataclass_fields__})
        for k in ("q", "kv_cache", "block_tables", "seq_lens", "key", "value", "slot_mapping"):
            setattr(w, k, getattr(self, k).to(device))
        return w


@dataclass
class Spec:
    name: str
    num_seqs: int
    num_heads: int
    num_kv_heads: int
    head_size: int
    block_size: int
    dtype: torch.dtype
    pool_factor: float = 1.25


SPECS = {
    "tiny": Spec("tiny", 4, 4, 4, 64, 16, torch.float16),
    "mha7b": Spec("mha7b", 64, 32, 32, 128, 16, torch.float16),
    "gqa8b": Spec("gqa8b", 256, 32, 8, 128, 16, torch.bfloat16),
    "long": Spec("long", 8, 64, 8, 128, 32, torch.bfloat16),
    "prefix": Spec("prefix", 128, 32, 8, 128, 16, torch.bfloat16),
}


def _lengths(name: str, rng: np.random.Generator, spec: Spec) -> np.ndarray:
    if name == "tiny":
        return np.array([1, 17, 33, 64], dtype=np.int64)
    if name == "mha7b":
        return rng.integers(128, 2048, size=spec.num_seqs, endpoint=True)
    if name == "gqa8b":
        z = rng.standard_normal(spec.num_seqs)
        return np.clip(np.rint(np.exp(math.log(500.0) + z)), 16, 4096).astype(np.int64)
    if name == "long":
        return np.full(spec.num_seqs, 131072, dtype=np.int64)
    if name == "prefix":
        return 2000 + rng.integers(50, 500, size=spec.num_seqs, endpoint=True)
    raise KeyError(name)


def _randn(shape, gen: torch.Generator, device, dtype, chunk_rows: int = 1 << 14):
    """N(0,1) rounded to dtype, drawn chunk by chunk along dim 0 to bound
    the fp32 transient."""
    out = torch.empty(shape, dtype=dtype, device=device)
    n0 = shape[0]
    for i in range(0, n0, chunk_rows):
        j = min(n0, i + chunk_rows)
        out[i:j] = torch.randn((j - i,) + tuple(shape[1:]), generator=gen, device=device,
                               dtype=torch.float32).to(dtype)
    return out


def make(name: str, seed: int | None = None, device="cpu", poison: bool = False,
         num_seqs: int | None = None, lengths=None, **overrides) -> Workload:
    """Build one workload.  ``num_seqs``/``lengths``/spec fields may be
    overridden to make smaller cases with the same structure."""
    if seed is None:
        seed = CONFIG_NAMES.index(name) + 1
    spec = SPECS[name]
    spec = Spec(**{**spec.__dict__, **{k: v for k, v in overrides.items()
                                       if k in spec.__dict__}})
    if num_seqs is not None:
        spec.num_seqs = num_seqs
    rng = np.random.default_rng(seed)
    if lengths is not None:
        L = np.asarray(lengths, dtype=np.int64)
        spec.num_seqs = L.size
    else:
        L = _lengths(name, rng, spec)[: spec.num_seqs]
    B, H, Hkv, D, bs = spec.num_seqs, spec.num_heads, spec.num_kv_heads, spec.head_size, spec.block_size
    nblk = -(-L // bs)                      # blocks each sequence owns
    MB = max(1, int(nblk.max()) if B else 1)

    if name == "prefix" and lengths is None:
        shared = 2000 // bs                 # 125 blocks shared by every sequence
        private = nblk - shared
        need = shared + int(private.sum())
    else:
        shared = 0
        need = int(nblk.sum())
    if name == "tiny" and lengths is None:
        NB = 32
    else:
        NB = max(1, need, int(math.ceil(spec.pool_factor * need)))

    perm = rng.permutation(NB).astype(np.int32)
    tables = np.full((B, MB), -1, dtype=np.int32)
    cursor = 0
    prefix_ids = perm[:shared]
    cursor = shared
    for s in range(B):
        tables[s, :shared] = prefix_ids
        k = int(nblk[s]) - shared
        tables[s, shared:shared + k] = perm[cursor:cursor + k]
        cursor += k

    gen = torch.Generator(device=device)
    gen.manual_seed(seed)
    q = _randn((B, H, D), gen, device, spec.dtype)
    cache = torch.empty((2, NB, bs, Hkv, D), dtype=spec.dtype, device=device)
    cache[0] = _randn((NB, bs, Hkv, D), gen, device, spec.dtype, chunk_rows=1 << 12)
    cache[1] = _randn((NB, bs, Hkv, D), gen, device, spec.dtype, chunk_rows=1 << 12)
    if name == "long":
        # 1% of the (token, kv head) key rows get 8x magnitude.
        for i in range(0, NB, 1 << 12):
            j = min(NB, i + (1 << 12))
            sel = torch.rand((j - i, bs, Hkv, 1), generator=gen, device=device) < 0.01
            blk = cache[0, i:j]
            blk.copy_(torch.where(sel, blk.float() * 8.0, blk.float()).to(spec.dtype))

    # New tokens, one per sequence, written at position seq_len - 1.
    T = B
    key = _randn((T, Hkv, D), gen, device, spec.dtype)
    value = _randn((T, Hkv, D), gen, device, spec.dtype)
    slots = np.empty(T, dtype=np.int64)
    for s in range(T):
        pos = int(L[s]) - 1
        slots[s] = int(tables[s, pos // bs]) * bs + pos % bs if pos >= 0 else -1
    if name == "tiny" and T > 2:
        slots[2] = -1                       # one padding token

    if poison:
        owned = np.zeros((NB, bs), dtype=bool)
        for s in range(B):
            for j in range(int(nblk[s])):
                n = min(bs, int(L[s]) - j * bs)
                owned[tables[s, j], :n] = True
        mask = torch.from_numpy(~owned).to(device)
        nan = torch.tensor(float("nan"), dtype=spec.dtype, device=device)
        for plane in range(2):
            cache[plane][mask] = nan

    return Workload(
        name=name, q=q, kv_cache=cache,
        block_tables=torch.from_numpy(tables).to(device),
        seq_lens=torch.from_numpy(L.astype(np.int32)).to(device),
        key=key, value=value, slot_mapping=torch.from_numpy(slots).to(device),
        block_size=bs, scale=1.0 / math.sqrt(D), num_heads=H, num_kv_heads=Hkv,
        head_size=D, meta={"seed": seed, "shared_blocks": shared, "poison": poison},
    )


def bits(t: torch.Tensor) -> np.ndarray:
    """Host uint16 view of an fp16/bf16 tensor's bit patterns."""
    return t.detach().cpu().contiguous().view(torch.int16).numpy().view(np.uint16)


ORACLE_DTYPE = {torch.float16: 0, torch.bfloat16: 1}


# ---------------------------------------------------------------------------
# Prefill / chunked-prefill workloads
# ---------------------------------------------------------------------------

PREFILL_NAMES = ("prefill_tiny", "prefill_mha7b", "prefill_gqa8b")

PREFILL_SPECS = {
    "prefill_tiny": Spec("prefill_tiny", 4, 4, 2, 128, 16, torch.float16),
    "prefill_mha7b": Spec("prefill_mha7b", 16, 32, 32, 128, 16, torch.float16),
    "prefill_gqa8b": Spec("prefill_gqa8b", 16, 32, 8, 128, 16, torch.bfloat16),
}


@dataclass
class PrefillWorkload:
    name: str
    q: torch.Tensor                 # [T, H, D] packed new query tokens
    kv_cache: torch.Tensor          # [2, NB, bs, Hkv, D]
    block_tables: torch.Tensor      # [R, MB] int32, unused entries -1
    seq_lens: torch.Tensor          # [R] int32, cached + new tokens
    query_start_loc: torch.Tensor   # [R + 1] int32
    key: torch.Tensor               # [T, Hkv, D] new tokens' keys
    value: torch.Tensor             # [T, Hkv, D]
    slot_mapping: torch.Tensor      # [T] int64
    block_size: int
    scale: float
    num_heads: int
    num_kv_heads: int
    head_size: int
    meta: dict = field(default_factory=dict)

    @property
    def num_reqs(self) -> int:
        return int(self.seq_lens.shape[0])

    @property
    def num_tokens(self) -> int:
        return int(self.q.shape[0])

    @property
    def num_blocks(self) -> int:
        return int(self.kv_cache.shape[1])

    @property
    def dtype(self) -> torch.dtype:
        return self.q.dtype

    def q_lens(self) -> np.ndarray:
        qsl = self.query_start_loc.cpu().numpy().astype(np.int64)
        return qsl[1:] - qsl[:-1]

    def causal_pairs(self) -> int:
        """(query row, key) pairs a causal pass attends, per query head."""
        L = self.seq_lens.cpu().numpy().astype(np.int64)
        ql = self.q_lens()
        ctx = L - ql
        return int((ql * ctx + ql * (ql + 1) // 2).sum())


def make_prefill(name: str, seed: int | None = None, device="cpu", poison: bool = False,
                 q_lens=None, ctx_lens=None, **overrides) -> PrefillWorkload:
    """Build one prefill workload; ``q_lens``/``ctx_lens``/spec fields may be
    overridden to make smaller cases with the same structure."""
    if seed is None:
        seed = 101 + PREFILL_NAMES.index(name)
    spec = PREFILL_SPECS[name]
    spec = Spec(**{**spec.__dict__, **{k: v for k, v in overrides.items()
                                       if k in spec.__dict__}})
    rng = np.random.default_rng(seed)
    if q_lens is not None:
        ql = np.asarray(q_lens, dtype=np.int64)
        cx = np.zeros_like(ql) if ctx_lens is None else np.asarray(ctx_lens, dtype=np.int64)
    elif name == "prefill_tiny":
        ql = np.array([1, 20, 37, 130], dtype=np.int64)
        cx = np.array([0, 5, 0, 70], dtype=np.int64)
    else:
        R = spec.num_seqs
        ql = rng.integers(256, 2048, size=R, endpoint=True)
        cx = np.where(np.arange(R) % 2 == 1, rng.integers(0, 4096, size=R, endpoint=True), 0)
    R = ql.size
    L = ql + cx
    H, Hkv, D, bs = spec.num_heads, spec.num_kv_heads, spec.head_size, spec.block_size
    nblk = -(-L // bs)
    MB = max(1, int(nblk.max()) if R else 1)
    need = int(nblk.sum())
    NB = max(1, need, int(math.ceil(spec.pool_factor * need)))
    perm = rng.permutation(NB).astype(np.int32)
    tables = np.full((R, MB), -1, dtype=np.int32)
    cursor = 0
    for r in range(R):
        k = int(nblk[r])
        tables[r, :k] = perm[cursor:cursor + k]
        cursor += k
    qsl = np.zeros(R + 1, dtype=np.int64)
    qsl[1:] = np.cumsum(ql)
    T = int(qsl[-1])

    gen = torch.Generator(device=device)
    gen.manual_seed(seed)
    q = _randn((T, H, D), gen, device, spec.dtype)
    cache = torch.empty((2, NB, bs, Hkv, D), dtype=spec.dtype, device=device)
    cache[0] = _randn((NB, bs, Hkv, D), gen, device, spec.dtype, chunk_rows=1 << 12)
    cache[1] = _randn((NB, bs, Hkv, D), gen, device, spec.dtype, chunk_rows=1 << 12)
    key = _randn((T, Hkv, D), gen, device, spec.dtype)
    value = _randn((T, Hkv, D), gen, device, spec.dtype)
    slots = np.empty(T, dtype=np.int64)
    for r in range(R):
        for i in range(int(ql[r])):
            pos = int(cx[r]) + i
            slots[qsl[r] + i] = int(tables[r, pos // bs]) * bs + pos % bs

    if poison:
        owned = np.zeros((NB, bs), dtype=bool)
        for r in range(R):
            for j in range(int(nblk[r])):
                n = min(bs, int(L[r]) - j * bs)
                owned[tables[r, j], :n] = True
        mask = torch.from_numpy(~owned).to(device)
        nan = torch.tensor(float("nan"), dtype=spec.dtype, device=device)
        for plane in range(2):
            cache[plane][mask] = nan

    return PrefillWorkload(
        name=name, q=q, kv_cache=cache,
        block_tables=torch.from_numpy(tables).to(device),
        seq_lens=torch.from_numpy(L.astype(np.int32)).to(device),
        query_start_loc=torch.from_numpy(qsl.astype(np.int32)).to(device),
        key=key, value=value, slot_mapping=torch.from_numpy(slots).to(device),
        block_size=bs, scale=1.0 / math.sqrt(D), num_heads=H, num_kv_heads=Hkv,
        head_size=D, meta={"seed": seed, "poison": poison},
    )


# ---------------------------------------------------------------------------
# FP8 (e4m3) pools
# ---------------------------------------------------------------------------

def make_fp8(name: str, seed: int | None = None, device="cpu", poison: bool = False,
             k_scale: float = 0.5, v_scale: float = 0.5, **kw) -> Workload:
    """The decode workload ``name`` with its pool replaced by e4m3 codes
    (uint8 [2, NB, bs, Hkv, D]); meta holds k_scale and v_scale."""
    w = make(name, seed=seed, device=device, poison=poison, **kw)
    gen = torch.Generator(device=device)
    gen.manual_seed(1000 + int(w.meta["seed"]))
    shape = tuple(w.kv_cache.shape)
    pool = torch.empty(shape, dtype=torch.uint8, device=device)
    for plane in range(2):
        for i in range(0, shape[1], 1 << 12):
            j = min(shape[1], i + (1 << 12))
            x = torch.randn((j - i,) + shape[2:], generator=gen, device=device) * 2.0
            pool[plane, i:j] = x.to(torch.float8_e4m3fn).view(torch.uint8)
    if poison:
        nan16 = torch.isnan(w.kv_cache)
        pool[nan16] = 0x7F
    w.kv_cache = pool
    w.meta = {**w.meta, "k_scale": float(k_scale), "v_scale": float(v_scale), "fp8": True}
    return w
