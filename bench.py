#!/usr/bin/env python
"""Benchmark of the paged decode-attention hot path.

Metric: effective KV-read GB/s (and % of the HBM peak) plus sequences/s.
KV bytes per step = sum_s seq_len_s * num_kv_heads * head_size * 2 (K and V)
* element size: each (sequence, token, kv head) row of K and of V counted once,
no block-tail padding and no re-reads by grouped query heads.

Default workload (one GPU): the long-context split-K decode -- 8 sequences of
131072 tokens, 64 q / 8 kv heads, head_size 128, block_size 32, bf16 pool of
4.3 GB of keys and values (1.25x the blocks in use, scattered at random), 1% of
the key rows scaled by 8.  One step = the cache write of the 8 new tokens
(pa_reshape_and_cache) followed by one decode pass over all sequences
(pa_decode_splitk with 512-token partitions and the log-sum-exp reduce).  The
pool is far larger than the 129 MB L2, so no L2 flush is needed between
steps.  The other decode configurations (MHA 7B-like, GQA 8B-like, prefix
sharing, tiny) are measured the same way and reported per configuration under
``roofline.by_config``; prefill, cascade, FP8 and block-copy workloads follow
under ``workloads``.

Usage:  python bench.py [--gpus N] [--steps K] [--warmup W] [--impl ours|reference]
With N > 1 the script runs under torch.distributed.run, one replica per GPU on
its own seeded batch (weak scaling, no data-path collective); the timed region
is bracketed by barriers and the slowest rank's time is used.
"""
from __future__ import annotations

import argparse
import hashlib
import json
import os
import re
import statistics
import subprocess
import sys
import tempfile
import time

ROOT = os.path.dirname(os.path.abspath(__file__))
if ROOT not in sys.path:
    sys.path.insert(0, ROOT)

METRIC = "paged decode attention: effective KV-read GB/s (% of HBM peak), seqs/s"
UNIT = "GB/s"
WORKLOAD_TEXT = {
    "mha7b": "MHA 7B-like decode layer: 64 seqs, seq_lens U[128,2048], 32 q / 32 kv heads, "
             "head_size 128, block_size 16, fp16 cache, blocks scattered in a 1.25x pool, "
             "+ cache write of 64 new tokens",
    "gqa8b": "GQA 8B-like decode: 256 seqs, lognormal seq_lens (median 500, sigma 1) clipped to "
             "[16,4096], 32 q / 8 kv heads, head_size 128, block_size 16, bf16",
    "long": "long-context split-K: 8 seqs x 131072 tokens, 64 q / 8 kv heads, head_size 128, "
            "block_size 32, bf16, 512-token partitions",
    "prefix": "prefix sharing: 128 seqs sharing a 2000-token prefix + U[50,500] suffix, "
              "32 q / 8 kv heads, head_size 128, block_size 16, bf16",
    "tiny": "tiny: 4 seqs {1,17,33,64}, 4/4 heads, head_size 64, block_size 16, fp16",
}
PREFILL_TEXT = {
    "prefill_mha7b": "chunked prefill, MHA 7B-like: 16 requests, q_len U[256,2048], even ones "
                     "fresh (ctx 0), odd ones ctx U[0,4096]; 32/32 heads, head_size 128, "
                     "block_size 16, fp16, causal",
    "prefill_gqa8b": "chunked prefill, GQA 8B-like: the same lengths, 32 q / 8 kv heads, "
                     "head_size 128, block_size 16, bf16, causal",
}
DECODE_SOURCES = ["paged_kv_cache_136_gb300/csrc/pa_decode.cuh",
                  "paged_kv_cache_136_gb300/csrc/pa_decode_tc.cuh",
                  "paged_kv_cache_136_gb300/csrc/pa_ptx.cuh"]


# ---------------------------------------------------------------------------
# Distributed plumbing (replicas only: barriers and max/sum of scalars)
# ---------------------------------------------------------------------------

def dist_env():
    rank = int(os.environ.get("RANK", "0"))
    world = int(os.environ.get("WORLD_SIZE", "1"))
    local = int(os.environ.get("LOCAL_RANK", "0"))
    return rank, world, local


def init_dist(world: int, backend: str):
    import torch.distributed as dist
    if world > 1 and not dist.is_initialized():
        dist.init_process_group(backend=backend)
    return dist if world > 1 else None


def reduce_scalar(x: float, op: str, dist_mod, device="cpu") -> float:
    """max or sum of one float over all ranks (identity on one rank)."""
    if dist_mod is None:
        return float(x)
    import torch
    t = torch.tensor([float(x)], dtype=torch.float64, device=device)
    dist_mod.all_reduce(t, op=dist_mod.ReduceOp.MAX if op == "max" else dist_mod.ReduceOp.SUM)
    return float(t.item())


def barrier(dist_mod):
    if dist_mod is not None:
        dist_mod.barrier()


# ---------------------------------------------------------------------------
# Clocks during the timed region
# ---------------------------------------------------------------------------

class ClockSampler:
    FIELDS = ("index,clocks.sm,clocks.max.sm,power.draw,clocks_event_reasons.active,"
              "clocks_event_reasons.hw_slowdown,clocks_event_reasons.hw_thermal_slowdown,"
              "clocks_event_reasons.sw_thermal_slowdown,clocks_event_reasons.sw_power_cap")

    def __init__(self, gpu_index: int):
        self.gpu = gpu_index
        self.proc = None
        self.path = None

    def start(self):
        try:
            fd, self.path = tempfile.mkstemp(suffix=".csv")
            os.close(fd)
            self.f = open(self.path, "w")
            self.proc = subprocess.Popen(
                ["nvidia-smi", f"--query-gpu={self.FIELDS}", "--format=csv,noheader,nounits",
                 "-lms", "100", "-i", str(self.gpu)], stdout=self.f, stderr=subprocess.DEVNULL)
            time.sleep(0.4)
        except (OSError, FileNotFoundError):
            self.proc = None

    def stop(self) -> dict | None:
        if self.proc is None:
            return None
        self.proc.terminate()
        try:
            self.proc.wait(timeout=5)
        except subprocess.TimeoutExpired:
            self.proc.kill()
        self.f.close()
        rows = []
        for line in open(self.path):
            parts = [p.strip() for p in line.split(",")]
            if len(parts) < 9:
                continue
            try:
                rows.append((float(parts[1]), float(parts[2]), parts[5:9]))
            except ValueError:
                continue
        os.unlink(self.path)
        if not rows:
            return {"sm_mhz": None, "sm_max_mhz": None, "reasons": [], "samples": 0}
        names = ["hw_slowdown", "hw_thermal_slowdown", "sw_thermal_slowdown", "sw_power_cap"]
        reasons = sorted({names[i] for _, _, r in rows for i, v in enumerate(r)
                          if v.lower() == "active"})
        return {"sm_mhz": statistics.median(r[0] for r in rows),
                "sm_max_mhz": max(r[1] for r in rows), "reasons": reasons,
                "samples": len(rows)}


# ---------------------------------------------------------------------------
# Byte accounting (algorithmic, per step / per launch)
# ---------------------------------------------------------------------------

def kv_bytes(w) -> int:
    return w.kv_bytes()


SPLIT_RUN = 4   # full partitions per run item of the library's split-K work list


def _sm_count() -> int:
    try:
        import torch
        if torch.cuda.is_available():
            return torch.cuda.get_device_properties(0).multi_processor_count
    except Exception:
        pass
    return 152


def split_partials(w, partition: int, sms: int | None = None) -> tuple[int, int, int]:
    """Partial-state traffic of pa_decode_splitk for this workload: (bytes the
    partition kernel writes, bytes the reduce reads, output bytes the reduce
    writes).

    It follows the library's split-K work list: with head_size 128 (the
    tensor-core kernel) a one-partition sequence writes its output directly;
    a longer one writes one partial state (o: head_size floats, m, l) per
    work item -- a run of SPLIT_RUN partitions, a single partition or the
    last one -- and two floats that mark each partition a run covered as
    empty; each sequence keeps enough trailing single partitions that about
    three waves of single items (of the persistent grid of at most one CTA
    per SM) end the list.  The reduce reads every partition's (m, l) and the
    vectors of the non-empty ones.  With head_size 64 (the CUDA-core kernel)
    every partition of every sequence writes a partial state and the reduce
    writes every output row."""
    import math
    sms = sms or _sm_count()
    L = [int(x) for x in w.seq_lens.cpu().tolist()]
    H, D = w.num_heads, w.head_size
    el = w.kv_cache.element_size()
    row_out = H * D * el
    state = (D + 2) * 4
    nparts = [(x + partition - 1) // partition for x in L]
    if D != 128:
        n_all = sum(nparts)
        return H * n_all * state, H * n_all * state, sum(1 for n in nparts if n > 0) * row_out
    G = H // w.num_kv_heads
    hg = 16 // G if w.num_kv_heads % (16 // G) == 0 else 1
    groups = w.num_kv_heads // hg
    max_parts = max(1, math.ceil(max(L + [0]) / partition))
    grid = min(w.num_seqs * groups * max_parts, sms)
    runs = 1 < max_parts <= 4096
    keep = max(0, math.ceil(3 * grid / (w.num_seqs * groups)) - 1) if runs else 0
    written = read = out_rows = 0
    for n in nparts:
        if n <= 1:
            continue
        nfull = n - 1
        in_runs = nfull - keep if runs and nfull > keep else 0
        nruns = in_runs // SPLIT_RUN
        items = nruns + (nfull - nruns * SPLIT_RUN) + 1
        covered = nruns * (SPLIT_RUN - 1)
        written += H * (items * state + covered * 8)
        read += H * (n * 8 + items * D * 4)
        out_rows += 1
    return written, read, out_rows * row_out


def decode_launch_bytes(w, split: bool, partition: int) -> int:
    """Bytes the whole decode call must move: KV rows once, q, out, the
    block-table entries in use, seq_lens, and for split-K the partial states
    written by the partition kernel and read back by the reduce."""
    import torch
    el = w.kv_cache.element_size()
    L = w.seq_lens.to(torch.int64)
    nblk = int(((L + w.block_size - 1) // w.block_size).sum().item())
    b = kv_bytes(w) + 2 * w.q.numel() * el + nblk * 4 + w.num_seqs * 4
    if split:
        written, read, _ = split_partials(w, partition)
        b += written + read
    return b


def decode_kernel_bytes(w, split: bool, partition: int) -> int:
    """Bytes the main attention kernel alone must move: KV rows once, q, the
    block-table entries in use, seq_lens, the output rows it writes itself
    and the partial states (written once; the reduce reads them and writes
    the other output rows)."""
    import torch
    el = w.kv_cache.element_size()
    L = w.seq_lens.to(torch.int64)
    nblk = int(((L + w.block_size - 1) // w.block_size).sum().item())
    b = kv_bytes(w) + w.q.numel() * el + nblk * 4 + w.num_seqs * 4
    if not split:
        return b + w.q.numel() * el
    written, _, reduce_out = split_partials(w, partition)
    return b + (w.q.numel() * el - reduce_out) + written


def decode_launches(w, split: bool, partition: int) -> int:
    """Kernels one decode call launches: one-pass = 1; split-K = plan +
    decode + (reduce when a sequence can span several partitions) for the
    tensor-core path (head_size 128), decode + reduce otherwise."""
    if not split:
        return 1
    msl = int(w.seq_lens.max().item())
    if w.head_size == 128:
        return 2 + (1 if msl > partition else 0)
    return 2


def reshape_launch_bytes(w) -> int:
    valid = int((w.slot_mapping >= 0).sum().item())
    row = w.num_kv_heads * w.head_size * w.kv_cache.element_size()
    return 2 * 2 * valid * row + w.slot_mapping.numel() * 8


def source_digest() -> str:
    h = hashlib.sha256()
    for rel in DECODE_SOURCES:
        with open(os.path.join(ROOT, rel), "rb") as f:
            h.update(f.read())
    return h.hexdigest()[:16]


def recorded_traffic(config: str, decode: str) -> int | None:
    """DRAM bytes per launch of the decode kernel from the committed ncu
    summary, if it was taken on the current kernel source."""
    path = os.path.join(ROOT, "profiles", f"decode_{decode}_{config}.md")
    if not os.path.exists(path):
        return None
    m = re.search(r"bench-traffic:\s*bytes=(\d+)\s+source=([0-9a-f]+)", open(path).read())
    if not m or m.group(2) != source_digest():
        return None
    return int(m.group(1))


def measured_peaks() -> dict:
    path = os.path.join(ROOT, "MEASURED_PEAKS.json")
    if os.path.exists(path):
        with open(path) as f:
            d = json.load(f)
        return {"hbm_gbs": float(d["hbm_gbs"]), "bf16_tflops": float(d["bf16_tflops"]),
                "source": "measured"}
    return {"hbm_gbs": 6800.0, "bf16_tflops": 1900.0, "source": "fallback"}


# ---------------------------------------------------------------------------
# CPU oracle timing (the baseline)
# ---------------------------------------------------------------------------

def oracle_sample_run(w, groups, nthreads: int):
    """Run the oracle on (seq, kv head) groups, all query heads of each group;
    returns (seconds, kv bytes covered)."""
    import numpy as np
    import workload as wl
    from oracle.oracle import get
    orc = get()
    G = w.num_heads // w.num_kv_heads
    items = np.array([s * w.num_heads + kvh * G + g for s, kvh in groups for g in range(G)],
                     dtype=np.int32)
    q = wl.bits(w.q)
    cache = wl.bits(w.kv_cache)
    bt = w.block_tables.cpu().numpy()
    sl = w.seq_lens.cpu().numpy()
    el = w.kv_cache.element_size()
    t = time.perf_counter()
    orc.decode(q, cache, bt, sl, w.num_kv_heads, w.block_size, w.scale,
               wl.ORACLE_DTYPE[w.dtype], items=items, nthreads=nthreads)
    dt = time.perf_counter() - t
    covered = sum(int(sl[s]) for s, _ in groups) * w.head_size * el * 2
    return dt, covered


def cpu_baseline(w, budget_s: float = 10.0) -> dict:
    nthreads = os.cpu_count() or 1
    groups_all = [(s, k) for s in range(w.num_seqs) for k in range(w.num_kv_heads)]
    # pilot: one sequence's groups, then scale the sample to the budget
    pilot = groups_all[: w.num_kv_heads]
    dt, _ = oracle_sample_run(w, pilot, nthreads)
    per_group = max(dt / len(pilot), 1e-6)
    n = int(min(len(groups_all), max(len(pilot), budget_s / per_group)))
    n = max(w.num_kv_heads, n // w.num_kv_heads * w.num_kv_heads)   # whole sequences
    sample = groups_all[:n]
    # Repeat the sample until the budget is spent (the whole workload can take
    # far less than the budget on many cores).
    dt, covered, passes = 0.0, 0, 0
    while passes == 0 or dt < budget_s:
        t, c = oracle_sample_run(w, sample, nthreads)
        dt += t
        covered += c
        passes += 1
    seqs = n // w.num_kv_heads
    return {"value": covered / dt / 1e9, "unit": UNIT, "cores": nthreads, "kind": "oracle",
            "sample": f"decode of sequences 0-{seqs - 1} of {w.num_seqs} (all heads), "
                      f"{passes} pass(es), fp64 two-pass oracle, {dt:.2f} s",
            "seconds": dt, "seqs_per_s": passes * seqs / dt}


# ---------------------------------------------------------------------------
# Our arm
# ---------------------------------------------------------------------------

def main_kernel_name(w, split: bool) -> str:
    """The attention kernel a decode call launches for this shape (mirrors the
    library's choice: tensor cores for head_size 128 in split-K and for
    grouped heads; PA_DECODE_KERNEL forces a family)."""
    forced = os.environ.get("PA_DECODE_KERNEL", "")
    G = w.num_heads // w.num_kv_heads
    tc = w.head_size == 128 and forced != "simt" and (forced == "tcgen05" or split or G >= 2)
    return "pa::tc::decode_tc_kernel" if tc else "pa::decode_kernel"


def time_main_kernel(pa, decode, n: int, stream) -> float:
    """Mean duration (ms) of the main attention kernel of `n` decode calls,
    from CUDA events the library records on the call's stream right before
    and after that kernel (pa_profile_kernel_events)."""
    import torch
    evs = [(torch.cuda.Event(enable_timing=True), torch.cuda.Event(enable_timing=True))
           for _ in range(n)]
    for a, b in evs:                       # torch creates events on first record
        a.record(stream)
        b.record(stream)
    torch.cuda.synchronize()
    try:
        for a, b in evs:
            pa.pa_profile_kernel_events(a, b)
            decode()
    finally:
        pa.pa_profile_kernel_events(None, None)
    torch.cuda.synchronize()
    return statistics.mean(a.elapsed_time(b) for a, b in evs)


def decode_config_entry(name: str, args, peak_gbs: float, w=None) -> dict:
    """One decode configuration through the bench step (cache write +
    pa_decode_splitk), device-resident: the step, the decode call and its main
    kernel, each timed with CUDA events on the launching stream."""
    import torch
    import paged_kv_cache_136_gb300 as pa
    import workload as wl
    own = w is None
    if own:
        w = wl.make(name, device="cuda", seed=args.seed)
    out = torch.empty_like(w.q)
    msl = int(w.seq_lens.max().item())
    P = args.partition
    ws = torch.empty(pa.pa_decode_splitk_workspace_size(w.num_seqs, w.num_heads, w.head_size,
                                                        msl, P), dtype=torch.uint8,
                     device="cuda")
    stream = torch.cuda.current_stream()

    def decode():
        pa.pa_decode_splitk(out, w.q, w.kv_cache, w.block_tables, w.seq_lens, w.scale,
                            w.block_size, msl, ws, P)

    for _ in range(5):
        pa.pa_reshape_and_cache(w.key, w.value, w.kv_cache, w.slot_mapping, w.block_size)
        decode()
    n = max(3, args.workload_steps)
    t0, t1 = torch.cuda.Event(enable_timing=True), torch.cuda.Event(enable_timing=True)
    torch.cuda.synchronize()
    t0.record(stream)
    for _ in range(n):
        pa.pa_reshape_and_cache(w.key, w.value, w.kv_cache, w.slot_mapping, w.block_size)
        decode()
    t1.record(stream)
    torch.cuda.synchronize()
    ms = t0.elapsed_time(t1) / n
    ev = [[torch.cuda.Event(enable_timing=True) for _ in range(2)] for _ in range(n)]
    for i in range(n):
        pa.pa_reshape_and_cache(w.key, w.value, w.kv_cache, w.slot_mapping, w.block_size)
        ev[i][0].record(stream)
        decode()
        ev[i][1].record(stream)
    torch.cuda.synchronize()
    call_ms = statistics.mean(e[0].elapsed_time(e[1]) for e in ev)
    kern_ms = time_main_kernel(pa, decode, n, stream)
    kvb = kv_bytes(w)
    cb = decode_launch_bytes(w, True, P)
    kb = decode_kernel_bytes(w, True, P)
    res = {"workload": WORKLOAD_TEXT[name], "call": "pa_decode_splitk", "partition_size": P,
           "steps": n, "kv_bytes_per_step": kvb,
           "ms_per_step": round(ms, 5), "step_gbs": round(kvb / ms / 1e6, 2),
           "seqs_per_s": round(w.num_seqs / (ms / 1e3), 1),
           "call_ms": round(call_ms, 5), "call_bytes": cb,
           "call_gbs": round(cb / call_ms / 1e6, 2),
           "call_frac": round(cb / call_ms / 1e6 / peak_gbs, 4),
           "kernel": main_kernel_name(w, True), "kernel_ms": round(kern_ms, 5),
           "kernel_bytes": kb, "kernel_gbs": round(kb / kern_ms / 1e6, 2),
           "kernel_frac": round(kb / kern_ms / 1e6 / peak_gbs, 4),
           "device_error_flags": pa.pa_device_errors(clear=True)}
    if name == "prefix":
        ub = w.unique_kv_bytes()
        res["unique_kv_bytes_per_step"] = ub
        res["unique_call_gbs"] = round(ub / call_ms / 1e6, 2)
        res["note"] = ("the shared 8 MB prefix is read from L2 by all 128 sequences, so logical "
                       "bytes exceed the HBM rate; the unique bytes are the HBM-bound figure")
    if name == "tiny":
        res["note"] = "117,760 KV bytes: launch-latency bound, no HBM roofline applies"
        res["c_abi_latency"] = c_abi_latency()
    if own:
        del w
    del ws, out
    torch.cuda.empty_cache()
    return res


def c_abi_latency() -> dict | None:
    """The library's own latency floor on the tiny workload, from the host
    program built beside libpa.so (no Python in its timed loops): host time
    per API call, device time per call, and a synchronous step."""
    import paged_kv_cache_136_gb300 as pa
    tool = os.path.join(os.path.dirname(pa.lib_path()), "pa_latency")
    if not os.path.exists(tool):
        return None
    try:
        r = subprocess.run([tool, "2000"], capture_output=True, text=True, timeout=120)
    except subprocess.TimeoutExpired:
        return {"error": "timed out"}
    if r.returncode != 0:
        return {"error": (r.stderr or r.stdout).strip()[-200:]}
    return json.loads(r.stdout.strip().splitlines()[-1])


def run_ours(args) -> dict | None:
    import torch
    rank, world, local = dist_env()
    dist_mod = init_dist(world, "nccl")
    torch.cuda.set_device(local)
    import paged_kv_cache_136_gb300 as pa
    import workload as wl

    split = args.decode == "splitk"
    P = args.partition
    w = wl.make(args.config, seed=args.seed + rank, device="cuda")
    dev = w.q.device
    stream = torch.cuda.current_stream()
    out = torch.empty_like(w.q)
    msl = int(w.seq_lens.max().item())
    ws = torch.empty(pa.pa_decode_splitk_workspace_size(w.num_seqs, w.num_heads, w.head_size,
                                                        msl, P), dtype=torch.uint8, device=dev)

    def decode():
        if split:
            pa.pa_decode_splitk(out, w.q, w.kv_cache, w.block_tables, w.seq_lens, w.scale,
                                w.block_size, msl, ws, P)
        else:
            pa.pa_decode(out, w.q, w.kv_cache, w.block_tables, w.seq_lens, w.scale,
                         w.block_size)

    def step():
        pa.pa_reshape_and_cache(w.key, w.value, w.kv_cache, w.slot_mapping, w.block_size)
        decode()

    for _ in range(args.warmup):
        step()
    torch.cuda.synchronize()
    pa.pa_device_errors(clear=True)

    # The timed region: K steps back to back, events only at its two ends
    # (an event between two kernels would stop the next one's launch from
    # overlapping the previous one's tail).
    K = args.steps
    t_start = torch.cuda.Event(enable_timing=True)
    t_stop = torch.cuda.Event(enable_timing=True)
    clocks = ClockSampler(local) if rank == 0 else None
    if clocks:
        clocks.start()
    barrier(dist_mod)
    torch.cuda.synchronize()
    t_start.record(stream)
    for _ in range(K):
        step()
    t_stop.record(stream)
    torch.cuda.synchronize()
    barrier(dist_mod)
    clk = clocks.stop() if clocks else None
    ms_local = t_start.elapsed_time(t_stop)
    flags = pa.pa_device_errors(clear=True)

    # Per-call times (outside the timed region): events around each call.
    n_calls = max(3, min(K, 200))
    ev = [[torch.cuda.Event(enable_timing=True) for _ in range(3)] for _ in range(n_calls)]
    torch.cuda.synchronize()
    for i in range(n_calls):
        ev[i][0].record(stream)
        pa.pa_reshape_and_cache(w.key, w.value, w.kv_cache, w.slot_mapping, w.block_size)
        ev[i][1].record(stream)
        decode()
        ev[i][2].record(stream)
    torch.cuda.synchronize()
    dec_ms = statistics.mean(e[1].elapsed_time(e[2]) for e in ev)
    rsh_ms = statistics.mean(e[0].elapsed_time(e[1]) for e in ev)

    ms_max = reduce_scalar(ms_local, "max", dist_mod, dev)
    bytes_all = reduce_scalar(float(kv_bytes(w)) * K, "sum", dist_mod, dev)
    seqs_all = reduce_scalar(float(w.num_seqs) * K, "sum", dist_mod, dev)
    value = bytes_all / (ms_max / 1e3) / 1e9

    # The main attention kernel alone (outside the timed region above: the
    # events between the kernels of a call stop its launch overlap).
    kern_ms = time_main_kernel(pa, decode, n_calls, stream)

    # End to end through the public API: per step, copy the step's inputs
    # from pinned host memory, run the step, read the result back, and wait
    # for it on the host (a decode loop needs step i's output before it can
    # build step i+1's input).  The inputs live in one staging buffer (one
    # copy per step, as a serving engine stages them).  The headline runs the
    # Python API calls eagerly, every host-side check and launch included;
    # the same step replayed as a CUDA graph is reported beside it.
    names = ("q", "key", "value", "slot_mapping", "block_tables", "seq_lens")
    offs, total = {}, 0
    for k in names:
        t = getattr(w, k)
        offs[k] = total
        total += (t.numel() * t.element_size() + 255) // 256 * 256
    dev_buf = torch.empty(total, dtype=torch.uint8, device=dev)
    host_buf = torch.empty(total, dtype=torch.uint8).pin_memory()
    for k in names:
        t = getattr(w, k)
        nbytes = t.numel() * t.element_size()
        view = dev_buf[offs[k]:offs[k] + nbytes].view(t.dtype).view(t.shape)
        view.copy_(t)
        host_buf[offs[k]:offs[k] + nbytes].copy_(t.cpu().contiguous().view(-1).view(torch.uint8))
        setattr(w, k, view)
    h2d_len = offs[names[-1]] + getattr(w, names[-1]).numel() * 4
    out_h = torch.empty(out.shape, dtype=out.dtype).pin_memory()
    h2d = sum(getattr(w, k).numel() * getattr(w, k).element_size() for k in names)
    d2h = out_h.numel() * out_h.element_size()
    e2e_steps = max(1, min(K, args.e2e_steps))

    def e2e_body():
        pa.pa_stage_copy(dev_buf[:h2d_len], host_buf[:h2d_len])
        step()
        pa.pa_stage_copy(out_h, out)

    def e2e_eager():
        e2e_body()
        torch.cuda.current_stream().synchronize()

    for _ in range(3):
        e2e_eager()
    barrier(dist_mod)
    t0 = time.perf_counter()
    for _ in range(e2e_steps):
        e2e_eager()
    e2e_local = time.perf_counter() - t0
    barrier(dist_mod)
    e2e_max = reduce_scalar(e2e_local, "max", dist_mod, dev)
    e2e_bytes = reduce_scalar(float(kv_bytes(w)) * e2e_steps, "sum", dist_mod, dev)

    graph = None
    try:
        graph = torch.cuda.CUDAGraph()
        with torch.cuda.graph(graph):
            e2e_body()
        torch.cuda.synchronize()
    except Exception:                      # capture unavailable on this setup
        graph = None
        torch.cuda.synchronize()
    g_value = None
    if graph is not None:
        for _ in range(3):
            graph.replay()
            torch.cuda.current_stream().synchronize()
        barrier(dist_mod)
        t0 = time.perf_counter()
        for _ in range(e2e_steps):
            graph.replay()
            torch.cuda.current_stream().synchronize()
        g_local = time.perf_counter() - t0
        barrier(dist_mod)
        g_max = reduce_scalar(g_local, "max", dist_mod, dev)
        g_value = round(e2e_bytes / g_max / 1e9, 2)

    if rank != 0:
        return None
    peaks = measured_peaks()
    call_bytes = decode_launch_bytes(w, split, P)
    kern_bytes = decode_kernel_bytes(w, split, P)
    achieved = kern_bytes / (kern_ms / 1e3) / 1e9
    call_gbs = call_bytes / (dec_ms / 1e3) / 1e9
    line = {
        "metric": METRIC, "value": round(value, 2), "unit": UNIT, "n_gpus": world,
        "steps": K, "warmup": args.warmup, "ms_per_step": round(ms_max / K, 5),
        "higher_is_better": True, "scaling": "weak", "vs_baseline": None, "dtype": "f32",
        "data": "synthetic",
        "config": {"workload": WORKLOAD_TEXT[args.config], "name": args.config,
                   "batch": w.num_seqs, "num_heads": w.num_heads,
                   "num_kv_heads": w.num_kv_heads, "head_size": w.head_size,
                   "block_size": w.block_size, "storage_dtype": str(w.dtype).replace("torch.", ""),
                   "decode": "pa_decode_splitk" if split else "pa_decode",
                   "partition_size": P if split else None,
                   "kv_bytes_per_step": kv_bytes(w),
                   "l2": "inputs larger than L2: the KV pool exceeds the 129 MB L2, no flush",
                   "parallelism": f"replicas x{world}", "seed": args.seed},
        "seqs_per_s": round(seqs_all / (ms_max / 1e3), 1),
        "pct_hbm_peak": round(100.0 * value / peaks["hbm_gbs"], 2),
        "roofline": {"bound": "hbm", "kernel": main_kernel_name(w, split),
                     "achieved": round(achieved, 2),
                     "peak": peaks["hbm_gbs"], "peak_source": peaks["source"] + " copy, burst",
                     "unit": "GB/s", "frac": round(achieved / peaks["hbm_gbs"], 4),
                     "traffic": recorded_traffic(args.config, "splitk" if split else "onepass"),
                     "algorithmic_bytes_per_launch": kern_bytes,
                     "ms_per_launch": round(kern_ms, 5),
                     "timing": "CUDA events recorded by the library right before and after "
                               "the kernel (pa_profile_kernel_events), mean of the launches",
                     "call": {"what": ("pa_decode_splitk call: plan, partition and reduce "
                                       "kernels") if split else "pa_decode call",
                              "ms_per_launch": round(dec_ms, 5),
                              "algorithmic_bytes_per_launch": call_bytes,
                              "achieved": round(call_gbs, 2),
                              "frac": round(call_gbs / peaks["hbm_gbs"], 4)}},
        "reshape": {"ms_per_launch": round(rsh_ms, 5),
                    "algorithmic_bytes_per_launch": reshape_launch_bytes(w)},
        "e2e": {"value": round(e2e_bytes / e2e_max / 1e9, 2), "unit": UNIT,
                "h2d_bytes_per_step": h2d, "d2h_bytes_per_step": d2h, "steps": e2e_steps,
                "method": "eager Python API calls each step: one pinned staging copy in, "
                          "cache write, decode, result copy out (both copies on the SMs, "
                          "pa_stage_copy), host waits for the result",
                "graph_value": g_value,
                "graph_method": "the same step captured once as a CUDA graph and replayed"},
        "gpu_launches": K * (1 + decode_launches(w, split, P)),
        "clocks": clk,
        "device_error_flags": flags,
        "kernel_source": source_digest(),
    }
    if world == 1 and not args.no_cpu_baseline:
        line["cpu_baseline"] = cpu_baseline(w, budget_s=args.cpu_budget)
    del w, ws, out, out_h, dev_buf, host_buf, graph
    torch.cuda.empty_cache()
    if world == 1 and args.configs:
        by = {args.config: {"kernel": line["roofline"]["kernel"],
                            "kernel_frac": line["roofline"]["frac"],
                            "kernel_gbs": line["roofline"]["achieved"],
                            "kernel_ms": line["roofline"]["ms_per_launch"],
                            "call_frac": line["roofline"]["call"]["frac"],
                            "call_ms": line["roofline"]["call"]["ms_per_launch"],
                            "step_gbs": line["value"], "seqs_per_s": line["seqs_per_s"]}}
        for name in args.configs.split(","):
            if name and name != args.config:
                by[name] = decode_config_entry(name, args, peaks["hbm_gbs"])
        line["roofline"]["by_config"] = by
    if world == 1 and args.workloads:
        line["workloads"] = [other_workload(name, args, peaks["hbm_gbs"])
                             for name in args.workloads.split(",") if name]
    return line


def copy_blocks_workload(args, peak_gbs: float) -> dict:
    """Copy-on-write block copies on the mha7b pool: a quarter of the pool's
    blocks copied into another quarter per launch (disjoint sources and
    destinations, shuffled), timed per launch with CUDA events.  Bytes per
    pair: the K and V planes of one block read and written."""
    import numpy as np
    import torch
    import paged_kv_cache_136_gb300 as pa
    import workload as wl
    w = wl.make("mha7b", device="cuda", seed=args.seed)
    nb = w.num_blocks
    n = nb // 4
    ids = np.random.default_rng(args.seed).permutation(nb)
    mapping = torch.from_numpy(np.stack([ids[:n], ids[n:2 * n]], 1).astype(np.int64)).cuda()
    plane = w.block_size * w.num_kv_heads * w.head_size * w.kv_cache.element_size()
    nbytes = n * 2 * 2 * plane + mapping.numel() * 8
    stream = torch.cuda.current_stream()
    for _ in range(5):
        pa.pa_copy_blocks(w.kv_cache, mapping, w.block_size)
    k = max(3, args.workload_steps)
    ev = [[torch.cuda.Event(enable_timing=True) for _ in range(2)] for _ in range(k)]
    torch.cuda.synchronize()
    for i in range(k):
        ev[i][0].record(stream)
        pa.pa_copy_blocks(w.kv_cache, mapping, w.block_size)
        ev[i][1].record(stream)
    torch.cuda.synchronize()
    ms = statistics.mean(e[0].elapsed_time(e[1]) for e in ev)
    res = {"name": "copy_blocks", "call": "pa_copy_blocks",
           "workload": f"{n} (src, dst) block pairs of the mha7b pool ({nb} blocks, "
                       f"{plane} B per K or V block plane), disjoint, shuffled",
           "launches": k, "bytes_per_launch": nbytes, "ms_per_launch": round(ms, 5),
           "gbs": round(nbytes / ms / 1e6, 2),
           "frac": round(nbytes / ms / 1e6 / peak_gbs, 4),
           "device_error_flags": pa.pa_device_errors(clear=True)}
    del w, mapping
    torch.cuda.empty_cache()
    return res


def prefill_workload(name: str, args, peaks: dict) -> dict:
    """Prefill step (cache write of the new tokens + causal prefill attention
    over the paged pool), device-resident, timed per call with CUDA events.
    Work per call: 4 * head_size flops per (query row, attended key, query
    head) -- the QK^T and PV contractions -- over the causal pairs only."""
    import torch
    import paged_kv_cache_136_gb300 as pa
    import workload as wl
    w = wl.make_prefill(name, device="cuda")
    out = torch.empty_like(w.q)
    mq = int(w.q_lens().max())
    stream = torch.cuda.current_stream()

    def call():
        pa.pa_prefill(out, w.q, w.kv_cache, w.block_tables, w.seq_lens, w.query_start_loc,
                      w.scale, w.block_size, mq)

    for _ in range(5):
        pa.pa_reshape_and_cache(w.key, w.value, w.kv_cache, w.slot_mapping, w.block_size)
        call()
    k = max(3, args.workload_steps)
    ev = [[torch.cuda.Event(enable_timing=True) for _ in range(3)] for _ in range(k)]
    torch.cuda.synchronize()
    for i in range(k):
        ev[i][0].record(stream)
        pa.pa_reshape_and_cache(w.key, w.value, w.kv_cache, w.slot_mapping, w.block_size)
        ev[i][1].record(stream)
        call()
        ev[i][2].record(stream)
    torch.cuda.synchronize()
    step_ms = statistics.mean(e[0].elapsed_time(e[2]) for e in ev)
    ms = statistics.mean(e[1].elapsed_time(e[2]) for e in ev)
    flops = 4 * w.head_size * w.num_heads * w.causal_pairs()
    tf = flops / ms / 1e9
    peak = peaks.get("bf16_tflops")
    res = {"name": name, "call": "pa_prefill (causal)", "workload": PREFILL_TEXT[name],
           "launches": k, "tokens": w.num_tokens, "flops_per_call": flops,
           "ms_per_call": round(ms, 5), "tflops": round(tf, 2),
           "roofline": {"bound": "tensor", "achieved": round(tf, 2), "peak": peak,
                        "unit": "TFLOP/s", "frac": round(tf / peak, 4),
                        "peak_source": peaks["source"] + " bf16 dense (cuBLAS), burst; "
                                       "fp16 has the same nominal rate"},
           "ms_per_step": round(step_ms, 5),
           "tokens_per_s": round(w.num_tokens / (step_ms / 1e3), 1),
           "device_error_flags": pa.pa_device_errors(clear=True)}
    del w, out
    torch.cuda.empty_cache()
    return res


def cascade_workload(args, peak_gbs: float) -> dict:
    """The shared-prefix workload through pa_cascade_decode (prefix attended
    once for all sequences, suffixes split-K, merged), with the cache write,
    timed like the other workloads.  Throughput is reported on the same
    logical KV bytes as the plain decode (every sequence's full length), and
    on the distinct bytes the cascade has to read."""
    import torch
    import paged_kv_cache_136_gb300 as pa
    import workload as wl
    w = wl.make("prefix", device="cuda")
    out = torch.empty_like(w.q)
    msl = int(w.seq_lens.max().item())
    pb = w.meta["shared_blocks"]
    P = args.partition
    n = pa.pa_cascade_decode_workspace_size(w.num_seqs, w.num_heads, w.head_size,
                                            w.block_tables.shape[1], pb, msl, w.block_size, P)
    ws = torch.empty(n, dtype=torch.uint8, device="cuda")
    stream = torch.cuda.current_stream()

    def call():
        pa.pa_cascade_decode(out, w.q, w.kv_cache, w.block_tables, w.seq_lens, w.scale,
                             w.block_size, pb, msl, ws, P)

    for _ in range(5):
        pa.pa_reshape_and_cache(w.key, w.value, w.kv_cache, w.slot_mapping, w.block_size)
        call()
    k = max(3, args.workload_steps)
    ev = [[torch.cuda.Event(enable_timing=True) for _ in range(3)] for _ in range(k)]
    torch.cuda.synchronize()
    for i in range(k):
        ev[i][0].record(stream)
        pa.pa_reshape_and_cache(w.key, w.value, w.kv_cache, w.slot_mapping, w.block_size)
        ev[i][1].record(stream)
        call()
        ev[i][2].record(stream)
    torch.cuda.synchronize()
    step_ms = statistics.mean(e[0].elapsed_time(e[2]) for e in ev)
    ms = statistics.mean(e[1].elapsed_time(e[2]) for e in ev)
    kvb = kv_bytes(w)
    ub = w.unique_kv_bytes()
    res = {"name": "prefix_cascade", "call": "pa_cascade_decode", "workload": WORKLOAD_TEXT["prefix"],
           "prefix_blocks": pb, "partition_size": P, "steps": k,
           "kv_bytes_per_step": kvb, "unique_kv_bytes_per_step": ub,
           "ms_per_call": round(ms, 5), "ms_per_step": round(step_ms, 5),
           "decode_gbs_logical": round(kvb / ms / 1e6, 2),
           "decode_gbs_unique": round(ub / ms / 1e6, 2),
           "unique_frac_of_peak": round(ub / ms / 1e6 / peak_gbs, 4),
           "seqs_per_s": round(w.num_seqs / (step_ms / 1e3), 1),
           "gpu_launches_per_call": 5 + (1 if msl - pb * w.block_size > P else 0),
           "device_error_flags": pa.pa_device_errors(clear=True)}
    del w, ws, out
    torch.cuda.empty_cache()
    return res


def fp8_workload(name: str, args, peak_gbs: float) -> dict:
    """A decode workload with an FP8 (e4m3) pool: quantising cache write of the
    new tokens + split-K decode over the FP8 pool.  KV bytes are the e4m3
    codes read (one byte per element)."""
    import torch
    import paged_kv_cache_136_gb300 as pa
    import workload as wl
    base = name[len("fp8_"):]
    w = wl.make_fp8(base, device="cuda")
    ks, vs = w.meta["k_scale"], w.meta["v_scale"]
    out = torch.empty_like(w.q)
    msl = int(w.seq_lens.max().item())
    P = args.partition
    ws = torch.empty(pa.pa_decode_splitk_fp8_workspace_size(w.num_seqs, w.num_heads,
                                                            w.head_size, msl, P),
                     dtype=torch.uint8, device="cuda")
    stream = torch.cuda.current_stream()

    def write():
        pa.pa_reshape_and_cache_fp8(w.key, w.value, w.kv_cache, w.slot_mapping, w.block_size,
                                    ks, vs)

    def call():
        pa.pa_decode_splitk_fp8(out, w.q, w.kv_cache, w.block_tables, w.seq_lens, w.scale,
                                w.block_size, ks, vs, msl, ws, P)

    for _ in range(5):
        write()
        call()
    k = max(3, args.workload_steps)
    ev = [[torch.cuda.Event(enable_timing=True) for _ in range(3)] for _ in range(k)]
    torch.cuda.synchronize()
    for i in range(k):
        ev[i][0].record(stream)
        write()
        ev[i][1].record(stream)
        call()
        ev[i][2].record(stream)
    torch.cuda.synchronize()
    step_ms = statistics.mean(e[0].elapsed_time(e[2]) for e in ev)
    ms = statistics.mean(e[1].elapsed_time(e[2]) for e in ev)
    kvb = kv_bytes(w)
    res = {"name": name, "call": "pa_decode_splitk_fp8", "workload": WORKLOAD_TEXT[base] +
           "; FP8 e4m3 pool (k_scale = v_scale = 0.5)", "partition_size": P, "steps": k,
           "kv_bytes_per_step": kvb, "ms_per_call": round(ms, 5), "ms_per_step": round(step_ms, 5),
           "decode_gbs": round(kvb / ms / 1e6, 2), "decode_frac": round(kvb / ms / 1e6 / peak_gbs, 4),
           "step_gbs": round(kvb / step_ms / 1e6, 2),
           "seqs_per_s": round(w.num_seqs / (step_ms / 1e3), 1),
           "device_error_flags": pa.pa_device_errors(clear=True)}
    del w, ws, out
    torch.cuda.empty_cache()
    return res


def other_workload(name: str, args, peak_gbs: float) -> dict:
    """Short device-resident measurement of another workload, reported beside
    the main line."""
    if name == "copy_blocks":
        return copy_blocks_workload(args, peak_gbs)
    if name.startswith("prefill_"):
        return prefill_workload(name, args, measured_peaks())
    if name == "prefix_cascade":
        return cascade_workload(args, peak_gbs)
    if name.startswith("fp8_"):
        return fp8_workload(name, args, peak_gbs)
    return dict(decode_config_entry(name, args, peak_gbs), name=name)


# ---------------------------------------------------------------------------
# Reference arm: the CPU oracle on the host cores
# ---------------------------------------------------------------------------

def run_reference(args) -> dict | None:
    rank, world, _ = dist_env()
    if rank != 0:
        return None
    import workload as wl
    w = wl.make(args.config, seed=args.seed, device="cpu")
    nthreads = os.cpu_count() or 1
    groups_all = [(s, k) for s in range(w.num_seqs) for k in range(w.num_kv_heads)]
    dt, _ = oracle_sample_run(w, groups_all[:1], nthreads)
    budget_per_step = max(0.05, args.ref_budget / max(1, args.steps + args.warmup))
    n = int(max(1, min(len(groups_all), budget_per_step / max(dt, 1e-6))))
    sample = groups_all[:n]
    for _ in range(args.warmup):
        oracle_sample_run(w, sample, nthreads)
    tot_t, tot_b = 0.0, 0
    for _ in range(args.steps):
        dt, b = oracle_sample_run(w, sample, nthreads)
        tot_t += dt
        tot_b += b
    value = tot_b / tot_t / 1e9
    desc = f"{n} (sequence, kv head) groups of {len(groups_all)} per step, all query heads"
    return {
        "impl": "reference", "metric": METRIC, "value": round(value, 4), "unit": UNIT,
        "n_gpus": world, "steps": args.steps, "warmup": args.warmup,
        "ms_per_step": round(1e3 * tot_t / args.steps, 3), "higher_is_better": True,
        "scaling": "weak", "vs_baseline": None, "dtype": "f64", "data": "synthetic",
        "config": {"workload": WORKLOAD_TEXT[args.config], "name": args.config,
                   "sample": desc},
        "cpu_baseline": {"value": round(value, 4), "unit": UNIT, "cores": nthreads,
                         "kind": "oracle", "sample": desc},
        "e2e": {"value": round(value, 4), "unit": UNIT, "h2d_bytes_per_step": 0,
                "d2h_bytes_per_step": 0},
        "gpu_launches": 0,
    }


def run_profile_case(name: str, repeat: int, num_seqs: int | None = None) -> None:
    """Run one case `repeat` times and exit, for a profiler's launch capture:
    splitk_<config> (a bench step: cache write, split-K decode), prefill_<name>,
    fp8_<config>, prefix_cascade."""
    import torch
    import paged_kv_cache_136_gb300 as pa
    import workload as wl
    if name.startswith("prefill_"):
        w = wl.make_prefill(name, device="cuda")
        out = torch.empty_like(w.q)
        mq = int(w.q_lens().max())
        for _ in range(repeat):
            pa.pa_prefill(out, w.q, w.kv_cache, w.block_tables, w.seq_lens, w.query_start_loc,
                          w.scale, w.block_size, mq)
    elif name.startswith("fp8_"):
        w = wl.make_fp8(name[4:], device="cuda")
        msl = int(w.seq_lens.max())
        ws = torch.empty(pa.pa_decode_splitk_fp8_workspace_size(w.num_seqs, w.num_heads,
                                                                w.head_size, msl, 512),
                         dtype=torch.uint8, device="cuda")
        out = torch.empty_like(w.q)
        for _ in range(repeat):
            pa.pa_decode_splitk_fp8(out, w.q, w.kv_cache, w.block_tables, w.seq_lens, w.scale,
                                    w.block_size, w.meta["k_scale"], w.meta["v_scale"], msl,
                                    ws, 512)
    elif name.startswith("splitk_"):
        w = wl.make(name[7:], device="cuda", num_seqs=num_seqs)
        msl = int(w.seq_lens.max())
        ws = torch.empty(pa.pa_decode_splitk_workspace_size(w.num_seqs, w.num_heads,
                                                            w.head_size, msl, 512),
                         dtype=torch.uint8, device="cuda")
        out = torch.empty_like(w.q)
        for _ in range(repeat):
            pa.pa_reshape_and_cache(w.key, w.value, w.kv_cache, w.slot_mapping, w.block_size)
            pa.pa_decode_splitk(out, w.q, w.kv_cache, w.block_tables, w.seq_lens, w.scale,
                                w.block_size, msl, ws, 512)
    elif name == "prefix_cascade":
        w = wl.make("prefix", device="cuda")
        msl = int(w.seq_lens.max())
        pb = w.meta["shared_blocks"]
        n = pa.pa_cascade_decode_workspace_size(w.num_seqs, w.num_heads, w.head_size,
                                                w.block_tables.shape[1], pb, msl,
                                                w.block_size, 512)
        ws = torch.empty(n, dtype=torch.uint8, device="cuda")
        out = torch.empty_like(w.q)
        for _ in range(repeat):
            pa.pa_cascade_decode(out, w.q, w.kv_cache, w.block_tables, w.seq_lens, w.scale,
                                 w.block_size, pb, msl, ws, 512)
    else:
        raise SystemExit(f"unknown profile case {name}")
    torch.cuda.synchronize()
    print(f"{name}: {repeat} runs, device error flags {pa.pa_device_errors()}")


def parse_args(argv=None):
    ap = argparse.ArgumentParser(description=__doc__, formatter_class=argparse.RawDescriptionHelpFormatter)
    ap.add_argument("--gpus", type=int, default=1)
    ap.add_argument("--steps", type=int, default=2000)
    ap.add_argument("--warmup", type=int, default=20)
    ap.add_argument("--impl", choices=["ours", "reference"], default="ours")
    ap.add_argument("--config", choices=sorted(WORKLOAD_TEXT), default="long")
    ap.add_argument("--decode", choices=["splitk", "onepass"], default="splitk")
    ap.add_argument("--partition", type=int, default=512)
    ap.add_argument("--seed", type=int, default=2)
    ap.add_argument("--cpu-budget", type=float, default=10.0)
    ap.add_argument("--ref-budget", type=float, default=60.0)
    ap.add_argument("--no-cpu-baseline", action="store_true")
    ap.add_argument("--e2e-steps", type=int, default=50,
                    help="steps in the end-to-end (host buffers) measurement")
    ap.add_argument("--configs", default="mha7b,gqa8b,prefix,tiny",
                    help="other decode configurations measured like the main one and "
                         "reported under roofline.by_config ('' for none)")
    ap.add_argument("--workloads",
                    default="prefix_cascade,copy_blocks,prefill_mha7b,prefill_gqa8b,fp8_mha7b,"
                            "fp8_gqa8b",
                    help="other workloads measured briefly beside the main line ('' for none)")
    ap.add_argument("--workload-steps", type=int, default=50)
    ap.add_argument("--profile-case", default=None,
                    help="run one case --repeat times for a profiler and exit (no JSON): "
                         "splitk_<config>, prefill_<name>, fp8_<config>, prefix_cascade")
    ap.add_argument("--repeat", type=int, default=3)
    ap.add_argument("--profile-seqs", type=int, default=None,
                    help="with --profile-case splitk_<config>: only the first N sequences")
    return ap.parse_args(argv)


def main(argv=None):
    args = parse_args(argv)
    if args.profile_case:
        run_profile_case(args.profile_case, max(1, args.repeat), args.profile_seqs)
        return 0
    if args.warmup < 3:
        args.warmup = 3
    line = run_reference(args) if args.impl == "reference" else run_ours(args)
    if line is not None:
        print(json.dumps(line), flush=True)
    return 0


if __name__ == "__main__":
    sys.exit(main())
