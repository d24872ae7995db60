"""Benchmark: paged decode attention on the 8k-context GQA workload.

One step = one decode iteration of an 80-layer model for 100 sequences of
8192 tokens (64 query / 8 KV heads, head_dim 128, block 16): per layer the
step's new K/V rows are scattered into the paged cache (pa_kv_write) and the
decode attention runs over the whole cache (pa_decode).  The 80 layers share
one layer's cache (3.36 GB, far larger than the 129 MB L2, so nothing is
served from L2 across layers; no flush is needed).  The step has no
copy-on-write pairs (no sharing in this workload), so pa_block_copy is not
launched.  The allocation of the step's slots is done by the host allocator
before the timed region.

value  = decode tokens/s = sequences x steps / timed seconds (device-resident inputs)
e2e    = the same through the public API with pinned host buffers: every step
         copies its block tables, lengths and slot mapping, and every layer its
         query and new K/V rows, host -> device, and every layer's output back.

Steps that compute several new tokens per sequence (--workload spec72b: 4
speculative tokens per sequence; chunked: prompt chunks mixed into a decode
batch) run pa_attention_causal instead of pa_decode; there value counts the
query tokens computed per second.

Usage: python bench.py [--gpus N] [--steps K] [--warmup W] [--impl ours|reference]
Multi-GPU (torchrun): each rank runs its own replica of the workload (weak
scaling); the time is the maximum over ranks.
"""
from __future__ import annotations

import argparse
import json
import math
import os
import statistics
import subprocess
import sys
import time

import numpy as np

ROOT = os.path.dirname(os.path.abspath(__file__))
if ROOT not in sys.path:
    sys.path.insert(0, ROOT)

WORKLOAD = "gqa72b"
LAYERS = 80
METRIC = "paged decode attention tokens/s and KV GB/s vs GB300 HBM roofline"


def parse():
    p = argparse.ArgumentParser()
    p.add_argument("--gpus", type=int, default=1)
    p.add_argument("--steps", type=int, default=30)
    p.add_argument("--warmup", type=int, default=3)
    p.add_argument("--impl", choices=["ours", "reference"], default="ours")
    p.add_argument("--layers", type=int, default=None, help="default: 80 for gqa72b, 1 for the others")
    p.add_argument("--workload", default=WORKLOAD,
                   help="gqa72b (the headline), mha7b, mix, cow16, cow32, tiny; several tokens per sequence: "
                        "spec72b, chunked")
    p.add_argument("--kv-dtype", choices=["f16", "bf16", "fp8"], default="f16",
                   help="cache element type: fp16 (the pages'), bf16, or fp8 E4M3 codes with one scale per cache")
    p.add_argument("--no-cpu-baseline", action="store_true")
    p.add_argument("--no-graph", action="store_true", help="skip the CUDA Graph replay measurement")
    p.add_argument("--no-records", action="store_true",
                   help="headline run: skip the per-layer records of the other workloads")
    p.add_argument("--shared-prefix", action="store_true",
                   help="parallel-sampling workloads: decode with pa_decode_shared_prefix (samples of one prompt "
                        "read its blocks together)")
    p.add_argument("--spec-tokens", type=int, default=4,
                   help="spec72b: new (speculative) tokens per sequence (default 4)")
    p.add_argument("--seqs", type=int, default=None,
                   help="same shape with fewer sequences (small cases for profiling); default: the full 100")
    return p.parse_args()


def dist_env():
    return int(os.environ.get("RANK", 0)), int(os.environ.get("LOCAL_RANK", 0)), int(os.environ.get("WORLD_SIZE", 1))


def max_over_ranks(ms: float, device=None) -> float:
    """The largest of every rank's timing (ranks run independent replicas, so
    the job takes as long as the slowest one); the value itself when alone."""
    import torch
    import torch.distributed as dist
    if not (dist.is_available() and dist.is_initialized()) or dist.get_world_size() == 1:
        return float(ms)
    t = torch.tensor([float(ms)], dtype=torch.float64, device=device)
    dist.all_reduce(t, op=dist.ReduceOp.MAX)
    return float(t.item())


def job_tokens_per_s(world: int, seqs: int, steps: int, max_ms: float) -> float:
    """Whole-job decode throughput: every rank decodes `seqs` sequences per step."""
    return world * seqs * steps / (max_ms / 1e3)


KV_CODES = {"f16": 0, "bf16": 1, "fp8": 2}
FP8_SCALES = (1.0 / 64, 1.0 / 32)      # K and V scales of the fp8 caches (N(0, 1) data spans about +-5)


def inputs(w, kv_dtype):
    """Host arrays of the step in the cache's element type: (k_pool, v_pool,
    query, query_multi, new_key, new_value).  bf16: the fp16 draws truncated to
    bf16 patterns; fp8: seeded random finite E4M3 codes for the pools (any codes
    serve as cache content) and fp16 queries and new rows (quantised by the
    write)."""
    if kv_dtype == "f16":
        return w.k_pool, w.v_pool, w.query, w.query_multi, w.new_key, w.new_value
    if kv_dtype == "bf16":
        bf = lambda x: (np.asarray(x, dtype=np.float32).view(np.uint32) >> 16).astype(np.uint16)
        return (bf(w.k_pool), bf(w.v_pool), bf(w.query), bf(w.query_multi), bf(w.new_key), bf(w.new_value))
    shape = (w.num_blocks, w.num_kv_heads, w.block_size, w.head_dim)
    pools = []
    for stream in (1, 2):
        c = np.random.default_rng([w.seed, stream]).integers(0, 256, size=shape, dtype=np.uint8)
        c[(c & 0x7F) == 0x7F] = 0x38
        pools.append(c)
    return pools[0], pools[1], w.query, w.query_multi, w.new_key, w.new_value


def elem_bytes(kv_dtype) -> int:
    return 1 if kv_dtype == "fp8" else 2


def decode_bytes(w, esz=2) -> int:
    """Algorithmic bytes of one decode over the workload: every context token's
    K and V rows, the query, the output, the block-table entries the contexts
    need and the lengths."""
    L = w.context_lens.astype(np.int64)
    kv = int((L * 2 * w.num_kv_heads * w.head_dim * esz).sum())
    qo = 2 * w.num_seqs * w.num_heads * w.head_dim * 2
    tables = int((-(-L // w.block_size)).sum()) * 4
    return kv + qo + tables + 4 * w.num_seqs


def multi_token(w) -> bool:
    """Several new tokens per sequence are query rows of this step."""
    return bool(w.multi)


def causal_bytes(w, esz=2) -> int:
    """Algorithmic bytes of one multi-token call: every context token's K and
    V rows once per sequence (its new tokens share them), every query and
    output row, the block-table entries and the lengths and query offsets."""
    L = w.context_lens.astype(np.int64)
    kv = int((L * 2 * w.num_kv_heads * w.head_dim * esz).sum())
    qo = 2 * w.num_new_tokens * w.num_heads * w.head_dim * 2
    tables = int((-(-L // w.block_size)).sum()) * 4
    return kv + qo + tables + 4 * (2 * w.num_seqs + 1)


def causal_flops(w) -> int:
    """Multiply-adds x 2 of Q K^T and P V: new token j of sequence i sees
    L_i - T_i + j + 1 positions, for every query head."""
    L = w.context_lens.astype(np.int64)
    T = w.new_counts.astype(np.int64)
    seen = (T * (L - T + 1) + T * (T - 1) // 2).sum()       # sum over rows of the positions seen
    return int(4 * seen * w.num_heads * w.head_dim)


def prefill_launch(w, kv_dtype) -> bool:
    """Whether a multi-token call also launches the tensor-core kernel for long
    runs of new tokens (the library's rule: head_dim 128, G dividing 128, more
    than 16 query rows in the call; PA_PREFILL=0 disables)."""
    G = w.num_heads // w.num_kv_heads
    return (multi_token(w) and os.environ.get("PA_PREFILL", "1")[:1] != "0" and w.head_dim == 128
            and 128 % G == 0 and w.num_new_tokens * G >= 17)


def narrow_launch(w, kv_dtype) -> bool:
    """Whether a multi-token call that launches the tensor-core kernels also
    launches the narrow one, for sequences of at most 32 query rows (the
    library's rule; PA_NARROW=0 disables)."""
    return prefill_launch(w, kv_dtype) and os.environ.get("PA_NARROW", "1")[:1] != "0"


def shared_on_tensor_cores(w, kv_dtype) -> bool:
    """Whether pa_decode_shared_prefix reduces the shared ranges on the
    tensor-core kernel (the library's rule: fp16 cache, head_dim 128, G
    dividing 128; PA_PREFILL=0 or PA_SHARED_TC=0 disable)."""
    G = w.num_heads // w.num_kv_heads
    return (kv_dtype == "f16" and w.head_dim == 128 and 128 % G == 0
            and os.environ.get("PA_PREFILL", "1")[:1] != "0" and os.environ.get("PA_SHARED_TC", "1")[:1] != "0")


def kv_write_bytes(w, esz=2) -> int:
    """fp16/bf16 rows read, cache elements written, slots read."""
    T = w.num_new_tokens
    return 2 * (T * w.num_kv_heads * w.head_dim * (2 + esz)) + 8 * T


KERNEL_SOURCES = ("decode_common.cuh", "decode.cu", "common.cuh")   # what the fp16 decode kernel is built from


def kernel_traffic():
    """DRAM bytes per full decode launch from the committed ncu capture, or None
    when the decode kernel's source has changed since the capture was taken."""
    import hashlib
    try:
        rec = json.load(open(os.path.join(ROOT, "profiles", "decode_kernel_traffic.json")))
        src = b"".join(open(os.path.join(ROOT, "paged_kv_cache_12_gb300", "csrc", f), "rb").read()
                       for f in KERNEL_SOURCES)
        if hashlib.sha256(src).hexdigest() == rec["source_sha256"]:
            return int(rec["dram_bytes_per_launch"])
    except Exception:
        pass
    return None


def measured_peaks():
    try:
        return json.load(open(os.path.join(ROOT, "MEASURED_PEAKS.json")))
    except Exception:
        return None


class ClockSampler:
    """nvidia-smi samples of SM clock and throttle reasons during the timed region."""

    FIELDS = ("index,clocks.sm,clocks.max.sm,power.draw,clocks_event_reasons.active,"
              "clocks_event_reasons.hw_slowdown,clocks_event_reasons.hw_thermal_slowdown,"
              "clocks_event_reasons.sw_thermal_slowdown,clocks_event_reasons.sw_power_cap")

    def __init__(self, gpu_index: int):
        self.gpu = gpu_index
        self.proc = None

    def __enter__(self):
        try:
            self.proc = subprocess.Popen(
                ["nvidia-smi", "-i", str(self.gpu), f"--query-gpu={self.FIELDS}", "--format=csv,noheader,nounits",
                 "-lms", "200"], stdout=subprocess.PIPE, stderr=subprocess.DEVNULL, text=True)
        except Exception:
            self.proc = None
        return self

    def __exit__(self, *exc):
        self.lines = []
        if self.proc is not None:
            self.proc.terminate()
            try:
                out, _ = self.proc.communicate(timeout=5)
            except Exception:
                self.proc.kill()
                out, _ = self.proc.communicate()
            self.lines = [l for l in out.splitlines() if l.strip()]

    def summary(self):
        sm, mx, reasons = [], None, set()
        names = ("hw_slowdown", "hw_thermal_slowdown", "sw_thermal_slowdown", "sw_power_cap")
        for l in getattr(self, "lines", []):
            parts = [x.strip() for x in l.split(",")]
            if len(parts) < 9:
                continue
            try:
                sm.append(float(parts[1]))
                mx = float(parts[2])
            except ValueError:
                continue
            for n, v in zip(names, parts[5:9]):
                if v.lower() == "active":
                    reasons.add(n)
        if not sm:
            return {"sm_mhz": None, "sm_max_mhz": mx, "reasons": sorted(reasons), "samples": 0}
        return {"sm_mhz": statistics.median(sm), "sm_max_mhz": mx, "reasons": sorted(reasons), "samples": len(sm)}


# --------------------------------------------------------------- oracle timing

class OracleSample:
    """The oracle (as it stands, never tuned) on a bounded sample of the same
    workload: the first n of its sequences, one layer, on all host cores.
    n is calibrated once so that one timed call takes about `target_s`."""

    def __init__(self, w, tables, lens, target_s, kv_dtype="f16"):
        import oracle
        self.oracle, self.w, self.tables, self.lens = oracle, w, tables, lens
        self.kv_dtype = kv_dtype
        self.kpool, self.vpool, self.q, self.qm, _, _ = inputs(w, kv_dtype)
        self.threads = oracle.default_threads()
        self.multi = multi_token(w)
        # multi-token steps: sequences in index order, leaving out any one whose
        # rows alone would take the oracle longer than the whole sample (a long
        # prompt chunk; the oracle runs one sequence per thread)
        if self.multi:
            T = w.new_counts.astype(np.int64)
            cost = T * w.context_lens.astype(np.int64) * w.num_heads * w.head_dim * 4 / 1e9   # ~s at 1 GFLOP/s
            self.order = [i for i in range(w.num_seqs) if T[i] > 0 and cost[i] < target_s]
            self.skipped = w.num_seqs - len(self.order)
        else:
            self.order = list(range(w.num_seqs))
            self.skipped = 0
        n = min(self.threads, len(self.order))
        t = self.run(n)
        if t < target_s / 2 and n < len(self.order):
            n = min(len(self.order), int(n * target_s / max(t, 1e-3)))
            if n >= self.threads:
                n = (n // self.threads) * self.threads
        self.n = max(1, n)

    def rows(self, n):
        qs = self.w.query_start
        return int(sum(qs[i + 1] - qs[i] for i in self.order[:n]))

    def run(self, n):
        w = self.w
        t0 = time.perf_counter()
        kv = KV_CODES[self.kv_dtype]
        ks, vs = FP8_SCALES if self.kv_dtype == "fp8" else (1.0, 1.0)
        if self.multi:
            idx = np.asarray(self.order[:n])
            qs = w.query_start
            rows = np.concatenate([np.arange(qs[i], qs[i + 1]) for i in idx])
            sub_qs = np.concatenate([[0], np.cumsum(qs[idx + 1] - qs[idx])]).astype(np.int32)
            self.oracle.paged_attention_typed(self.qm[rows], self.kpool, self.vpool, self.tables[idx],
                                              self.lens[idx], sub_qs, w.num_kv_heads, w.block_size, w.scale, kv,
                                              ks, vs, threads=self.threads)
        elif self.kv_dtype == "f16":
            self.oracle.paged_decode(w.query, w.k_pool, w.v_pool, self.tables, self.lens, w.num_kv_heads,
                                     w.block_size, w.scale, threads=self.threads, seq_range=(0, n))
        else:
            self.oracle.paged_attention_typed(self.q[:n], self.kpool, self.vpool, self.tables[:n], self.lens[:n],
                                              None, w.num_kv_heads, w.block_size, w.scale, kv, ks, vs,
                                              threads=self.threads)
        return time.perf_counter() - t0

    def rate(self, layers=LAYERS):
        """(tokens/s for the `layers`-layer step, seconds of this call)"""
        secs = self.run(self.n)
        units = self.rows(self.n) if self.multi else self.n
        return units / (secs * layers), secs

    def describe(self, secs, layers=LAYERS):
        if self.multi:
            left = f", leaving out {self.skipped} sequence(s) too long for the sample" if self.skipped else ""
            return (f"{self.n} of {self.w.num_seqs} sequences ({self.rows(self.n)} of {self.w.num_new_tokens} "
                    f"query rows{left}), 1 of {layers} layer(s) ({secs:.1f} s per call), scaled to the "
                    f"{layers}-layer step")
        return (f"{self.n} of {self.w.num_seqs} sequences x {int(self.w.context_lens[0])} tokens, "
                f"1 of {layers} layers ({secs:.1f} s per call), scaled to the {layers}-layer step")


# ------------------------------------------------------------------ our arm

def workload(args):
    from paged_kv_cache_12_gb300 import workloads
    w = workloads.make(args.workload, spec_tokens=args.spec_tokens) if args.workload == "spec72b" \
        else workloads.make(args.workload)
    if args.seqs is None or args.seqs == w.num_seqs:
        return w
    if w.num_prompts:
        raise SystemExit("--seqs applies to the single-context workloads only")
    pick = (lambda a: list(a[: args.seqs]) if args.seqs <= w.num_seqs else [int(a[0])] * args.seqs)
    return workloads.custom(name=f"{w.name}-{args.seqs}seqs", seed=w.seed, num_seqs=args.seqs,
                            num_heads=w.num_heads, num_kv_heads=w.num_kv_heads, head_dim=w.head_dim,
                            block_size=w.block_size, context_lens=pick(w.context_lens), new_tokens=pick(w.new_counts),
                            multi=w.multi)


def history_allocator(w, pa):
    """A host allocator holding the workload's history (parallel-sampling
    workloads: one prompt per group, forked to its samples, the parent
    released): the state the step starts from."""
    al = pa.Allocator(w.num_blocks, w.block_size, free_order=w.free_order)
    ids = list(range(w.num_seqs))
    if w.num_prompts:
        for p in range(w.num_prompts):
            parent = 1_000_000 + p
            al.add_seq(parent)
            al.append([parent], [w.prompt_len])
            for k in range(w.samples_per_prompt):
                al.fork(parent, p * w.samples_per_prompt + k)
            al.free_seq(parent)
    else:
        for s in ids:
            al.add_seq(s)
        al.append(ids, w.history_lens)
    return al


def step_allocation(al, w):
    """The step's host allocation (step a1): slots for the step's new tokens
    (and the copy-on-write pairs they need), then the block tables and lengths
    the kernels read."""
    ids = list(range(w.num_seqs))
    slots, pairs = al.append(ids, w.new_counts)
    tables, lens = al.block_tables(ids, w.max_blocks_per_seq)
    return slots, pairs.reshape(-1, 2), tables, lens


def allocate(w, pa):
    """history_allocator, then the step's allocation.  Returns the allocator,
    the step's slot mapping and copy pairs, block tables, lengths and the
    step's allocation time in microseconds."""
    al = history_allocator(w, pa)
    t0 = time.perf_counter()
    slots, pairs, tables, lens = step_allocation(al, w)
    alloc_us = (time.perf_counter() - t0) * 1e6
    return al, slots, pairs, tables, lens, alloc_us


def unique_kv_bytes(w, tables, lens) -> int:
    """K/V bytes of the distinct cache slots the decode reads (shared prompt
    blocks counted once)."""
    bs = w.block_size
    slots = []
    for i in range(w.num_seqs):
        t = np.arange(int(lens[i]))
        slots.append(tables[i][t // bs].astype(np.int64) * bs + t % bs)
    n = len(np.unique(np.concatenate(slots))) if slots else 0
    return n * 2 * w.num_kv_heads * w.head_dim * 2


def describe(w, layers):
    L = w.context_lens
    ctx = f"{int(L[0])}-token context" if (L == L[0]).all() else f"context {int(L.min())}..{int(L.max())} tokens"
    extra = (f", {w.num_prompts} prompts x {w.samples_per_prompt} samples sharing a {w.prompt_len}-token prompt"
             if w.num_prompts else "")
    if multi_token(w):
        T = w.new_counts
        extra += (f", {w.num_new_tokens} new tokens computed causally (per sequence {int(T.min())}..{int(T.max())})")
    return (f"{w.name}: {w.num_seqs} sequences, {ctx}{extra}, {w.num_heads} query / {w.num_kv_heads} KV heads, "
            f"head_dim {w.head_dim}, block {w.block_size}, {layers} layer(s) per step sharing one layer's cache")


def run_ours(args):
    import torch

    import paged_kv_cache_12_gb300 as pa

    rank, local_rank, world = dist_env()
    if world > 1:
        import torch.distributed as dist
        dist.init_process_group("nccl", device_id=torch.device("cuda", local_rank))
    torch.cuda.set_device(local_rank)
    dev = torch.device("cuda", local_rank)
    w = workload(args)
    layers = args.layers if args.layers is not None else (LAYERS if w.name == WORKLOAD else 1)

    # ---- allocation (host) for this step
    al, slots, pairs, tables, lens, alloc_us = allocate(w, pa)
    has_pairs = len(pairs) > 0

    # ---- device-resident inputs
    multi = multi_token(w)
    kvd = args.kv_dtype
    kpool, vpool, q1, qmulti, nk_host, nv_host = inputs(w, kvd)
    q_host = qmulti if multi else q1
    cache_dt = {"f16": torch.float16, "bf16": torch.bfloat16, "fp8": torch.uint8}[kvd]
    row_dt = torch.bfloat16 if kvd == "bf16" else torch.float16
    dv = lambda a, dt: torch.from_numpy(np.ascontiguousarray(a)).to(dev).view(dt)
    k = dv(kpool, cache_dt)
    v = dv(vpool, cache_dt)
    q = dv(q_host, row_dt)
    nk = dv(nk_host, row_dt)
    nv = dv(nv_host, row_dt)
    ks, vs = FP8_SCALES if kvd == "fp8" else (1.0, 1.0)
    typed = kvd != "f16"
    d_slots = torch.from_numpy(slots).to(dev)
    d_pairs = torch.from_numpy(np.ascontiguousarray(pairs)).to(dev)
    d_tables = torch.from_numpy(tables).to(dev)
    d_lens = torch.from_numpy(lens).to(dev)
    out = torch.empty_like(q)
    shared_mode = bool(args.shared_prefix and w.num_prompts)
    if multi:
        d_qs = torch.from_numpy(w.query_start).to(dev)
        nws = pa.pa_attention_causal_workspace_size(w.num_seqs, w.num_new_tokens, w.num_heads, w.num_kv_heads,
                                                    w.head_dim, w.max_context_len)
    elif shared_mode:
        S = w.samples_per_prompt
        d_lead = torch.from_numpy(np.repeat(np.arange(w.num_prompts) * S, S).astype(np.int32)).to(dev)
        d_shl = torch.full((w.num_seqs,), w.prompt_len, dtype=torch.int32, device=dev)
        nws = pa.pa_decode_shared_prefix_workspace_size(w.num_seqs, w.num_heads, w.num_kv_heads, w.head_dim,
                                                        w.max_context_len)
    else:
        nws = pa.pa_decode_workspace_size(w.num_seqs, w.num_heads, w.num_kv_heads, w.head_dim, w.max_context_len)
    ws = torch.zeros(nws, dtype=torch.uint8, device=dev)
    stream = torch.cuda.current_stream()

    def writes_on(st, nk=nk, nv=nv):
        if has_pairs:
            pa.pa_block_copy(k, v, d_pairs, st)
        if kvd == "fp8":
            pa.pa_kv_write_fp8(nk, nv, d_slots, k, v, ks, vs, st)
        else:
            pa.pa_kv_write(nk, nv, d_slots, k, v, st)

    def decode_on(st, q=q, out=out):
        if multi and typed:
            pa.pa_attention_causal_typed(out, q, k, v, d_tables, d_lens, d_qs, w.scale, w.max_context_len, ws, ks, vs,
                                         st)
        elif multi:
            pa.pa_attention_causal(out, q, k, v, d_tables, d_lens, d_qs, w.scale, w.max_context_len, ws, st)
        elif typed:
            pa.pa_decode_typed(out, q, k, v, d_tables, d_lens, w.scale, w.max_context_len, ws, ks, vs, st)
        elif shared_mode:
            pa.pa_decode_shared_prefix(out, q, k, v, d_tables, d_lens, d_lead, d_shl, w.scale, w.max_context_len, ws,
                                       st)
        else:
            pa.pa_decode(out, q, k, v, d_tables, d_lens, w.scale, w.max_context_len, ws, st)

    def writes():
        writes_on(stream)

    def decode():
        decode_on(stream)

    def barrier():
        if world > 1:
            torch.distributed.barrier()
        torch.cuda.synchronize()

    # ---- device-resident timing, with per-decode events for the roofline
    for _ in range(args.warmup):
        for _ in range(layers):
            writes()
            decode()
    barrier()
    ev = [(torch.cuda.Event(enable_timing=True), torch.cuda.Event(enable_timing=True))
          for _ in range(args.steps * layers)]
    start, stop = torch.cuda.Event(enable_timing=True), torch.cuda.Event(enable_timing=True)
    with ClockSampler(local_rank) as clk:
        barrier()
        start.record(stream)
        i = 0
        for _ in range(args.steps):
            for _ in range(layers):
                writes()
                ev[i][0].record(stream)
                decode()
                ev[i][1].record(stream)
                i += 1
        stop.record(stream)
        barrier()
    assert pa.pa_workspace_status(ws) == pa.PA_OK
    total_ms = max_over_ranks(start.elapsed_time(stop), dev)
    dec_ms = [a.elapsed_time(b) for a, b in ev]

    # ---- the same step captured once in a CUDA Graph and replayed
    graph_ms = None
    if not args.no_graph:
        cs = torch.cuda.Stream()
        cs.wait_stream(stream)
        g = torch.cuda.CUDAGraph()
        with torch.cuda.stream(cs):
            with torch.cuda.graph(g, stream=cs):
                for _ in range(layers):
                    writes_on(cs)
                    decode_on(cs)
        stream.wait_stream(cs)
        for _ in range(args.warmup):
            g.replay()
        barrier()
        g0, g1 = torch.cuda.Event(enable_timing=True), torch.cuda.Event(enable_timing=True)
        g0.record(stream)
        for _ in range(args.steps):
            g.replay()
        g1.record(stream)
        barrier()
        graph_ms = max_over_ranks(g0.elapsed_time(g1), dev)
        del g

    # ---- end to end through the public API with pinned host buffers.  Every
    # step starts from its own allocator holding the history (made before the
    # timed region) and does the step's host allocation inside it: slots and
    # copy pairs for the new tokens, block tables and lengths, written into
    # pinned buffers (two sets, reused once their previous copies are done).
    n_e2e = args.warmup + args.steps
    fresh = [history_allocator(w, pa) for _ in range(n_e2e)]
    hbufs = [{"tables": torch.from_numpy(tables).pin_memory(), "lens": torch.from_numpy(lens).pin_memory(),
              "slots": torch.from_numpy(slots).pin_memory(),
              "pairs": torch.from_numpy(np.ascontiguousarray(pairs)).pin_memory()} for _ in range(2)]
    hdone = [torch.cuda.Event() for _ in range(2)]
    for ev_h in hdone:
        ev_h.record(stream)
    e2e_alloc_s = []
    h_tables, h_lens, h_slots, h_pairs = (hbufs[0][k] for k in ("tables", "lens", "slots", "pairs"))
    h_q = torch.from_numpy(np.ascontiguousarray(q_host)).pin_memory().view(row_dt)
    h_qs = torch.from_numpy(w.query_start).pin_memory() if multi else None
    h_nk = torch.from_numpy(np.ascontiguousarray(nk_host)).pin_memory().view(row_dt)
    h_nv = torch.from_numpy(np.ascontiguousarray(nv_host)).pin_memory().view(row_dt)
    h_out = torch.empty((layers,) + tuple(out.shape), dtype=out.dtype).pin_memory()

    # Layer l's inputs are copied in on a copy stream while layer l - 1 computes
    # (two device buffers of each), and its output is copied out while layer
    # l + 1 computes; every copy stays inside the timed region.
    cps = torch.cuda.Stream()
    qb, nkb, nvb, outb = [q, torch.empty_like(q)], [nk, torch.empty_like(nk)], [nv, torch.empty_like(nv)], \
        [out, torch.empty_like(out)]
    ev_in = [torch.cuda.Event() for _ in range(2)]       # buffer b's inputs are on the device
    ev_used = [torch.cuda.Event() for _ in range(2)]     # buffer b's inputs consumed, its output written
    ev_out = [torch.cuda.Event() for _ in range(2)]      # buffer b's output copied out
    for b in range(2):
        ev_used[b].record(stream)
        ev_out[b].record(stream)

    def copy_in(l):
        b = l & 1
        with torch.cuda.stream(cps):
            cps.wait_event(ev_used[b])
            qb[b].copy_(h_q, non_blocking=True)
            nkb[b].copy_(h_nk, non_blocking=True)
            nvb[b].copy_(h_nv, non_blocking=True)
            ev_in[b].record(cps)

    def e2e_step(i):
        t_a = time.perf_counter()
        s_i, p_i, tab_i, len_i = step_allocation(fresh[i], w)
        e2e_alloc_s.append(time.perf_counter() - t_a)
        assert len(p_i) == len(pairs)
        hb = hbufs[i & 1]
        hdone[i & 1].synchronize()          # this set's copies of two steps ago are done
        hb["tables"].numpy()[...] = tab_i
        hb["lens"].numpy()[...] = len_i
        hb["slots"].numpy()[...] = s_i
        d_tables.copy_(hb["tables"], non_blocking=True)
        d_lens.copy_(hb["lens"], non_blocking=True)
        d_slots.copy_(hb["slots"], non_blocking=True)
        if has_pairs:
            hb["pairs"].numpy()[...] = p_i
            d_pairs.copy_(hb["pairs"], non_blocking=True)
        hdone[i & 1].record(stream)
        if multi:
            d_qs.copy_(h_qs, non_blocking=True)
        copy_in(0)
        for l in range(layers):
            b = l & 1
            if l + 1 < layers:
                copy_in(l + 1)
            stream.wait_event(ev_in[b])
            stream.wait_event(ev_out[b])
            writes_on(stream, nkb[b], nvb[b])
            decode_on(stream, qb[b], outb[b])
            ev_used[b].record(stream)
            with torch.cuda.stream(cps):
                cps.wait_event(ev_used[b])
                h_out[l].copy_(outb[b], non_blocking=True)
                ev_out[b].record(cps)
        stream.wait_stream(cps)   # the step's last output is on the host

    for i in range(args.warmup):
        e2e_step(i)
    barrier()
    e2e_alloc_s.clear()
    e0, e1 = torch.cuda.Event(enable_timing=True), torch.cuda.Event(enable_timing=True)
    t_host = time.perf_counter()
    e0.record(stream)
    for i in range(args.steps):
        e2e_step(args.warmup + i)
    e1.record(stream)
    barrier()
    e2e_host_ms = (time.perf_counter() - t_host) * 1e3
    # the device clock from the step's first command to its last, or the host's
    # clock around the whole loop if that is longer (host-side allocation that
    # the device waited for)
    e2e_ms = max_over_ranks(max(e0.elapsed_time(e1), e2e_host_ms), dev)
    del fresh
    h2d = h_tables.numel() * 4 + h_lens.numel() * 4 + h_slots.numel() * 8 + (h_pairs.numel() * 8 if has_pairs else 0) \
        + (h_qs.numel() * 4 if multi else 0) + layers * (h_q.numel() * 2 + h_nk.numel() * 2 + h_nv.numel() * 2)
    d2h = layers * out.numel() * 2

    if rank != 0:
        if world > 1:
            torch.distributed.barrier()
            torch.distributed.destroy_process_group()
        return

    # ---- numbers
    B = w.num_new_tokens if multi else w.num_seqs      # query tokens computed per layer step
    tok_s = job_tokens_per_s(world, B, args.steps, total_ms)
    esz = elem_bytes(kvd)
    dbytes = causal_bytes(w, esz) if multi else decode_bytes(w, esz)
    step_bytes = layers * (dbytes + kv_write_bytes(w, esz) + (2 * len(pairs) * w.num_kv_heads * w.block_size *
                                                        w.head_dim * esz * 2))
    kv_gbs = world * step_bytes * args.steps / (total_ms / 1e3) / 1e9
    dec_avg_ms = statistics.mean(dec_ms)
    achieved = dbytes / (dec_avg_ms / 1e3) / 1e9
    peaks = measured_peaks()
    peak = peaks["hbm_gbs"] if peaks else 6800.0
    # multi-token steps: the binding roof is HBM or the tensor cores (fp16 MMA
    # at the measured bf16 rate), whichever takes longer for the call's work
    flops = causal_flops(w) if multi else None
    tpeak = (peaks.get("bf16_tflops_sustained") or peaks.get("bf16_tflops")) if peaks else 1700.0
    tensor_bound = bool(multi and flops / (tpeak * 1e12) > dbytes / (peak * 1e9))
    headline = w.name == WORKLOAD and args.seqs is None
    line = {
        "metric": METRIC,
        "value": round(tok_s, 2),
        "unit": "tokens/s",
        "n_gpus": world,
        "steps": args.steps,
        "warmup": args.warmup,
        "ms_per_step": round(total_ms / args.steps, 4),
        "higher_is_better": True,
        "scaling": "weak",
        "vs_baseline": None,
        "dtype": {"f16": "f16", "bf16": "bf16", "fp8": "fp8_e4m3 cache, f16 MMA"}[kvd],
        "data": "synthetic",
        "config": {
            "workload": describe(w, layers),
            "num_seqs": w.num_seqs, "context_len_max": int(w.context_lens.max()), "num_heads": w.num_heads,
            "num_kv_heads": w.num_kv_heads, "head_dim": w.head_dim, "block_size": w.block_size,
            "layers": layers, "parallelism": f"replicas x{world}", "kv_dtype": kvd,
            "l2": f"K/V read per layer {dbytes / 1e9:.2f} GB vs 129 MB L2; no flush",
        },
        "kv_gbs": round(kv_gbs, 1),
        "decode_ms": {"mean": round(dec_avg_ms, 5), "p10": round(float(np.percentile(dec_ms, 10)), 5),
                      "p90": round(float(np.percentile(dec_ms, 90)), 5)},
        "roofline": {
            "kernel": ("pa_attention_causal (prep, tensor-core kernels for sequences of more than 16 query "
                       "rows -- narrow for up to 32, 128-row tiles beyond -- decode pipeline beside them)"
                       if multi else
                       "pa_decode_shared_prefix (prep, shared ranges on the tensor-core kernel, own ranges and "
                       "merges on the decode kernel)" if shared_mode else
                       "pa_decode (prep + persistent partition kernel with fused log-sum-exp merge)"),
            "bound": "hbm", "achieved": round(achieved, 1), "peak": peak, "unit": "GB/s",
            "frac": round(achieved / peak, 4),
            "traffic": kernel_traffic() if headline else None,
            "algorithmic_bytes_per_launch": dbytes,
            "peak_source": "MEASURED_PEAKS.json hbm_gbs (of measured)" if peaks else "fallback 6.8 TB/s (of fallback)",
        },
        "e2e": {"value": round(job_tokens_per_s(world, B, args.steps, e2e_ms), 2), "unit": "tokens/s",
                "h2d_bytes_per_step": int(h2d), "d2h_bytes_per_step": int(d2h),
                "host_alloc_us_per_step": round(1e6 * statistics.mean(e2e_alloc_s), 1),
                "includes": "per step: host allocation (slots, copy pairs, block tables) from the history state, "
                            "host->device copies of tables, lengths, slots and every layer's query and new K/V, "
                            "the kernels, and every layer's output back to pinned host memory"},
        "graph": None if graph_ms is None else {
            "value": round(job_tokens_per_s(world, B, args.steps, graph_ms), 2), "unit": "tokens/s",
            "ms_per_step": round(graph_ms / args.steps, 4),
            "note": "the whole step captured once in a CUDA Graph and replayed"},
        # per layer: KV write, prep, decode pipeline, block copy (if pairs), the
        # tensor-core kernels (narrow, one-tile, and two-tile for 16-bit caches)
        "gpu_launches": args.steps * layers * (3 + (1 if has_pairs else 0) +
                                               ((1 + (kvd != "fp8") + narrow_launch(w, kvd))
                                                if prefill_launch(w, kvd) else 0) +
                                               (1 if shared_mode and shared_on_tensor_cores(w, kvd) else 0)),
        "alloc_us_per_step": round(alloc_us, 1),
        "clocks": clk.summary(),
    }
    if multi:
        tf = flops / (dec_avg_ms / 1e3) / 1e12
        line["roofline"]["flops_per_launch"] = flops
        line["roofline"]["achieved_tflops"] = round(tf, 1)
        line["roofline"]["tensor_peak_tflops"] = tpeak
        if tensor_bound:
            line["roofline"].update({"bound": "tensor", "achieved": round(tf, 1), "peak": tpeak, "unit": "TFLOP/s",
                                     "frac": round(tf / tpeak, 4),
                                     "peak_source": "MEASURED_PEAKS.json bf16_tflops_sustained (of measured; fp16 "
                                                    "MMA runs at the bf16 rate)" if peaks else
                                                    "fallback 1.7 PFLOP/s (of fallback)"})
        line["query_tokens_per_layer_step"] = int(w.num_new_tokens)
    if w.num_prompts:
        ub = unique_kv_bytes(w, tables, lens)
        line["roofline"]["unique_kv_bytes_per_launch"] = ub
        line["roofline"]["achieved_unique"] = round(ub / (dec_avg_ms / 1e3) / 1e9, 1)
        line["copy_pairs"] = int(len(pairs))
        line["decode_call"] = "pa_decode_shared_prefix" if shared_mode else "pa_decode"
    if headline and world == 1 and not args.no_records:
        line["workloads"] = []
        for n, kd, sh in RECORDS:
            line["workloads"].append(workload_record(n, kd, sh, pa, torch, dev))
            torch.cuda.empty_cache()
    if not args.no_cpu_baseline and world == 1 and not w.num_prompts:
        smp = OracleSample(w, tables, lens, target_s=10.0, kv_dtype=kvd)
        rate, secs = smp.rate(layers)
        line["cpu_baseline"] = {"value": round(rate, 6), "unit": "tokens/s", "cores": smp.threads, "kind": "oracle",
                                "sample": smp.describe(secs, layers)}
    print(json.dumps(line), flush=True)
    if world > 1:
        torch.distributed.barrier()
        torch.distributed.destroy_process_group()


# ------------------------------------------- the other workloads, per layer

# (workload, cache type, shared-prefix decode): the configurations timed beside
# the headline, one record each in its JSON line
RECORDS = (("mha7b", "f16", False), ("mix", "f16", False), ("cow16", "f16", False), ("cow16", "f16", True),
           ("gqa72b", "fp8", False), ("spec72b", "f16", False), ("spec72b", "fp8", False), ("chunked", "f16", False))


def workload_record(name, kvd, shared, pa, torch, dev, seconds=0.4, warmup=3):
    """One layer of a workload, timed call by call with CUDA events on the
    launching stream: block copy (copy-on-write pairs, if any), KV write and
    the attention call, each with its algorithmic bytes (and FLOPs) and the
    fraction of the measured roof; the SM clock sampled meanwhile (as many
    calls as take about `seconds`, so that the sampler sees them).  Inputs
    are larger than L2, so nothing is flushed between calls."""
    from paged_kv_cache_12_gb300 import workloads
    w = workloads.make(name)
    al, slots, pairs, tables, lens, alloc_us = allocate(w, pa)
    multi = multi_token(w)
    kpool, vpool, q1, qm, nk_h, nv_h = inputs(w, kvd)
    cache_dt = {"f16": torch.float16, "bf16": torch.bfloat16, "fp8": torch.uint8}[kvd]
    row_dt = torch.bfloat16 if kvd == "bf16" else torch.float16
    up = lambda a, dt=None: (lambda t: t.view(dt) if dt is not None else t)(
        torch.from_numpy(np.ascontiguousarray(a)).to(dev))
    k, v = up(kpool, cache_dt), up(vpool, cache_dt)
    q = up(qm if multi else q1, row_dt)
    nk, nv = up(nk_h, row_dt), up(nv_h, row_dt)
    d_slots, d_pairs, d_tables, d_lens = up(slots), up(pairs), up(tables), up(lens)
    out = torch.empty_like(q)
    ks, vs = FP8_SCALES if kvd == "fp8" else (1.0, 1.0)
    typed = kvd != "f16"
    st = torch.cuda.current_stream()
    if multi:
        d_qs = up(w.query_start)
        nws = pa.pa_attention_causal_workspace_size(w.num_seqs, w.num_new_tokens, w.num_heads, w.num_kv_heads,
                                                    w.head_dim, w.max_context_len)
    elif shared:
        S = w.samples_per_prompt
        d_lead = up(np.repeat(np.arange(w.num_prompts) * S, S).astype(np.int32))
        d_shl = torch.full((w.num_seqs,), w.prompt_len, dtype=torch.int32, device=dev)
        nws = pa.pa_decode_shared_prefix_workspace_size(w.num_seqs, w.num_heads, w.num_kv_heads, w.head_dim,
                                                        w.max_context_len)
    else:
        nws = pa.pa_decode_workspace_size(w.num_seqs, w.num_heads, w.num_kv_heads, w.head_dim, w.max_context_len)
    ws = torch.zeros(nws, dtype=torch.uint8, device=dev)

    def call():
        if multi and typed:
            pa.pa_attention_causal_typed(out, q, k, v, d_tables, d_lens, d_qs, w.scale, w.max_context_len, ws, ks, vs,
                                         st)
        elif multi:
            pa.pa_attention_causal(out, q, k, v, d_tables, d_lens, d_qs, w.scale, w.max_context_len, ws, st)
        elif typed:
            pa.pa_decode_typed(out, q, k, v, d_tables, d_lens, w.scale, w.max_context_len, ws, ks, vs, st)
        elif shared:
            pa.pa_decode_shared_prefix(out, q, k, v, d_tables, d_lens, d_lead, d_shl, w.scale, w.max_context_len, ws,
                                       st)
        else:
            pa.pa_decode(out, q, k, v, d_tables, d_lens, w.scale, w.max_context_len, ws, st)

    has_pairs = len(pairs) > 0
    E = lambda: torch.cuda.Event(enable_timing=True)

    def one(evs=None):
        if evs:
            evs[0].record(st)
        if has_pairs:
            pa.pa_block_copy(k, v, d_pairs, st)
        if evs:
            evs[1].record(st)
        if kvd == "fp8":
            pa.pa_kv_write_fp8(nk, nv, d_slots, k, v, ks, vs, st)
        else:
            pa.pa_kv_write(nk, nv, d_slots, k, v, st)
        if evs:
            evs[2].record(st)
        call()
        if evs:
            evs[3].record(st)

    t_w = time.perf_counter()
    for _ in range(warmup):
        one()
    torch.cuda.synchronize()
    per_call = (time.perf_counter() - t_w) / warmup
    calls = int(min(2000, max(20, seconds / max(per_call, 1e-6))))
    evs = [[E() for _ in range(4)] for _ in range(calls)]
    with ClockSampler(dev.index or 0) as clk:
        for e in evs:
            one(e)
        torch.cuda.synchronize()
    assert pa.pa_workspace_status(ws) == pa.PA_OK
    t_copy = [a[0].elapsed_time(a[1]) for a in evs]
    t_write = [a[1].elapsed_time(a[2]) for a in evs]
    t_call = [a[2].elapsed_time(a[3]) for a in evs]
    esz = elem_bytes(kvd)
    peaks = measured_peaks()
    peak = peaks["hbm_gbs"] if peaks else 6800.0
    tpeak = (peaks.get("bf16_tflops_sustained") or peaks.get("bf16_tflops")) if peaks else 1700.0
    dbytes = causal_bytes(w, esz) if multi else decode_bytes(w, esz)
    ms = statistics.mean(t_call)
    gbs = dbytes / (ms / 1e3) / 1e9
    call_name = ("pa_attention_causal" + ("_typed" if typed else "") if multi else
                 "pa_decode_shared_prefix" if shared else "pa_decode_typed" if typed else "pa_decode")
    rec = {"workload": name, "kv_dtype": kvd, "call": call_name, "num_seqs": w.num_seqs, "calls": calls,
           "ms": {"mean": round(ms, 5), "p10": round(float(np.percentile(t_call, 10)), 5),
                  "p90": round(float(np.percentile(t_call, 90)), 5)},
           "algorithmic_bytes": dbytes, "achieved_gbs": round(gbs, 1), "hbm_frac": round(gbs / peak, 4),
           "bound": "hbm", "frac": round(gbs / peak, 4)}
    if multi:
        flops = causal_flops(w)
        tf = flops / (ms / 1e3) / 1e12
        rec.update({"query_tokens": int(w.num_new_tokens), "flops": flops, "achieved_tflops": round(tf, 1),
                    "tensor_frac": round(tf / tpeak, 4)})
        if flops / (tpeak * 1e12) > dbytes / (peak * 1e9):
            rec.update({"bound": "tensor", "frac": round(tf / tpeak, 4)})
    if w.num_prompts:
        ub = unique_kv_bytes(w, tables, lens)
        rec.update({"unique_kv_bytes": ub, "achieved_unique_gbs": round(ub / (ms / 1e3) / 1e9, 1),
                    "frac": round(ub / (ms / 1e3) / 1e9 / peak, 4), "frac_on": "unique bytes",
                    "copy_pairs": int(len(pairs))})
    wb = kv_write_bytes(w, esz)
    rec["kv_write"] = {"ms": round(statistics.mean(t_write), 5), "algorithmic_bytes": wb,
                       "achieved_gbs": round(wb / (statistics.mean(t_write) / 1e3) / 1e9, 1)}
    if has_pairs:
        cb = 2 * len(pairs) * w.num_kv_heads * w.block_size * w.head_dim * esz * 2
        rec["block_copy"] = {"ms": round(statistics.mean(t_copy), 5), "algorithmic_bytes": cb,
                             "achieved_gbs": round(cb / (statistics.mean(t_copy) / 1e3) / 1e9, 1)}
    rec["host_alloc_us"] = round(alloc_us, 1)
    rec["clocks"] = clk.summary()
    w.drop_arrays()
    return rec


# ------------------------------------------------------------ reference arm

def run_reference(args):
    """The oracle, as it stands, on the host cores: same workload, metric and
    unit; each step times one bounded sample (the first n sequences, one
    layer, about two seconds) and scales it to the 80-layer step."""
    rank, _, world = dist_env()
    if rank != 0:
        return
    import oracle
    from paged_kv_cache_12_gb300 import workloads
    w = workloads.make(WORKLOAD)
    al = oracle.OracleAllocator(w.num_blocks, w.block_size, free_order=w.free_order)
    ids = list(range(w.num_seqs))
    for i in ids:
        al.add_seq(i)
    al.append_batch(ids, [int(x) for x in w.context_lens])
    tables, lens = al.tables(ids, w.max_blocks_per_seq)
    smp = OracleSample(w, tables, lens, target_s=2.0)
    rates, secs_list = [], []
    for i in range(args.warmup + args.steps):
        rate, secs = smp.rate()
        if i >= args.warmup:
            rates.append(rate)
            secs_list.append(secs)
    value = statistics.mean(rates)
    line = {
        "impl": "reference",
        # a step is one timed sample call (what ms_per_step x steps adds up to);
        # value is the metric of the whole 80-layer, 100-sequence step that the
        # sample stands for (see "extrapolation")
        "metric": METRIC, "value": round(value, 6), "unit": "tokens/s", "n_gpus": world, "steps": args.steps,
        "warmup": args.warmup, "ms_per_step": round(1e3 * statistics.mean(secs_list), 3),
        "extrapolation": {"sequences_per_step": smp.n, "of_sequences": w.num_seqs, "layers_per_step": 1,
                          "of_layers": LAYERS,
                          "full_step_ms": round(1e3 * w.num_seqs / value, 3),
                          "rule": "tokens/s = sequences timed / (seconds of the sample x 80 layers)"},
        "higher_is_better": True, "scaling": "weak", "vs_baseline": None, "dtype": "f64", "data": "synthetic",
        "config": {"workload": f"{WORKLOAD}: GQA 72B-shaped decode, {w.num_seqs} sequences x 8192-token context, "
                               f"64 query / 8 KV heads, head_dim 128, block 16, {LAYERS} layers per step",
                   "num_seqs": w.num_seqs, "context_len": int(w.context_lens[0]), "layers": LAYERS},
        "cpu_baseline": {"value": round(value, 6), "unit": "tokens/s", "cores": smp.threads, "kind": "oracle",
                         "sample": smp.describe(secs)},
        "e2e": {"value": round(value, 6), "unit": "tokens/s", "h2d_bytes_per_step": 0, "d2h_bytes_per_step": 0},
    }
    print(json.dumps(line), flush=True)


if __name__ == "__main__":
    a = parse()
    if a.impl == "reference":
        run_reference(a)
    else:
        run_ours(a)
