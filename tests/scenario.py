"""Test harness: one decode step of a workload, run through the library and
through the oracle on the same seeded bytes.

Setup (identical on both sides): the allocator hands out blocks in the
workload's free order; each sequence's history is appended (for the
parallel-sampling workloads: one prompt per group, forked to its samples, the
parent released).  Every cache slot that holds no history token is poisoned
with NaN, so a read past a context or from an unassigned block shows up in the
output.  The step then appends the new tokens (which may produce copy-on-write
pairs), copies the pairs' blocks, writes the new K/V rows and decodes.
"""
from __future__ import annotations

import numpy as np

import oracle
import paged_kv_cache_12_gb300 as pa

NAN16 = np.uint16(0x7E00)


def seq_ids_of(w):
    return list(range(w.num_seqs))


def build_allocators(w):
    """Run the workload's allocation history on both allocators, compare them,
    and return (oracle_alloc, product_alloc, used_mask_before_step)."""
    ref = oracle.OracleAllocator(w.num_blocks, w.block_size, free_order=w.free_order)
    dut = pa.Allocator(w.num_blocks, w.block_size, free_order=w.free_order)
    if w.num_prompts:
        for p in range(w.num_prompts):
            parent = 1_000_000 + p
            ref.add_seq(parent)
            dut.add_seq(parent)
            rs, _ = ref.append_tokens(parent, w.prompt_len)
            ds, _ = dut.append([parent], [w.prompt_len])
            assert list(ds) == rs
            for k in range(w.samples_per_prompt):
                child = p * w.samples_per_prompt + k
                ref.fork(parent, child)
                dut.fork(parent, child)
            ref.free_seq(parent)
            dut.free_seq(parent)
    else:
        ids = seq_ids_of(w)
        for s in ids:
            ref.add_seq(s)
            dut.add_seq(s)
        hist = [int(x) for x in w.history_lens]
        rs, rp = ref.append_batch(ids, hist)
        ds, dp = dut.append(ids, hist)
        assert list(ds) == rs and len(dp) == 0 and rp == []
    return ref, dut, ref.used_slot_mask()


def step_allocation(w, ref, dut):
    """The step's appends on both allocators: (slot_mapping, pairs), compared."""
    ids = seq_ids_of(w)
    counts = [int(x) for x in w.new_counts]
    rs, rp = ref.append_batch(ids, counts)
    ds, dp = dut.append(ids, counts)
    assert list(ds) == rs
    assert [tuple(x) for x in dp.tolist()] == [tuple(x) for x in rp]
    return np.asarray(rs, dtype=np.int64), np.asarray(rp, dtype=np.int64).reshape(-1, 2)


def poisoned_pools(w, used_mask):
    k = w.k_pool.copy()
    v = w.v_pool.copy()
    unused = ~used_mask                          # [num_blocks, block_size]
    kb = k.view(np.uint16).transpose(0, 2, 1, 3)  # [blocks, offset, heads, dim] view
    vb = v.view(np.uint16).transpose(0, 2, 1, 3)
    kb[unused] = NAN16
    vb[unused] = NAN16
    return k, v


class Step:
    """Everything one decode step needs, on the host."""

    def __init__(self, w):
        self.w = w
        self.ref, self.dut, used = build_allocators(w)
        self.k0, self.v0 = poisoned_pools(w, used)
        self.slots, self.pairs = step_allocation(w, self.ref, self.dut)
        ids = seq_ids_of(w)
        mb = w.max_blocks_per_seq
        self.tables, self.lens = self.dut.block_tables(ids, mb)
        rt, rl = self.ref.tables(ids, mb)
        assert np.array_equal(rt, self.tables) and np.array_equal(rl, self.lens)
        assert np.array_equal(self.lens, w.context_lens)

    # ---- oracle side
    def oracle_caches(self):
        kc, vc = oracle.block_copy(self.k0, self.v0, self.pairs)
        return oracle.kv_write(kc, vc, self.w.new_key, self.w.new_value, self.slots, self.w.block_size)

    def oracle_out(self, kc, vc, seq_range=None):
        w = self.w
        return oracle.paged_decode(w.query, kc, vc, self.tables, self.lens, w.num_kv_heads, w.block_size, w.scale,
                                   seq_range=seq_range)

    # ---- library side
    def upload(self, torch, device="cuda"):
        t = lambda a: torch.from_numpy(np.ascontiguousarray(a)).to(device)
        d = {
            "k": t(self.k0), "v": t(self.v0), "q": t(self.w.query),
            "nk": t(self.w.new_key), "nv": t(self.w.new_value),
            "slots": t(self.slots), "pairs": t(self.pairs),
            "tables": t(self.tables), "lens": t(self.lens),
        }
        d["out"] = torch.full_like(d["q"], float("nan"))
        nws = pa.pa_decode_workspace_size(self.w.num_seqs, self.w.num_heads, self.w.num_kv_heads, self.w.head_dim,
                                          self.w.max_context_len)
        d["ws"] = torch.zeros(nws, dtype=torch.uint8, device=device)
        return d

    def run_library(self, d):
        pa.pa_block_copy(d["k"], d["v"], d["pairs"])
        pa.pa_kv_write(d["nk"], d["nv"], d["slots"], d["k"], d["v"])
        pa.pa_decode(d["out"], d["q"], d["k"], d["v"], d["tables"], d["lens"], self.w.scale,
                     self.w.max_context_len, d["ws"])


def compare(gpu_out, ref_out, abs_tol=2e-3, rel_tol=1e-2):
    """Tolerance of the decode path: max |g - o| <= abs_tol over all elements,
    and, per (sequence, head) row, max |g - o| / max(max |o|, 1e-6) <= rel_tol
    (normwise relative error).  Returns (max_abs, max_rel) and asserts."""
    g = gpu_out.astype(np.float64)
    o = ref_out.astype(np.float64)
    assert np.isfinite(g).all(), "non-finite values in the GPU output"
    err = np.abs(g - o)
    max_abs = float(err.max()) if err.size else 0.0
    rows_err = err.reshape(-1, err.shape[-1]).max(axis=1)
    rows_ref = np.maximum(np.abs(o).reshape(-1, o.shape[-1]).max(axis=1), 1e-6)
    max_rel = float((rows_err / rows_ref).max()) if rows_err.size else 0.0
    assert max_abs <= abs_tol, f"max abs error {max_abs:.3e} > {abs_tol}"
    assert max_rel <= rel_tol, f"max normwise rel error {max_rel:.3e} > {rel_tol}"
    return max_abs, max_rel
