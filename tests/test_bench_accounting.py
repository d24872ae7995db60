"""The algorithmic bytes and FLOPs that bench.py divides by its CUDA-event
times (roofline.achieved), checked against counts made another way: bytes by
walking every sequence's tokens and the block-table entries they need, FLOPs
by counting, row by row, the positions each new token sees (the causal rule:
new token j of a sequence with L positions, the last T new, sees the first
L - T + j + 1).  No GPU and no pool values are needed: the workloads draw
their pools only when asked."""
import numpy as np
import pytest

import bench
from paged_kv_cache_12_gb300 import workloads


def walked_bytes(w, esz, rows_per_seq):
    """K and V rows of every token each sequence attends, the block-table
    entries those tokens live in, the query and output rows, and the lengths
    (plus the query offsets for a multi-token call)."""
    kv = tables = 0
    for L in w.context_lens.tolist():
        tokens = np.arange(L)
        kv += tokens.size * 2 * w.num_kv_heads * w.head_dim * esz
        tables += np.unique(tokens // w.block_size).size * 4
    rows = int(sum(rows_per_seq))
    qo = 2 * rows * w.num_heads * w.head_dim * 2
    ints = 4 * w.num_seqs + (4 * (w.num_seqs + 1) if w.multi else 0)
    return kv + tables + qo + ints


@pytest.mark.parametrize("name", ["tiny", "mha7b", "gqa72b", "mix", "cow16"])
@pytest.mark.parametrize("esz", [2, 1])
def test_decode_bytes_walked(name, esz):
    w = workloads.make(name)
    assert bench.decode_bytes(w, esz) == walked_bytes(w, esz, [1] * w.num_seqs)


def test_headline_bytes_as_quoted():
    # the figure the headline roofline and its ncu traffic ratio are quoted against
    assert bench.decode_bytes(workloads.make("gqa72b")) == 3_358_925_200


@pytest.mark.parametrize("name,spec", [("spec72b", 4), ("spec72b", 3), ("spec72b", 8), ("chunked", 4)])
@pytest.mark.parametrize("esz", [2, 1])
def test_causal_bytes_walked(name, spec, esz):
    w = workloads.make(name, spec_tokens=spec)
    assert bench.causal_bytes(w, esz) == walked_bytes(w, esz, w.new_counts.tolist())


@pytest.mark.parametrize("name,spec", [("spec72b", 4), ("spec72b", 3), ("chunked", 4)])
def test_causal_flops_row_by_row(name, spec):
    w = workloads.make(name, spec_tokens=spec)
    seen = 0
    for L, T in zip(w.context_lens.tolist(), w.new_counts.tolist()):
        for j in range(T):
            seen += L - T + j + 1
    # Q K^T and P V: 2 flops per multiply-add each, per query head and dim
    assert bench.causal_flops(w) == 4 * seen * w.num_heads * w.head_dim
