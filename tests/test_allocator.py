"""The library's C++ block allocator against the oracle allocator: the pages'
worked examples and random operation sequences, compared exactly (slots,
copy pairs, block tables, reference counts, free-queue effects, errors)."""
import json
import os

import numpy as np
import pytest

import paged_kv_cache_12_gb300 as pa
from oracle import OracleAllocator, OracleError

CODES = {"INVALID_ARG": pa.PA_ERR_INVALID_ARG, "OUT_OF_BLOCKS": pa.PA_ERR_OUT_OF_BLOCKS, "STATE": pa.PA_ERR_STATE}


def order_starting(first, n):
    return list(first) + [b for b in range(n) if b not in first]


def test_deeplearn_block4_example(golden_dir):
    g = json.load(open(os.path.join(golden_dir, "alloc_deeplearn_block4.json")))
    a = pa.Allocator(64, g["block_size"], free_order=order_starting(g["block_table"], 64))
    a.add_seq(0)
    s1, p1 = a.append([0], [3])
    slots = list(s1)
    for _ in range(3):
        s, p = a.append([0], [1])
        assert len(p) == 0
        slots += list(s)
    tab, lens = a.block_tables([0], 4)
    assert list(tab[0][:2]) == g["block_table"] and lens[0] == 6
    assert slots == [42 * 4, 42 * 4 + 1, 42 * 4 + 2, 42 * 4 + 3, 7 * 4, 7 * 4 + 1]
    assert 2 * 4 - 6 == g["empty_slots_paged"]
    a.free_seq(0)
    st = a.stats()
    assert st["free_blocks"] == 64 and st["used_blocks"] == 0


def test_chester_block16_example(golden_dir):
    g = json.load(open(os.path.join(golden_dir, "alloc_chester_block16.json")))
    a = pa.Allocator(32, 16, free_order=order_starting(g["block_table"], 32))
    a.add_seq(5)
    slots, pairs = a.append([5], [64])
    assert len(pairs) == 0 and slots[17] == 33 and slots[63] == 79
    assert list(a.block_tables([5], 4)[0][0]) == g["block_table"]


def run_both(ops, nb, bs, order):
    """Apply the same operations to both allocators and compare every result."""
    ref = OracleAllocator(nb, bs, free_order=order)
    dut = pa.Allocator(nb, bs, free_order=order)
    for op in ops:
        kind = op[0]
        try:
            if kind == "add":
                ref.add_seq(op[1]); r_out = None
            elif kind == "append":
                rs, rp = ref.append_batch(op[1], op[2]); r_out = (rs, rp)
            elif kind == "fork":
                ref.fork(op[1], op[2]); r_out = None
            elif kind == "free":
                ref.free_seq(op[1]); r_out = None
            r_code = pa.PA_OK
        except OracleError as e:
            r_code, r_out = CODES[e.code], None
        try:
            if kind == "add":
                dut.add_seq(op[1]); d_out = None
            elif kind == "append":
                ds, dp = dut.append(op[1], op[2]); d_out = (list(ds), [tuple(x) for x in dp])
            elif kind == "fork":
                dut.fork(op[1], op[2]); d_out = None
            elif kind == "free":
                dut.free_seq(op[1]); d_out = None
            d_code = pa.PA_OK
        except pa.PAError as e:
            d_code, d_out = e.code, None
        assert d_code == r_code, op
        assert d_out == r_out, op
        # full state after every step
        ids = sorted(ref.seqs)
        if ids:
            maxb = max(1, max(len(ref.block_table(s)) for s in ids))
            rt, rl = ref.tables(ids, maxb)
            dt, dl = dut.block_tables(ids, maxb)
            assert np.array_equal(rt, dt) and np.array_equal(rl, dl)
        for b in range(nb):
            assert dut.refcount(b) == ref.ref[b]
        assert dut.stats() == ref.stats()


@pytest.mark.parametrize("seed,bs", [(0, 4), (1, 16), (2, 8), (3, 32)])
def test_random_sequences_match_oracle(seed, bs):
    rng = np.random.default_rng(seed)
    nb = 64
    ops, live, nxt = [], [], 0
    for _ in range(250):
        k = rng.integers(0, 10)
        if k == 0 or not live:
            ops.append(("add", nxt)); live.append(nxt); nxt += 1
        elif k == 1:
            ops.append(("fork", int(rng.choice(live)), nxt)); live.append(nxt); nxt += 1
        elif k == 2 and len(live) > 1:
            s = int(rng.choice(live)); ops.append(("free", s)); live.remove(s)
        elif k == 3:
            ops.append(("free", 10_000))                    # unknown id
        else:
            m = int(rng.integers(1, min(4, len(live)) + 1))
            ids = [int(x) for x in rng.choice(live, size=m, replace=False)]
            cnts = [int(x) for x in rng.integers(0, 3 * bs, size=m)]
            if rng.integers(0, 20) == 0:
                cnts[0] = -1                                 # invalid count
            ops.append(("append", ids, cnts))
    run_both(ops, nb, bs, list(rng.permutation(nb)))


def test_cow_parallel_sampling_pairs_in_index_order():
    bs, nb = 16, 200
    order = list(np.random.default_rng(9).permutation(nb))
    ops = [("add", 100), ("append", [100], [2048 + 5])]
    ops += [("fork", 100, k) for k in range(8)] + [("free", 100)]
    ops += [("append", list(range(8)), [3] * 8)]
    run_both(ops, nb, bs, order)
    a = pa.Allocator(nb, bs, free_order=order)
    a.add_seq(100)
    a.append([100], [2053])
    for k in range(8):
        a.fork(100, k)
    a.free_seq(100)
    _, pairs = a.append(list(range(8)), [1] * 8)
    assert len(pairs) == 7 and len(set(pairs[:, 0].tolist())) == 1   # samples 0..6 copy, sample 7 writes in place


def test_errors_leave_state_unchanged():
    a = pa.Allocator(3, 4)
    a.add_seq(0)
    a.add_seq(1)
    a.append([0], [5])
    before = (a.stats(), a.block_tables([0, 1], 3))
    with pytest.raises(pa.PAError) as e:
        a.append([1, 0], [4, 4])
    assert e.value.code == pa.PA_ERR_OUT_OF_BLOCKS
    after = (a.stats(), a.block_tables([0, 1], 3))
    assert before[0] == after[0] and all(np.array_equal(x, y) for x, y in zip(before[1], after[1]))
    for call in (lambda: a.add_seq(0), lambda: a.append([7], [1]), lambda: a.append([0, 0], [1, 1]),
                 lambda: a.fork(0, 1), lambda: a.free_seq(9), lambda: a.block_tables([0], 1)):
        with pytest.raises(pa.PAError) as e:
            call()
        assert e.value.code == pa.PA_ERR_INVALID_ARG
    with pytest.raises(pa.PAError):
        pa.Allocator(4, 4, free_order=[0, 0, 1, 2])
