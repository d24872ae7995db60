"""Pins for the oracle's block allocator: the pages' worked examples and the
invariants they state.  CPU only."""
import json
import os

import numpy as np
import pytest

from oracle import OracleAllocator, OracleError


def order_starting(first, num_blocks):
    rest = [b for b in range(num_blocks) if b not in first]
    return list(first) + rest


def test_deeplearn_block4_example(golden_dir):
    g = json.load(open(os.path.join(golden_dir, "alloc_deeplearn_block4.json")))
    bs = g["block_size"]
    a = OracleAllocator(64, bs, free_order=order_starting(g["block_table"], 64))
    a.add_seq(0)
    counts = []
    slots, pairs = a.append_tokens(0, len(g["prompt_tokens"]))
    counts.append(len(a.block_table(0)))
    for _ in g["generated_tokens"]:
        s, p = a.append_tokens(0, 1)
        slots += s
        pairs += p
        counts.append(len(a.block_table(0)))
    assert counts == [g["blocks_after_prompt"], g["blocks_after_nice"], g["blocks_after_today"],
                      g["blocks_after_bang"]]
    assert a.block_table(0) == g["block_table"]
    assert pairs == []
    b0, b1 = g["block_table"]
    assert slots == [b0 * bs + 0, b0 * bs + 1, b0 * bs + 2, b0 * bs + 3, b1 * bs + 0, b1 * bs + 1]
    # where each token sits, as the page's table prints it
    tokens = g["prompt_tokens"] + g["generated_tokens"]
    for blk, content in zip(g["block_table"], g["block_contents"]):
        for off, tok in enumerate(content):
            if tok is not None:
                assert slots[tokens.index(tok)] == blk * bs + off
    empty = len(a.block_table(0)) * bs - a.seq_len(0)
    assert empty == g["empty_slots_paged"]
    assert g["traditional_reserved_tokens"] - g["traditional_used_tokens"] == g["traditional_wasted_tokens"]
    # release returns everything
    a.free_seq(0)
    assert a.stats()["free_blocks"] == 64 and all(r == 0 for r in a.ref)


def test_chester_block16_example(golden_dir):
    g = json.load(open(os.path.join(golden_dir, "alloc_chester_block16.json")))
    bs = g["block_size"]
    a = OracleAllocator(32, bs, free_order=order_starting(g["block_table"], 32))
    a.add_seq("A")
    slots, pairs = a.append_tokens("A", g["tokens"])
    assert a.block_table("A") == g["block_table"] and pairs == []
    for lb, (t0, t1) in enumerate(g["logical_ranges"]):
        for t in range(t0, t1 + 1):
            assert slots[t] == g["block_table"][lb] * bs + (t - t0)
    assert slots[17] == 33 and slots[63] == 79


def test_waste_at_most_one_block_and_release():
    rng = np.random.default_rng(3)
    bs, nb = 8, 400
    a = OracleAllocator(nb, bs, free_order=rng.permutation(nb))
    live = []
    for step in range(300):
        op = rng.integers(0, 4)
        if op == 0 or not live:
            sid = step
            a.add_seq(sid)
            live.append(sid)
        elif op == 3 and len(live) > 1:
            sid = live.pop(int(rng.integers(len(live))))
            a.free_seq(sid)
        else:
            sid = live[int(rng.integers(len(live)))]
            try:
                a.append_tokens(sid, int(rng.integers(0, 20)))
            except OracleError as e:
                assert e.code == "OUT_OF_BLOCKS"
        for s in live:
            assert len(a.block_table(s)) == -(-a.seq_len(s) // bs)
    for s in live:
        a.free_seq(s)
    assert a.stats()["free_blocks"] == nb and sum(a.ref) == 0


def test_free_queue_head_out_tail_in():
    a = OracleAllocator(6, 2, free_order=[5, 4, 3, 2, 1, 0])
    a.add_seq(0)
    a.add_seq(1)
    a.append_tokens(0, 3)          # blocks 5, 4
    a.append_tokens(1, 1)          # block 3
    a.free_seq(0)                  # 5 then 4 go to the tail: queue = 2, 1, 0, 5, 4
    assert list(a.free) == [2, 1, 0, 5, 4]
    a.append_tokens(1, 4)          # fills block 3, then takes 2 and 1
    assert a.block_table(1) == [3, 2, 1]


def test_copy_on_write_rules():
    bs = 4
    a = OracleAllocator(16, bs)
    a.add_seq("p")
    a.append_tokens("p", 6)                      # blocks 0 (full), 1 (2 of 4)
    for c in range(3):
        a.fork("p", c)
    a.free_seq("p")
    assert a.ref[0] == 3 and a.ref[1] == 3
    # first writer onto the shared partial tail copies it
    s, p = a.append_tokens(0, 1)
    assert p == [(1, 2)] and a.block_table(0) == [0, 2] and s == [2 * bs + 2]
    assert a.ref[1] == 2 and a.ref[2] == 1
    s, p = a.append_tokens(1, 2)
    assert p == [(1, 3)] and s == [3 * bs + 2, 3 * bs + 3]
    # the last holder finds count 1 and writes in place
    s, p = a.append_tokens(2, 1)
    assert p == [] and s == [1 * bs + 2] and a.ref[1] == 1
    # the full shared block 0 is never copied: the next token starts a new block
    s, p = a.append_tokens(0, 2)
    assert p == [] and a.block_table(0)[0] == 0 and a.ref[0] == 3


def test_whole_block_prompt_needs_no_copy():
    bs = 16
    a = OracleAllocator(64, bs)
    a.add_seq("p")
    a.append_tokens("p", 32)
    for c in range(8):
        a.fork("p", c)
    a.free_seq("p")
    _, pairs = a.append_batch(list(range(8)), [1] * 8)
    assert pairs == []


def test_out_of_blocks_leaves_state_unchanged():
    a = OracleAllocator(3, 4)
    a.add_seq(0)
    a.add_seq(1)
    a.append_tokens(0, 5)
    before = (list(a.free), list(a.ref), {k: (v["len"], list(v["blocks"])) for k, v in a.seqs.items()})
    with pytest.raises(OracleError) as e:
        a.append_batch([1, 0], [4, 4])            # needs 1 + 1 blocks, one is free
    assert e.value.code == "OUT_OF_BLOCKS"
    after = (list(a.free), list(a.ref), {k: (v["len"], list(v["blocks"])) for k, v in a.seqs.items()})
    assert before == after


def test_bad_arguments():
    a = OracleAllocator(4, 4)
    a.add_seq(0)
    for call in (lambda: a.add_seq(0), lambda: a.append_tokens(9, 1), lambda: a.append_tokens(0, -1),
                 lambda: a.fork(9, 1), lambda: a.fork(0, 0), lambda: a.free_seq(9),
                 lambda: a.append_batch([0, 0], [1, 1])):
        with pytest.raises(OracleError) as e:
            call()
        assert e.value.code == "INVALID_ARG"
    with pytest.raises(OracleError):
        OracleAllocator(4, 4, free_order=[0, 1, 1, 2])
