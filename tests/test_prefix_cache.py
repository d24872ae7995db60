"""Prefix caching in the block allocator (deepsonar.com.cn page, section 2.4
and section VII step 5): chained block hashes, a hash -> block map, the free
queue as eviction order, prefix matching with the last prompt token always
recomputed.  CPU only."""
import hashlib

import numpy as np
import pytest

import paged_kv_cache_12_gb300 as pa
from oracle import OracleAllocator, OracleError, block_hash, ZERO_HASH

CODES = {"INVALID_ARG": pa.PA_ERR_INVALID_ARG, "OUT_OF_BLOCKS": pa.PA_ERR_OUT_OF_BLOCKS, "STATE": pa.PA_ERR_STATE}


# ------------------------------------------------------------------ SHA-256

def test_sha256_standard_examples():
    # the worked examples of the Secure Hash Standard (FIPS 180-2, appendix B)
    assert pa.pa_sha256(b"abc").hex() == "ba7816bf8f01cfea414140de5dae2223b00361a396177a9cb410ff61f20015ad"
    assert pa.pa_sha256(b"").hex() == "e3b0c44298fc1c149afbf4c8996fb92427ae41e4649b934ca495991b7852b855"
    msg = b"abcdbcdecdefdefgefghfghighijhijkijkljklmklmnlmnomnopnopq"
    assert pa.pa_sha256(msg).hex() == "248d6a61d20638b8e5c026930c3e6039a33ce45964ff2167f6ecedd419db06c1"


def test_sha256_every_padding_boundary():
    rng = np.random.default_rng(0)
    for n in list(range(0, 200)) + [511, 512, 513, 4096 + 55]:
        data = rng.integers(0, 256, size=n, dtype=np.uint8).tobytes()
        assert pa.pa_sha256(data) == hashlib.sha256(data).digest(), n


# ------------------------------------------------------- oracle semantics

def prompt(n, seed=0):
    return [int(x) for x in np.random.default_rng(seed).integers(0, 50000, size=n)]


def test_hit_miss_and_chain_divergence():
    bs = 4
    a = OracleAllocator(64, bs, prefix_cache=True)
    p = prompt(13)                               # 3 full blocks + 1 token
    assert a.match_prefix(0, p) == 0             # cold cache: the first lookup misses, matching stops
    a.append_batch([0], [13], p)
    assert a.prefix_stats()["cached_blocks"] == 3
    # the same prompt again: the 3 full blocks hit and are shared
    assert a.match_prefix(1, p) == 12
    assert a.block_table(1) == a.block_table(0)[:3]
    assert all(a.ref[b] == 2 for b in a.block_table(0)[:3])
    # one different token in block 1: block 0 hits, the chain breaks at block 1
    q = list(p)
    q[5] += 1
    assert a.match_prefix(2, q) == 4
    # a different extra key (e.g. another adapter) shares nothing
    assert a.match_prefix(3, p, extra_key=7) == 0
    st = a.prefix_stats()
    assert st["queries"] == 1 + 3 + 2 + 1 and st["hits"] == 3 + 1


def test_last_prompt_token_is_always_computed():
    bs = 4
    a = OracleAllocator(32, bs, prefix_cache=True)
    p = prompt(8, 1)                             # exactly two full blocks
    a.match_prefix(0, p)
    a.append_batch([0], [8], p)
    assert a.prefix_stats()["cached_blocks"] == 2
    # both blocks are cached, but the last token must be computed: only block 0 hits
    assert a.match_prefix(1, p) == 4
    # a longer prompt with the same two blocks reuses both
    assert a.match_prefix(2, p + [9]) == 8


def test_free_queue_is_the_eviction_order():
    bs = 2
    a = OracleAllocator(6, bs, free_order=[0, 1, 2, 3, 4, 5], prefix_cache=True)
    p = prompt(4, 2)
    a.match_prefix(0, p)
    a.append_batch([0], [4], p)                 # blocks 0, 1 cached
    a.free_seq(0)                               # both back at the tail: queue 2 3 4 5 0 1
    assert list(a.free) == [2, 3, 4, 5, 0, 1]
    # a hit on a free cached block takes it out of the middle of the queue
    assert a.match_prefix(1, p + [1]) == 4
    assert list(a.free) == [2, 3, 4, 5]
    a.free_seq(1)
    assert list(a.free) == [2, 3, 4, 5, 0, 1]
    # new work takes blocks from the head; reaching block 0 evicts its content
    a.add_seq(2)
    a.append_batch([2], [10])                   # blocks 2 3 4 5 0: block 0 reused
    assert 0 not in a.hash_of and a.prefix_stats()["cached_blocks"] == 1
    # block 1 is still cached but its parent's is gone: the chain misses at block 0
    assert a.match_prefix(3, p + [1]) == 0


def test_prefix_cache_must_be_on_and_ids_are_needed():
    a = OracleAllocator(8, 4)
    with pytest.raises(OracleError):
        a.match_prefix(0, prompt(9))
    b = OracleAllocator(8, 4, prefix_cache=True)
    b.add_seq(0)
    b.append_batch([0], [8])                    # no ids: nothing is hashed
    assert b.prefix_stats()["cached_blocks"] == 0


# ------------------------------------------------- library vs the oracle

def compare_state(ref, dut):
    ids = sorted(ref.seqs)
    if ids:
        maxb = max(1, max(len(ref.block_table(s)) for s in ids))
        rt, rl = ref.tables(ids, maxb)
        dt, dl = dut.block_tables(ids, maxb)
        assert np.array_equal(rt, dt) and np.array_equal(rl, dl)
    assert dut.free_queue() == list(ref.free)
    for b in range(ref.num_blocks):
        assert dut.refcount(b) == ref.ref[b]
        h, cached = dut.block_hash(b)
        if b in ref.hash_of:
            assert h == ref.hash_of[b] and cached == (ref.cached.get(ref.hash_of[b]) == b)
        else:
            assert h == bytes(32) and not cached
    assert dut.stats() == ref.stats()
    assert dut.prefix_stats() == ref.prefix_stats()


@pytest.mark.parametrize("seed,bs", [(3, 2), (4, 4), (5, 8), (6, 16)])
def test_library_matches_oracle_mixed_operations(seed, bs):
    rng = np.random.default_rng(seed)
    nb = 40
    order = list(rng.permutation(nb))
    ref = OracleAllocator(nb, bs, free_order=order, prefix_cache=True)
    dut = pa.Allocator(nb, bs, free_order=order, prefix_cache=True)
    bases = [prompt(int(rng.integers(bs, 5 * bs)), seed * 10 + k) for k in range(3)]
    live, nxt = [], 0
    for _ in range(250):
        op = int(rng.integers(0, 8))
        removed = None
        if op <= 1 or not live:
            toks = bases[int(rng.integers(0, 3))] + prompt(int(rng.integers(0, 2 * bs)), int(rng.integers(1 << 30)))
            extra = int(rng.integers(0, 2))
            sid = nxt

            def start(alloc, append):
                # a new request: reuse the cached prefix, then append the rest of the prompt
                c = alloc.match_prefix(sid, toks, extra)
                out = append(alloc, [sid], [len(toks) - c], toks[c:])
                return c, out

            calls = (lambda: start(ref, lambda al, i, n, t: al.append_batch(i, n, t)),
                     lambda: start(dut, lambda al, i, n, t: al.append_ids(i, n, t)))
            new = nxt
            nxt += 1
        elif op == 2:
            par = int(rng.choice(live))
            calls = (lambda: ref.fork(par, nxt), lambda: dut.fork(par, nxt))
            new = nxt
            nxt += 1
        elif op == 3 and len(live) > 1:
            s = int(rng.choice(live))
            calls = (lambda: ref.free_seq(s), lambda: dut.free_seq(s))
            new = None
            removed = s
        else:
            m = int(rng.integers(1, min(3, len(live)) + 1))
            ids = [int(x) for x in rng.choice(live, size=m, replace=False)]
            cnts = [int(x) for x in rng.integers(0, 3 * bs, size=m)]
            if rng.integers(0, 4):
                toks = prompt(sum(cnts), int(rng.integers(1 << 30)))
                calls = (lambda: ref.append_batch(ids, cnts, toks), lambda: dut.append_ids(ids, cnts, toks))
            else:
                calls = (lambda: ref.append_batch(ids, cnts), lambda: dut.append(ids, cnts))
            new = None
        try:
            r = calls[0]()
            rc = pa.PA_OK
        except OracleError as e:
            r, rc = None, CODES[e.code]
        try:
            d = calls[1]()
            d_rc = pa.PA_OK
        except pa.PAError as e:
            d, d_rc = None, e.code
        assert d_rc == rc
        if isinstance(r, tuple) and len(r) == 2 and isinstance(r[0], int):   # (cached tokens, append result)
            assert d[0] == r[0]
            r, d = r[1], d[1]
        if isinstance(r, tuple):      # (slots, pairs) from an append
            assert list(d[0]) == r[0] and [tuple(x) for x in d[1].tolist()] == [tuple(x) for x in r[1]]
        if rc == pa.PA_OK:
            if new is not None:
                live.append(new)
            if removed is not None:
                live.remove(removed)
        compare_state(ref, dut)
    hits = ref.prefix_stats()["hits"]
    assert hits > 10, hits            # the shared prompts were actually reused


def test_library_refuses_match_without_prefix_cache():
    a = pa.Allocator(8, 4)
    with pytest.raises(pa.PAError) as e:
        a.match_prefix(0, prompt(9))
    assert e.value.code == pa.PA_ERR_INVALID_ARG
    b = pa.Allocator(8, 4)
    b.add_seq(0)                                # only before any sequence exists
    assert pa.lib().pa_alloc_enable_prefix_cache(b._h) == pa.PA_ERR_INVALID_ARG
