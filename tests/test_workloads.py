"""The seeded input generator: determinism and the workload structure."""
import numpy as np

from paged_kv_cache_12_gb300 import workloads


def test_deterministic_and_independent_streams():
    a = workloads.make("tiny")
    b = workloads.make("tiny")
    assert np.array_equal(a.query, b.query) and np.array_equal(a.k_pool, b.k_pool)
    assert np.array_equal(a.free_order, b.free_order)
    assert not np.array_equal(a.k_pool, a.v_pool)
    # drawing one array does not move another's stream
    c = workloads.make("tiny")
    _ = c.v_pool
    assert np.array_equal(c.k_pool, a.k_pool)


def test_shapes_and_ranges():
    t = workloads.make("tiny")
    assert (t.num_seqs, t.num_heads, t.num_kv_heads, t.head_dim, t.block_size, t.num_blocks) == (4, 4, 2, 64, 16, 64)
    assert t.context_lens.min() >= 1 and t.context_lens.max() <= 100
    assert sorted(t.free_order.tolist()) == list(range(64))
    m = workloads.make("mha7b")
    assert m.context_lens.min() >= 512 and m.context_lens.max() <= 2048 and m.group == 1
    g = workloads.make("gqa72b")
    assert (g.context_lens == 8192).all() and g.group == 8 and g.num_blocks == 100 * 512 + 100
    x = workloads.make("mix")
    assert list(x.context_lens[:3]) == [600, 12000, 18000]
    assert x.context_lens.min() >= 64 and x.context_lens.max() <= 32768
    assert (x.new_counts == 1).all()
    for name, bs in (("cow16", 16), ("cow32", 32)):
        c = workloads.make(name)
        assert c.block_size == bs and 1 <= c.prompt_len - 2048 <= bs - 1
        assert (c.context_lens == c.prompt_len + c.divergent + 1).all()
        assert c.divergent.min() >= 0 and c.divergent.max() <= 512
        c0 = workloads.make(name, prompt_extra=0)
        assert c0.prompt_len == 2048
    s = workloads.make("spec72b")
    assert (s.new_counts == 4).all() and (s.context_lens == 8192).all() and s.group == 8 and s.multi
    assert list(s.query_start[:3]) == [0, 4, 8] and s.query_start[-1] == 400
    c = workloads.make("chunked")
    assert list(c.context_lens[:2]) == [12000, 600] and list(c.new_counts[:2]) == [2048, 600]
    assert (c.new_counts[2:] == 1).all() and c.num_new_tokens == 2048 + 600 + 62
    assert c.query_start[-1] == c.num_new_tokens and c.query_start[2] == 2648 and c.multi
    # the parallel-sampling steps append private tokens but decode one query per sequence
    assert not workloads.make("cow16").multi and not workloads.make("gqa72b").multi


def test_multi_token_query_rows():
    w = workloads.custom(seed=3, num_seqs=3, num_heads=4, num_kv_heads=2, head_dim=64, context_lens=[10, 5, 7],
                         new_tokens=[3, 0, 7])
    assert list(w.history_lens) == [7, 5, 0] and list(w.query_start) == [0, 3, 3, 10]
    assert w.query_multi.shape == (10, 4, 64) and w.query_multi.dtype == np.float16
    assert not np.array_equal(w.query_multi[:3], w.query[:3].reshape(3, 4, 64))


def test_values_are_rounded_standard_normal():
    t = workloads.make("mha7b")
    q = t.query.astype(np.float64)
    assert t.query.dtype == np.float16 and abs(q.mean()) < 0.01 and abs(q.std() - 1) < 0.01
