"""pa_decode_shared_prefix: decode where groups of sequences share the blocks
of a common prefix (parallel sampling over one prompt, deepsonar.com.cn
page section 2.3).  The result must be the same attention as the oracle's
(and pa_decode's) within the decode tolerance, and deterministic."""
import numpy as np
import pytest

import oracle
import paged_kv_cache_12_gb300 as pa
from paged_kv_cache_12_gb300 import workloads
from scenario import Step, compare, poisoned_pools

torch = pytest.importorskip("torch")
pytestmark = pytest.mark.gpu

if not torch.cuda.is_available():  # pragma: no cover
    pytest.skip("no CUDA device", allow_module_level=True)


def run_shared(d, w, leader, shared):
    t = lambda a: torch.from_numpy(np.ascontiguousarray(a, dtype=np.int32)).cuda()
    out = torch.full_like(d["q"], float("nan"))
    ws = torch.zeros(pa.pa_decode_shared_prefix_workspace_size(w.num_seqs, w.num_heads, w.num_kv_heads, w.head_dim,
                                                               w.max_context_len), dtype=torch.uint8, device="cuda")
    pa.pa_decode_shared_prefix(out, d["q"], d["k"], d["v"], d["tables"], d["lens"], t(leader), t(shared), w.scale,
                               w.max_context_len, ws)
    torch.cuda.synchronize()
    assert pa.pa_workspace_status(ws) == pa.PA_OK
    return out


@pytest.mark.parametrize("name,extra", [("cow16", None), ("cow16", 0), ("cow32", None)])
def test_parallel_sampling_groups(name, extra):
    w = workloads.make(name, prompt_extra=extra)
    st = Step(w)
    d = st.upload(torch)
    st.run_library(d)                       # block copies, KV writes, plain decode
    torch.cuda.synchronize()
    plain = d["out"].clone()
    S = w.samples_per_prompt
    leader = np.repeat(np.arange(w.num_prompts) * S, S)
    shared = np.full(w.num_seqs, w.prompt_len)
    out = run_shared(d, w, leader, shared)
    kc, vc = st.oracle_caches()
    compare(out.cpu().numpy(), st.oracle_out(kc, vc))
    compare(out.cpu().numpy(), plain.cpu().numpy().astype(np.float64))
    again = run_shared(d, w, leader, shared)
    assert torch.equal(out.view(torch.int16), again.view(torch.int16))


def grouped(seed, sizes, prefix_lens, H, Hkv, D, bs, max_private=300):
    """Groups of forked sequences: group k has sizes[k] members sharing a
    prefix of prefix_lens[k] tokens, then each member's own tokens and this
    step's token.  Both allocators run in lockstep."""
    rng = np.random.default_rng(seed)
    own = [int(rng.integers(0, max_private)) for _ in range(sum(sizes))]
    lens = []
    k = 0
    for sz, pl in zip(sizes, prefix_lens):
        for _ in range(sz):
            lens.append(pl + own[k] + 1)
            k += 1
    nb = sum(-(-pl // bs) for pl in prefix_lens) + sum(-(-(o + 1) // bs) + 1 for o in own) + 8
    w = workloads.custom(seed=seed, num_seqs=len(lens), num_heads=H, num_kv_heads=Hkv, head_dim=D, block_size=bs,
                         context_lens=lens, num_blocks=nb)
    ref = oracle.OracleAllocator(nb, bs, free_order=w.free_order)
    dut = pa.Allocator(nb, bs, free_order=w.free_order)
    leader, shared = [], []
    sid = 0
    for g, (sz, pl) in enumerate(zip(sizes, prefix_lens)):
        parent = 10_000 + g
        for al in (ref, dut):
            al.add_seq(parent)
        ref.append_tokens(parent, pl)
        dut.append([parent], [pl])
        for m in range(sz):
            ref.fork(parent, sid + m)
            dut.fork(parent, sid + m)
            leader.append(sid)
            shared.append(pl)
        ref.free_seq(parent)
        dut.free_seq(parent)
        sid += sz
    ids = list(range(len(lens)))
    ref.append_batch(ids, own)
    dut.append(ids, own)
    used = ref.used_slot_mask()
    rs, rp = ref.append_batch(ids, [1] * len(ids))
    ds, dp = dut.append(ids, [1] * len(ids))
    assert list(ds) == rs and [tuple(x) for x in dp.tolist()] == rp
    tables, tl = dut.block_tables(ids, w.max_blocks_per_seq)
    k0, v0 = poisoned_pools(w, used)
    t = lambda a: torch.from_numpy(np.ascontiguousarray(a)).cuda()
    d = {"k": t(k0), "v": t(v0), "q": t(w.query), "tables": t(tables), "lens": t(tl)}
    pairs = np.asarray(rp, dtype=np.int64).reshape(-1, 2)
    pa.pa_block_copy(d["k"], d["v"], t(pairs))
    pa.pa_kv_write(t(w.new_key), t(w.new_value), t(np.asarray(ds)), d["k"], d["v"])
    kc, vc = oracle.block_copy(k0, v0, pairs)
    kc, vc = oracle.kv_write(kc, vc, w.new_key, w.new_value, np.asarray(rs), bs)
    expect = oracle.paged_decode(w.query, kc, vc, tables, tl, Hkv, bs, w.scale)
    return w, d, np.asarray(leader), np.asarray(shared), expect


@pytest.mark.parametrize("H,Hkv,D,bs", [(8, 8, 128, 16), (16, 4, 128, 16), (32, 4, 64, 8), (16, 2, 128, 32),
                                        (16, 1, 128, 16)])
def test_mixed_groups(H, Hkv, D, bs):
    sizes = [1, 5, 2, 12, 1, 3, 8]
    prefix = [700, 1030, 17, 2100, 40, 513, 1536]
    w, d, leader, shared, expect = grouped(H * 7 + bs, sizes, prefix, H, Hkv, D, bs)
    out = run_shared(d, w, leader, shared)
    compare(out.cpu().numpy(), expect)


def test_member_outside_its_leaders_run_shares_nothing():
    sizes = [4, 4]
    prefix = [900, 600]
    w, d, leader, shared, expect = grouped(5, sizes, prefix, 16, 4, 128, 16)
    # member 1 names itself: leader 0's run is just {0}, and members 2 and 3,
    # which still name 0, are outside it; they all decode without sharing
    leader = leader.copy()
    leader[1] = 1
    out = run_shared(d, w, leader, shared)
    compare(out.cpu().numpy(), expect)


def test_out_of_range_block_in_a_shared_range():
    # an id past the pool in the shared blocks of the 12-member group (every
    # member's table, as sharing requires): that group's rows are NaN, the
    # other groups' rows are the oracle's
    sizes = [3, 12, 5]
    prefix = [900, 2100, 513]
    w, d, leader, shared, expect = grouped(77, sizes, prefix, 32, 8, 128, 16)
    bad = d["tables"].clone()
    g0, g1 = 3, 15                            # members 3 .. 14
    bad[g0:g1, 70] = w.num_blocks + 3        # positions 1120 .. 1135 of the 2100 shared
    d["tables"] = bad
    out = run_shared(d, w, leader, shared).cpu().numpy()
    assert np.isnan(out[g0:g1]).all()
    keep = np.r_[0:g0, g1:w.num_seqs]
    compare(out[keep].astype(np.float64), expect[keep])
