"""pa_attention_causal: a step in which sequences compute several new tokens
at once (a prompt chunk, or speculative candidates: deepsonar.com.cn page
section 2.5), each new token attending causally over the paged cache.  The
result must be the oracle's fp64 causal attention within the decode
tolerance, deterministic, and -- with one token per sequence -- the decode."""
import numpy as np
import pytest

import oracle
import paged_kv_cache_12_gb300 as pa
from paged_kv_cache_12_gb300 import workloads
from scenario import Step, compare

torch = pytest.importorskip("torch")
pytestmark = pytest.mark.gpu

if not torch.cuda.is_available():  # pragma: no cover
    pytest.skip("no CUDA device", allow_module_level=True)


def t(a):
    return torch.from_numpy(np.ascontiguousarray(a)).cuda()


def prepare(w):
    """Allocation history, the step's appends, block copies and KV writes."""
    st = Step(w)
    d = st.upload(torch)
    pa.pa_block_copy(d["k"], d["v"], d["pairs"])
    pa.pa_kv_write(d["nk"], d["nv"], d["slots"], d["k"], d["v"])
    d["qm"] = t(w.query_multi)
    d["qs"] = t(w.query_start)
    return st, d


def run_causal(w, d, qs=None, lens=None):
    nq = d["qm"].shape[0]
    out = torch.full_like(d["qm"], float("nan"))
    ws = torch.zeros(pa.pa_attention_causal_workspace_size(w.num_seqs, nq, w.num_heads, w.num_kv_heads, w.head_dim,
                                                           w.max_context_len), dtype=torch.uint8, device="cuda")
    pa.pa_attention_causal(out, d["qm"], d["k"], d["v"], d["tables"], d["lens"] if lens is None else lens,
                           d["qs"] if qs is None else qs, w.scale, w.max_context_len, ws)
    torch.cuda.synchronize()
    assert pa.pa_workspace_status(ws) == pa.PA_OK
    return out


def oracle_rows(st, w, kc, vc, seqs=None):
    """The oracle's causal attention for the given sequences (all by default):
    returns (rows, expected) with rows the query rows those sequences own."""
    qs = w.query_start
    seqs = range(w.num_seqs) if seqs is None else seqs
    rows = np.concatenate([np.arange(qs[i], qs[i + 1]) for i in seqs]).astype(np.int64)
    sub_qs = np.concatenate([[0], np.cumsum([qs[i + 1] - qs[i] for i in seqs])]).astype(np.int32)
    idx = np.asarray(list(seqs))
    ref = oracle.paged_attention_causal(w.query_multi[rows], kc, vc, st.tables[idx], st.lens[idx], sub_qs,
                                        w.num_kv_heads, w.block_size, w.scale)
    return rows, ref


@pytest.mark.parametrize("D", [64, 128])
@pytest.mark.parametrize("bs", [8, 16, 32])
@pytest.mark.parametrize("H,Hkv", [(8, 8), (8, 2), (64, 8), (16, 1), (12, 1)])
def test_ragged_chunks_against_oracle(D, bs, H, Hkv):
    # T = L (a whole prompt), T = 1 (decode), chunks crossing partition and
    # block boundaries, a sequence with no new token
    lens = [1, 5, 17, 40, 300, 1024, 1030, 2100, 700]
    T = [1, 5, 3, 16, 7, 1, 20, 150, 0]
    w = workloads.custom(seed=5 * D + bs + H, num_seqs=len(lens), num_heads=H, num_kv_heads=Hkv, head_dim=D,
                         block_size=bs, context_lens=lens, new_tokens=T)
    st, d = prepare(w)
    out = run_causal(w, d)
    kc, vc = st.oracle_caches()
    rows, ref = oracle_rows(st, w, kc, vc)
    assert np.array_equal(rows, np.arange(w.num_new_tokens))
    compare(out.cpu().numpy(), ref)
    again = run_causal(w, d)
    assert torch.equal(out.view(torch.int16), again.view(torch.int16))


@pytest.mark.parametrize("H,Hkv", [(8, 8), (32, 8), (64, 8)])
def test_one_token_per_sequence_is_the_decode(H, Hkv):
    lens = [1, 16, 100, 513, 1500, 3000, 2049]
    w = workloads.custom(seed=H, num_seqs=len(lens), num_heads=H, num_kv_heads=Hkv, head_dim=128, block_size=16,
                         context_lens=lens)
    st, d = prepare(w)
    d["qm"] = d["q"]                              # one query row per sequence: the decode's queries
    out = run_causal(w, d)
    pa.pa_decode(d["out"], d["q"], d["k"], d["v"], d["tables"], d["lens"], w.scale, w.max_context_len, d["ws"])
    torch.cuda.synchronize()
    kc, vc = st.oracle_caches()
    ref = st.oracle_out(kc, vc)
    compare(out.cpu().numpy(), ref)
    compare(out.cpu().numpy(), d["out"].cpu().numpy().astype(np.float64))


def test_rows_are_causal():
    # changing the K/V of the last new token changes only the last row's output
    lens, T = [300], [6]
    w = workloads.custom(seed=9, num_seqs=1, num_heads=16, num_kv_heads=2, head_dim=128, block_size=16,
                         context_lens=lens, new_tokens=T)
    st, d = prepare(w)
    before = run_causal(w, d)
    last_slot = int(st.slots[-1])
    blk, off = divmod(last_slot, w.block_size)
    d["k"][blk, :, off, :] += 1.0
    d["v"][blk, :, off, :] -= 2.0
    after = run_causal(w, d)
    assert torch.equal(before[:5].view(torch.int16), after[:5].view(torch.int16))
    assert not torch.equal(before[5], after[5])


def test_invalid_sequences_give_nan_rows():
    lens = [50, 40, 30]
    T = [3, 4, 2]
    w = workloads.custom(seed=4, num_seqs=3, num_heads=8, num_kv_heads=2, head_dim=64, block_size=16,
                         context_lens=lens, new_tokens=T)
    st, d = prepare(w)
    kc, vc = st.oracle_caches()
    _, ref = oracle_rows(st, w, kc, vc)
    # sequence 1 claims more new tokens than positions: its rows are NaN, the others are right
    bad = d["lens"].clone()
    bad[1] = 3
    out = run_causal(w, d, lens=bad).cpu().numpy()
    assert np.isnan(out[3:7]).all()
    compare(out[:3], ref[:3])
    compare(out[7:], ref[7:])
    # a query_start that does not cover the rows: every row is NaN
    for qs in ([0, 3, 7, 8], [0, 5, 4, 9], [1, 3, 7, 9]):
        out = run_causal(w, d, qs=t(np.asarray(qs, dtype=np.int32))).cpu().numpy()
        assert np.isnan(out).all(), qs


@pytest.mark.slow
def test_speculative_workload_sampled():
    w = workloads.make("spec72b")
    st, d = prepare(w)
    out = run_causal(w, d).cpu().numpy()
    assert np.isfinite(out).all()
    kc, vc = st.oracle_caches()
    seqs = [0, 37, 99]
    rows, ref = oracle_rows(st, w, kc, vc, seqs)
    compare(out[rows], ref)


@pytest.mark.slow
def test_chunked_prefill_workload_sampled():
    w = workloads.make("chunked")
    st, d = prepare(w)
    out = run_causal(w, d).cpu().numpy()
    assert np.isfinite(out).all()
    kc, vc = st.oracle_caches()
    # the 600-token prompt and some decode sequences in full
    rows, ref = oracle_rows(st, w, kc, vc, [1, 2, 30, 63])
    compare(out[rows], ref)
    # rows of the 2048-token chunk: row j sees L - T + j + 1 positions, which is
    # the decode of a sequence that long over the same block table
    L, T = int(w.context_lens[0]), int(w.new_counts[0])
    js = np.array([0, 1, 15, 16, 17, 1000, 2046, 2047])
    vis = (L - T + js + 1).astype(np.int32)
    ref0 = oracle.paged_decode(w.query_multi[js], kc, vc, np.repeat(st.tables[:1], len(js), axis=0), vis,
                               w.num_kv_heads, w.block_size, w.scale)
    compare(out[js], ref0)
