"""CUDA Graph capture of the decode step, the debug-validation mode and
out-of-range block ids.

The pages say the engine captures its whole decode step in one CUDA Graph to
remove launch overhead ("PagedAttention de vLLM", deepsonar.com.cn, section
2.6).  The library's calls allow that: they never synchronise, read context
lengths on the device and size everything from host-side bounds, so a graph
captured once replays correctly for new lengths up to the captured bound."""
import os
import subprocess
import sys
import textwrap

import numpy as np
import pytest

import paged_kv_cache_12_gb300 as pa
from paged_kv_cache_12_gb300 import workloads
from scenario import Step, compare

torch = pytest.importorskip("torch")
pytestmark = pytest.mark.gpu

if not torch.cuda.is_available():  # pragma: no cover
    pytest.skip("no CUDA device", allow_module_level=True)

ROOT = os.path.dirname(os.path.dirname(os.path.abspath(__file__)))


def test_graph_replay_matches_eager_bits():
    layers = 3
    w = workloads.make("cow16")                 # block copies, multi-token writes, multi-partition decode
    st = Step(w)
    d = st.upload(torch)
    kc0, vc0 = d["k"].clone(), d["v"].clone()
    outs = [torch.empty_like(d["q"]) for _ in range(layers)]

    def step():
        for l in range(layers):
            pa.pa_block_copy(d["k"], d["v"], d["pairs"])
            pa.pa_kv_write(d["nk"], d["nv"], d["slots"], d["k"], d["v"])
            pa.pa_decode(outs[l], d["q"], d["k"], d["v"], d["tables"], d["lens"], w.scale, w.max_context_len,
                         d["ws"])

    # eager reference
    step()
    torch.cuda.synchronize()
    eager = [o.clone() for o in outs]
    compare(eager[0].cpu().numpy(), st.oracle_out(*st.oracle_caches()))

    # capture (after the warm-up call above), replay from a fresh cache
    s = torch.cuda.Stream()
    s.wait_stream(torch.cuda.current_stream())
    g = torch.cuda.CUDAGraph()
    with torch.cuda.stream(s):
        with torch.cuda.graph(g, stream=s):
            step()
    torch.cuda.current_stream().wait_stream(s)
    d["k"].copy_(kc0)
    d["v"].copy_(vc0)
    for o in outs:
        o.fill_(float("nan"))
    g.replay()
    torch.cuda.synchronize()
    for a, b in zip(eager, outs):
        assert torch.equal(a.view(torch.int16), b.view(torch.int16))

    # new step contents in the same buffers: shorter contexts, new queries
    lens2 = (d["lens"] - torch.arange(w.num_seqs, device="cuda", dtype=torch.int32) % 7).clamp_min(1)
    q2 = torch.randn_like(d["q"].float()).half()
    d["lens"].copy_(lens2)
    d["q"].copy_(q2)
    g.replay()
    torch.cuda.synchronize()
    got = [o.clone() for o in outs]
    d["k"].copy_(kc0)
    d["v"].copy_(vc0)
    step()
    torch.cuda.synchronize()
    for a, b in zip(got, outs):
        assert torch.equal(a.view(torch.int16), b.view(torch.int16))


def test_out_of_range_block_ids_give_nan_not_reads():
    w = workloads.custom(seed=51, num_seqs=4, num_heads=8, num_kv_heads=2, head_dim=128, block_size=16,
                         context_lens=[40, 1500, 700, 33])
    st = Step(w)
    d = st.upload(torch)
    st.run_library(d)
    torch.cuda.synchronize()
    good = d["out"].clone()
    tables = d["tables"].clone()
    tables[1, 50] = w.num_blocks + 1000         # inside sequence 1's context (1500 tokens = 94 blocks)
    tables[2, 0] = -5
    pa.pa_decode(d["out"], d["q"], d["k"], d["v"], tables, d["lens"], w.scale, w.max_context_len, d["ws"])
    torch.cuda.synchronize()
    out = d["out"].float()
    assert torch.isnan(out[1]).all() and torch.isnan(out[2]).all()
    assert torch.equal(out[0], good[0].float()) and torch.equal(out[3], good[3].float())
    assert pa.pa_workspace_status(d["ws"]) == pa.PA_OK


def test_debug_validation_mode_reports_bad_indices():
    code = textwrap.dedent("""
        import sys, torch
        sys.path.insert(0, %r)
        import paged_kv_cache_12_gb300 as pa
        dev = "cuda"
        k = torch.zeros((8, 2, 16, 64), dtype=torch.float16, device=dev)
        v = torch.zeros_like(k)
        key = torch.zeros((3, 2, 64), dtype=torch.float16, device=dev)
        codes = []
        def rc(f):
            try:
                f()
                return 0
            except pa.PAError as e:
                return e.code
        slots_dup = torch.tensor([5, 9, 5], dtype=torch.int64, device=dev)
        slots_oob = torch.tensor([5, 9, 8 * 16], dtype=torch.int64, device=dev)
        slots_ok = torch.tensor([5, -1, 9], dtype=torch.int64, device=dev)
        codes.append(rc(lambda: pa.pa_kv_write(key, key, slots_dup, k, v)))
        codes.append(rc(lambda: pa.pa_kv_write(key, key, slots_oob, k, v)))
        codes.append(rc(lambda: pa.pa_kv_write(key, key, slots_ok, k, v)))
        pairs_conflict = torch.tensor([[1, 2], [2, 3]], dtype=torch.int64, device=dev)
        pairs_dupdst = torch.tensor([[1, 3], [2, 3]], dtype=torch.int64, device=dev)
        pairs_ok = torch.tensor([[1, 3], [1, 4]], dtype=torch.int64, device=dev)
        codes.append(rc(lambda: pa.pa_block_copy(k, v, pairs_conflict)))
        codes.append(rc(lambda: pa.pa_block_copy(k, v, pairs_dupdst)))
        codes.append(rc(lambda: pa.pa_block_copy(k, v, pairs_ok)))
        q = torch.zeros((2, 4, 64), dtype=torch.float16, device=dev)
        out = torch.empty_like(q)
        ws = torch.zeros(pa.pa_decode_workspace_size(2, 4, 2, 64, 32), dtype=torch.uint8, device=dev)
        lens = torch.tensor([20, 3], dtype=torch.int32, device=dev)
        tab_bad = torch.tensor([[0, 9], [1, 2]], dtype=torch.int32, device=dev)
        tab_ok = torch.tensor([[0, 4], [1, 2]], dtype=torch.int32, device=dev)
        codes.append(rc(lambda: pa.pa_decode(out, q, k, v, tab_bad, lens, 0.125, 32, ws)))
        codes.append(rc(lambda: pa.pa_decode(out, q, k, v, tab_ok, lens, 0.125, 32, ws)))
        # shared prefix: two sequences claim to share 16 tokens; their first blocks differ
        lead = torch.tensor([0, 0], dtype=torch.int32, device=dev)
        shl = torch.tensor([16, 0], dtype=torch.int32, device=dev)
        ws2 = torch.zeros(pa.pa_decode_shared_prefix_workspace_size(2, 4, 2, 64, 32), dtype=torch.uint8, device=dev)
        tab_same = torch.tensor([[0, 4], [0, 2]], dtype=torch.int32, device=dev)
        lens2 = torch.tensor([20, 18], dtype=torch.int32, device=dev)
        codes.append(rc(lambda: pa.pa_decode_shared_prefix(out, q, k, v, tab_ok, lens2, lead, shl, 0.125, 32, ws2)))
        codes.append(rc(lambda: pa.pa_decode_shared_prefix(out, q, k, v, tab_same, lens2, lead, shl, 0.125, 32, ws2)))
        print(" ".join(map(str, codes)))
    """ % ROOT)
    env = dict(os.environ, PA_DEBUG_VALIDATE="1")
    res = subprocess.run([sys.executable, "-c", code], capture_output=True, text=True, env=env, timeout=300)
    assert res.returncode == 0, res.stderr
    codes = [int(x) for x in res.stdout.split()]
    E = pa.PA_ERR_INVALID_ARG
    assert codes == [E, E, 0, E, E, 0, E, 0, E, 0]


def test_bounded_wait_gives_up_and_context_survives():
    """The decode pipeline's waits are bounded.  The self-test runs that same
    bounded wait on a barrier nothing completes: it must give up, report
    PA_ERR_TIMEOUT, and leave the context usable -- no fault and no hang."""
    import time
    status = torch.full((1,), 12345, dtype=torch.int32, device="cuda")
    t0 = time.time()
    pa.pa_selftest_wait_timeout(2_000_000, status)      # ~1 ms at 2 GHz
    torch.cuda.synchronize()
    assert int(status.item()) == pa.PA_ERR_TIMEOUT and time.time() - t0 < 10
    # the context works on: a decode afterwards is correct and reports no error
    w = workloads.make("tiny")
    st = Step(w)
    d = st.upload(torch)
    st.run_library(d)
    torch.cuda.synchronize()
    assert pa.pa_workspace_status(d["ws"]) == pa.PA_OK
    compare(d["out"].cpu().numpy(), st.oracle_out(*st.oracle_caches()))
