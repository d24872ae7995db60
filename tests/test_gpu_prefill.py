"""The tensor-core kernel for long runs of new tokens (prompt chunks; deepsonar
page section 2.5): a sequence whose new tokens x G exceed 16 query rows is
computed in 128-row tiles with tcgen05 MMAs.  Results must be the oracle's
causal attention within the decode tolerance, for every G that divides the
tile, every block size, fp16, bf16 and FP8 E4M3 caches (FP8 codes are turned
into exact fp16 tiles on chip), chunks after long histories
(many KV tiles, running-maximum rescales), whole prompts, partial row tiles and
contexts that end inside a KV tile (the V rows past them are poisoned NaN)."""
import os
import subprocess
import sys

import numpy as np
import pytest

import oracle
import paged_kv_cache_12_gb300 as pa
from paged_kv_cache_12_gb300 import workloads
from test_gpu_kv_dtypes import KS, TypedStep, compare, as_f64, to_bf16_bits

torch = pytest.importorskip("torch")
pytestmark = pytest.mark.gpu

if not torch.cuda.is_available():  # pragma: no cover
    pytest.skip("no CUDA device", allow_module_level=True)

ROOT = os.path.dirname(os.path.dirname(os.path.abspath(__file__)))


def encode(x, kv):
    """fp64 values -> cache elements of type kv (fp8: the oracle's quantiser)."""
    if kv == pa.PA_KV_FP8_E4M3:
        return oracle.fp8_quantise(np.asarray(x, dtype=np.float64), KS)
    if kv == pa.PA_KV_BF16:
        return to_bf16_bits(x)
    return np.asarray(x, dtype=np.float16).view(np.uint16)


def plant_keys(st, plants):
    """Overwrite history keys: plants = [(seq, position, new token j, query head
    h, factor)] makes K at `position` of `seq` (kv head h // G) `factor` times
    the query row of new token j, head h, so that row's score there stands far
    above every other it sees."""
    w = st.w
    G = w.num_heads // w.num_kv_heads
    for seq, pos, j, h, f in plants:
        q = st.qm[w.query_start[seq] + j, h]
        qv = (q.astype(np.uint32) << 16).view(np.float32) if st.kv == pa.PA_KV_BF16 else q
        blk = st.tables[seq][pos // w.block_size]
        st.k0[blk, h // G, pos % w.block_size] = encode(f * np.asarray(qv, dtype=np.float64), st.kv)


def run_case(H, Hkv, bs, kv, lens, T, seed, plants=()):
    w = workloads.custom(seed=seed, num_seqs=len(lens), num_heads=H, num_kv_heads=Hkv, head_dim=128, block_size=bs,
                         context_lens=lens, new_tokens=T, multi=True)
    st = TypedStep(w, kv)
    plant_keys(st, plants)
    st.run_gpu()
    kc, vc = st.oracle_caches()
    out = st.causal()
    ref = oracle.paged_attention_typed(st.qm, kc, vc, st.tables, st.lens, w.query_start, Hkv, bs, w.scale, kv,
                                       *st.scales())
    return w, st, out, ref


@pytest.mark.parametrize("kv", [pa.PA_KV_F16, pa.PA_KV_BF16, pa.PA_KV_FP8_E4M3])
@pytest.mark.parametrize("H,Hkv", [(8, 8), (16, 8), (32, 8), (64, 8), (16, 1)])
@pytest.mark.parametrize("bs", [8, 16, 32])
def test_prompt_chunks_against_oracle(kv, H, Hkv, bs):
    G = H // Hkv
    # a whole prompt, chunks after a history (ending inside a KV tile), a
    # chunk of exactly one row tile, one with a partial last tile, and short
    # requests that stay on the decode pipeline in the same call
    tpt = 128 // G
    lens = [300, 1000 + 37, 700, 2 * tpt + 513, 5, 4000]
    T = [300, 200, tpt, 2 * tpt + 3, 2, 129]
    w, st, out, ref = run_case(H, Hkv, bs, kv, lens, T, seed=11 * H + bs + kv)
    compare(as_f64(out, kv), ref, kv)


def test_long_history_many_kv_tiles():
    # 16k positions before a 256-token chunk: 130 KV tiles of 128 tokens per
    # row tile (the running maximum grows a little, below the 2^8 rescale
    # threshold; test_running_maximum_grows_for_some_rows_of_a_warp crosses it)
    w, st, out, ref = run_case(32, 8, 16, pa.PA_KV_F16, [16384 + 256], [256], seed=5)
    compare(as_f64(out, pa.PA_KV_F16), ref, pa.PA_KV_F16)


@pytest.mark.parametrize("kv", [pa.PA_KV_F16, pa.PA_KV_BF16, pa.PA_KV_FP8_E4M3])
def test_running_maximum_grows_for_some_rows_of_a_warp(kv):
    # Keys planted in later KV tiles (positions 300, 1000, 1700, 2500) make the
    # running maximum of single query rows jump by far more than 2^8 after the
    # first tile, while the other rows of the same 32-row warp keep theirs:
    # the rescale of O in tensor memory must run for the whole warp, with
    # unchanged rows scaled by exactly 1.  With N(0, 1) data alone the maximum
    # never moves that far after the first tile.
    H, Hkv, bs = 32, 8, 16
    lens, T = [3000, 2600], [256, 40]
    plants = [(0, 300, 3, 1, 2.0), (0, 1000, 40, 6, 2.0), (0, 1700, 100, 9, 2.0), (1, 2500, 7, 30, 2.0),
              (1, 1000, 20, 5, 2.0)]
    w, st, out, ref = run_case(H, Hkv, bs, kv, lens, T, seed=41 + kv, plants=plants)
    compare(as_f64(out, kv), ref, kv)
    again = st.causal()
    assert torch.equal(out.view(torch.int16), again.view(torch.int16))


@pytest.mark.parametrize("kv", [pa.PA_KV_F16, pa.PA_KV_FP8_E4M3])
def test_several_items_per_cta_with_out_of_range_ids(kv):
    # 48 sequences x 4 new tokens at G = 8: 384 work items, so every CTA of the
    # persistent grid runs two or three, one behind the other; the producers
    # read ahead into the next item.  Three of every four sequences meet an
    # out-of-range block id: their rows are NaN, every other row is the oracle's.
    # (Contexts short enough that the fp8 pool is the oracle's quantisation of
    # N(0, 1) data, whose outputs the absolute bar is made for.)
    H, Hkv, bs = 64, 8, 16
    lens = [300 + 7 * i for i in range(48)]
    T = [4] * 48
    w, st, out, ref = run_case(H, Hkv, bs, kv, lens, T, seed=57 + kv)
    compare(as_f64(out, kv), ref, kv)
    bad = st.d["tables"].clone()
    for i in range(48):
        if i % 4 != 3:
            bad[i, (lens[i] // bs) // 2] = w.num_blocks + i
    st.d["tables"] = bad
    out2 = st.causal().cpu().numpy()
    qs = w.query_start
    for i in range(48):
        rows = out2[qs[i]:qs[i + 1]]
        if i % 4 != 3:
            assert np.isnan(rows).all(), f"sequence {i}"
        else:
            compare(rows.astype(np.float64), ref[qs[i]:qs[i + 1]], kv)


def test_deterministic_and_equal_to_the_decode_pipeline(tmp_path):
    H, Hkv, bs = 32, 8, 16
    lens, T = [900, 2500, 64], [300, 500, 16]
    w, st, out, ref = run_case(H, Hkv, bs, pa.PA_KV_F16, lens, T, seed=3)
    again = st.causal()
    assert torch.equal(out.view(torch.int16), again.view(torch.int16))
    # the same call with the tensor-core kernel switched off (PA_PREFILL=0, read
    # once per process): the decode pipeline's result, also within the bar
    np.save(tmp_path / "tc.npy", out.cpu().numpy())
    code = f"""
import sys, numpy as np
sys.path.insert(0, {ROOT!r}); sys.path.insert(0, {os.path.join(ROOT, 'tests')!r})
import test_gpu_prefill as t
import paged_kv_cache_12_gb300 as pa
w, st, out, ref = t.run_case({H}, {Hkv}, {bs}, pa.PA_KV_F16, {lens}, {T}, seed=3)
t.compare(t.as_f64(out, pa.PA_KV_F16), ref, pa.PA_KV_F16)
tc = np.load({str(tmp_path / 'tc.npy')!r}).astype(np.float64)
assert np.max(np.abs(tc - out.cpu().numpy().astype(np.float64))) <= 2e-3
"""
    env = dict(os.environ, PA_PREFILL="0")
    r = subprocess.run([sys.executable, "-c", code], env=env, capture_output=True, text=True, timeout=600)
    assert r.returncode == 0, r.stdout + r.stderr


@pytest.mark.parametrize("kv", [pa.PA_KV_F16, pa.PA_KV_BF16, pa.PA_KV_FP8_E4M3])
def test_long_ranges_of_mixed_lengths_against_oracle(kv):
    # Row tiles of very different KV lengths in one call, at G = 8: a chunk
    # after a 4000-token history (200 new tokens), a short chunk after 8936
    # positions (71 KV tiles), a whole 4200-token prompt (row tiles reading
    # 1 .. 33 KV tiles) and a decode row.
    lens, T = [4200, 9000, 3], [200, 64, 1]
    if kv == pa.PA_KV_F16:
        lens, T = lens + [4200], T + [4200]
    w, st, out, ref = run_case(8, 1, 16, kv, lens, T, seed=31 + kv)
    compare(as_f64(out, kv), ref, kv)
    again = st.causal()
    assert torch.equal(out.view(torch.int16), again.view(torch.int16))


def test_out_of_range_block_id_deep_in_a_long_range():
    # a bad id met 37 KV tiles into a 71-tile range: every row of that
    # sequence is NaN, the other sequence is untouched
    H, Hkv, bs = 16, 2, 16
    lens, T = [9000, 300], [64, 40]
    w, st, out, ref = run_case(H, Hkv, bs, pa.PA_KV_F16, lens, T, seed=23)
    compare(as_f64(out, pa.PA_KV_F16), ref, pa.PA_KV_F16)
    bad = st.d["tables"].clone()
    bad[0, 300] = w.num_blocks + 9          # position 4800
    st.d["tables"] = bad
    out2 = st.causal().cpu().numpy()
    qs = w.query_start
    assert np.isnan(out2[qs[0]:qs[1]]).all()
    compare(out2[qs[1]:qs[2]].astype(np.float64), ref[qs[1]:qs[2]], pa.PA_KV_F16)


def test_out_of_range_block_id_gives_nan_rows_of_that_sequence_only():
    H, Hkv, bs = 32, 8, 16
    lens, T = [900, 1200, 700], [300, 256, 40]
    w, st, out, ref = run_case(H, Hkv, bs, pa.PA_KV_F16, lens, T, seed=21)
    compare(as_f64(out, pa.PA_KV_F16), ref, pa.PA_KV_F16)
    bad = st.d["tables"].clone()
    bad[1, 0] = w.num_blocks + 5          # never read: the tiles that meet it write NaN
    st.d["tables"] = bad
    out2 = st.causal().cpu().numpy()
    qs = w.query_start
    assert np.isnan(out2[qs[1]:qs[2]]).all()
    keep = np.r_[qs[0]:qs[1], qs[2]:qs[3]]
    compare(out2[keep].astype(np.float64), ref[keep], pa.PA_KV_F16)


def test_graph_capture_of_a_mixed_call():
    # a prompt chunk (tensor-core kernel) and decode rows (decode pipeline) in one
    # call, captured once in a CUDA Graph: replays give the eager bits, also after
    # new query rows are copied into the captured buffer
    H, Hkv, bs = 32, 8, 16
    lens, T = [1500, 300, 64, 2000], [500, 1, 1, 3]
    w = workloads.custom(seed=8, num_seqs=len(lens), num_heads=H, num_kv_heads=Hkv, head_dim=128, block_size=bs,
                         context_lens=lens, new_tokens=T, multi=True)
    st = TypedStep(w, pa.PA_KV_F16)
    st.run_gpu()
    d = st.d
    qs = torch.from_numpy(w.query_start).cuda()
    out = torch.empty_like(d["qm"])
    ws = torch.zeros(pa.pa_attention_causal_workspace_size(w.num_seqs, w.num_new_tokens, H, Hkv, 128,
                                                           w.max_context_len), dtype=torch.uint8, device="cuda")

    def call(stream=None):
        pa.pa_attention_causal(out, d["qm"], d["k"], d["v"], d["tables"], d["lens"], qs, w.scale, w.max_context_len,
                               ws, stream)

    call()                                     # first call: one-time set-up outside the capture
    torch.cuda.synchronize()
    eager = out.clone()
    s = torch.cuda.Stream()
    s.wait_stream(torch.cuda.current_stream())
    g = torch.cuda.CUDAGraph()
    with torch.cuda.stream(s):
        with torch.cuda.graph(g, stream=s):
            call(s)
    torch.cuda.current_stream().wait_stream(s)
    out.zero_()
    g.replay()
    torch.cuda.synchronize()
    assert torch.equal(out.view(torch.int16), eager.view(torch.int16))
    d["qm"].copy_(torch.flip(d["qm"], dims=[0]))
    call()
    torch.cuda.synchronize()
    eager2 = out.clone()
    out.zero_()
    g.replay()
    torch.cuda.synchronize()
    assert torch.equal(out.view(torch.int16), eager2.view(torch.int16))
    assert not torch.equal(eager2.view(torch.int16), eager.view(torch.int16))
