"""The narrow tensor-core kernel: sequences whose new tokens fill 17 to 32 query
rows (new tokens x G: speculative steps, deepsonar page section 2.5) run with
the KV tokens on the MMAs' M side, S^T = K Q^T and O^T += V^T P^T, the row
maxima reduced across the four softmax warps.  Results must be the oracle's
causal attention within the decode tolerance for every G up to 16, every
block size and cache type, contexts that end inside a KV tile or are shorter
than one, the causal mask inside the last tiles, running maxima that jump for
single rows in late tiles, and calls that mix narrow, 128-row and
decode-pipeline sequences."""
import os
import subprocess
import sys

import numpy as np
import pytest

import paged_kv_cache_12_gb300 as pa
from test_gpu_kv_dtypes import compare, as_f64
from test_gpu_prefill import run_case

torch = pytest.importorskip("torch")
pytestmark = pytest.mark.gpu

if not torch.cuda.is_available():  # pragma: no cover
    pytest.skip("no CUDA device", allow_module_level=True)

ROOT = os.path.dirname(os.path.dirname(os.path.abspath(__file__)))

# new tokens per sequence that give 17 .. 32 rows at each G
NARROW_T = {1: [17, 24, 32], 2: [9, 16], 4: [5, 8], 8: [3, 4], 16: [2]}


@pytest.mark.parametrize("kv", [pa.PA_KV_F16, pa.PA_KV_BF16, pa.PA_KV_FP8_E4M3])
@pytest.mark.parametrize("H,Hkv", [(8, 8), (16, 8), (16, 4), (64, 8), (32, 2)])
@pytest.mark.parametrize("bs", [8, 16, 32])
def test_speculative_rows_against_oracle(kv, H, Hkv, bs):
    G = H // Hkv
    ts = NARROW_T[G]
    # contexts: the whole prompt, shorter than one KV tile, one tile exactly,
    # one position more, ending inside a later tile, long; then a decode row
    # and a 128-row chunk in the same call
    lens = [ts[0], 100, 128, 129 + ts[-1], 1000 + 37, 4100]
    T = [ts[i % len(ts)] for i in range(len(lens))]
    lens, T = lens + [700, 900], T + [1, 160 // G + 1]
    w, st, out, ref = run_case(H, Hkv, bs, kv, lens, T, seed=7 * H + bs + 3 * kv + Hkv)
    compare(as_f64(out, kv), ref, kv)
    again = st.causal()
    assert torch.equal(out.view(torch.int16), again.view(torch.int16))


@pytest.mark.parametrize("kv", [pa.PA_KV_F16, pa.PA_KV_BF16, pa.PA_KV_FP8_E4M3])
def test_maximum_grows_for_single_rows_in_late_tiles(kv):
    # Keys planted at positions in KV tiles 2, 7 and 19 make single rows'
    # maxima jump by far more than 2^8 there (rows of different warps' lanes
    # after the transposed reduction), while the other rows keep theirs: O^T
    # is rescaled column by column, unchanged rows by exactly 1.
    H, Hkv, bs = 64, 8, 16
    lens, T = [2600, 1000, 2500], [4, 3, 4]
    plants = [(0, 300, 1, 9, 2.0), (0, 900, 3, 62, 2.0), (0, 2500, 0, 0, 2.0), (1, 990, 2, 17, 2.0),
              (2, 2400, 3, 40, 2.0), (2, 260, 0, 41, 2.0)]
    w, st, out, ref = run_case(H, Hkv, bs, kv, lens, T, seed=61 + kv, plants=plants)
    compare(as_f64(out, kv), ref, kv)


def test_many_items_per_cta_of_varying_lengths():
    # 240 sequences x 8 kv heads = 1920 work items over the persistent grid,
    # contexts from 4 to 1500 positions
    rng = np.random.default_rng(5)
    lens = [int(x) for x in rng.integers(4, 1500, size=240)]
    T = [4] * 240
    w, st, out, ref = run_case(64, 8, 16, pa.PA_KV_F16, lens, T, seed=77)
    compare(as_f64(out, pa.PA_KV_F16), ref, pa.PA_KV_F16)


def test_equal_within_the_bar_to_the_128_row_kernel(tmp_path):
    # the same call with the narrow kernel switched off (PA_NARROW=0, read once
    # per process): the 128-row kernel's result, also within the bar
    H, Hkv, bs = 64, 8, 16
    lens, T = [900, 2500, 64, 4097], [4, 4, 3, 4]
    w, st, out, ref = run_case(H, Hkv, bs, pa.PA_KV_F16, lens, T, seed=13)
    compare(as_f64(out, pa.PA_KV_F16), ref, pa.PA_KV_F16)
    np.save(tmp_path / "narrow.npy", out.cpu().numpy())
    code = f"""
import sys, numpy as np
sys.path.insert(0, {ROOT!r}); sys.path.insert(0, {os.path.join(ROOT, 'tests')!r})
import test_gpu_prefill as t
import paged_kv_cache_12_gb300 as pa
w, st, out, ref = t.run_case({H}, {Hkv}, {bs}, pa.PA_KV_F16, {lens}, {T}, seed=13)
t.compare(t.as_f64(out, pa.PA_KV_F16), ref, pa.PA_KV_F16)
nw = np.load({str(tmp_path / 'narrow.npy')!r}).astype(np.float64)
assert np.max(np.abs(nw - out.cpu().numpy().astype(np.float64))) <= 2e-3
"""
    env = dict(os.environ, PA_NARROW="0")
    r = subprocess.run([sys.executable, "-c", code], env=env, capture_output=True, text=True, timeout=600)
    assert r.returncode == 0, r.stdout + r.stderr


@pytest.mark.parametrize("kv", [pa.PA_KV_F16, pa.PA_KV_FP8_E4M3])
@pytest.mark.parametrize("nseq,lens", [(4, [5000, 3000, 9000, 700]), (9, [2000 + 300 * i for i in range(9)]),
                                       (20, [1000 + 40 * i for i in range(20)])])
def test_split_last_round_against_oracle(kv, nseq, lens):
    # The last, partial round of (sequence, kv head) items is split into pieces
    # of their KV ranges so that it fills the grid (4 x 8 items on 152 SMs: 4
    # pieces each; 9 x 8: 2 pieces; 20 x 8: one full round, then 8 items in 7
    # pieces, the most their 14 KV tiles allow); the CTA that completes an
    # item's last piece merges the pieces.  Results stay the oracle's and repeat
    # bit for bit.  (Pools small enough that the fp8 cache is the oracle's
    # quantisation of N(0, 1) data, whose outputs the absolute bar is made for.)
    T = [4] * nseq
    w, st, out, ref = run_case(64, 8, 16, kv, lens, T, seed=90 + nseq + kv)
    compare(as_f64(out, kv), ref, kv)
    again = st.causal()
    assert torch.equal(out.view(torch.int16), again.view(torch.int16))


def test_out_of_range_block_in_one_piece_of_a_split_item():
    # an out-of-range id in the middle of sequence 0's range: the piece that
    # meets it carries NaN into the merge, so every row of sequence 0 is NaN;
    # the other sequences (also split) are the oracle's
    lens = [5000, 3000, 9000, 700]
    w, st, out, ref = run_case(64, 8, 16, pa.PA_KV_F16, lens, [4] * 4, seed=95)
    compare(as_f64(out, pa.PA_KV_F16), ref, pa.PA_KV_F16)
    bad = st.d["tables"].clone()
    bad[0, 150] = w.num_blocks + 3          # position 2400
    st.d["tables"] = bad
    out2 = st.causal().cpu().numpy()
    qs = w.query_start
    assert np.isnan(out2[qs[0]:qs[1]]).all()
    compare(out2[qs[1]:].astype(np.float64), ref[qs[1]:], pa.PA_KV_F16)
