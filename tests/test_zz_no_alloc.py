"""pa_decode_static_ws: decode for callers that cannot allocate device memory.

Such callers (a plugin living inside a framework that owns all device memory
through its own pool, or a serving loop that allocates nothing after
start-up) cannot hand pa_decode a workspace, so the library offers a variant
that uses its own fixed scratch array instead.  This file checks, through the
C ABI, that calls in a row give exactly the bits pa_decode gives for the same
inputs -- also when a later call needs more partitions and merge tickets than
an earlier one left in the shared array, and when it shrinks again -- that
those bits are the oracle's attention within the decode tolerance, that the
array's error word can be read back, and that a size needing more scratch than
the array holds is refused.  It is collected last so that a failure here never
hides the other tests' results."""
import numpy as np
import pytest

import paged_kv_cache_12_gb300 as pa
from paged_kv_cache_12_gb300 import workloads
from scenario import Step, compare

torch = pytest.importorskip("torch")
pytestmark = pytest.mark.gpu

if not torch.cuda.is_available():  # pragma: no cover
    pytest.skip("no CUDA device", allow_module_level=True)


def both_outputs(w):
    """(static-array output, pa_decode output, oracle output) for one step."""
    st = Step(w)
    d = st.upload(torch)
    st.run_library(d)                       # pa_decode with a caller-provided workspace
    expect = d["out"].clone()
    got = torch.full_like(d["out"], float("nan"))
    pa.pa_decode_static_ws(got, d["q"], d["k"], d["v"], d["tables"], d["lens"], w.scale, w.max_context_len)
    torch.cuda.synchronize()
    assert pa.pa_decode_static_ws_status() == pa.PA_OK
    kc, vc = st.oracle_caches()
    return got.cpu().numpy(), expect.cpu().numpy(), st.oracle_out(kc, vc)


def check_call(w):
    got, expect, ref = both_outputs(w)
    assert np.array_equal(got.view(np.uint16), expect.view(np.uint16)), "bits differ from pa_decode"
    compare(got, ref)


def test_calls_in_a_row_match_pa_decode_bit_for_bit():
    # a small first call: one query head per kv head, few partitions
    check_call(workloads.custom(seed=42, num_seqs=9, num_heads=8, num_kv_heads=8, head_dim=64, block_size=32,
                                context_lens=[1100, 64, 4097, 5, 0, 900, 2600, 513, 1]))
    # a larger one over the dirty array: 16 query heads per kv head, more
    # sequences with more partitions each (tickets and partials of the first
    # call are still in the array where this one puts its own)
    check_call(workloads.custom(seed=41, num_seqs=12, num_heads=32, num_kv_heads=2, head_dim=128, block_size=16,
                                context_lens=[3000, 1, 700, 2049, 513, 1500, 6000, 4100, 257, 9000, 33, 2500]))
    # and a smaller one again
    check_call(workloads.custom(seed=44, num_seqs=5, num_heads=16, num_kv_heads=4, head_dim=128, block_size=8,
                                context_lens=[300, 1300, 17, 2100, 800]))


def test_too_large_is_refused():
    # valid arguments (64 query / 8 KV heads) whose workspace would exceed the array
    need = pa.pa_decode_workspace_size(4096, 64, 8, 128, 32768)
    assert need > pa.PA_DECODE_STATIC_WS_BYTES
    cache = torch.zeros((16, 8, 16, 128), dtype=torch.float16, device="cuda")
    big_q = torch.zeros((4096, 64, 128), dtype=torch.float16, device="cuda")
    big_t = torch.zeros((4096, 1), dtype=torch.int32, device="cuda")
    big_l = torch.zeros((4096,), dtype=torch.int32, device="cuda")
    with pytest.raises(pa.PAError) as e:
        pa.pa_decode_static_ws(torch.empty_like(big_q), big_q, cache, cache, big_t, big_l, 0.088, 32768)
    assert e.value.code == pa.PA_ERR_WORKSPACE
    # an unsupported shape is reported as pa_decode reports it, before the size
    cache1 = torch.zeros((16, 1, 16, 128), dtype=torch.float16, device="cuda")
    with pytest.raises(pa.PAError) as e:
        pa.pa_decode_static_ws(torch.empty_like(big_q), big_q, cache1, cache1, big_t, big_l, 0.088, 32768)
    assert e.value.code == pa.PA_ERR_UNSUPPORTED
