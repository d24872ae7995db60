"""The test harness's allocation flow on CPU: both allocators agree through
the workloads' setup and step, and the copy-on-write counts follow the
parallel-sampling reading (a whole-block prompt needs no copy; a partial tail
block is copied by samples 0..6 and written in place by sample 7)."""
import numpy as np
import pytest

from paged_kv_cache_12_gb300 import workloads
from scenario import Step, build_allocators, compare, step_allocation


@pytest.mark.parametrize("name,extra,pairs", [("cow16", 0, 0), ("cow16", None, 7 * 32), ("cow32", 0, 0),
                                              ("cow32", None, 7 * 32)])
def test_cow_step_pairs(name, extra, pairs):
    w = workloads.make(name, prompt_extra=extra)
    ref, dut, used = build_allocators(w)
    assert ref.stats()["shared_blocks"] == 32 * (-(-w.prompt_len // w.block_size))
    slots, prs = step_allocation(w, ref, dut)
    assert len(prs) == pairs and len(slots) == w.num_new_tokens
    # every sample ends with ceil(len / bs) blocks
    for s in range(w.num_seqs):
        assert len(ref.block_table(s)) == -(-int(w.context_lens[s]) // w.block_size)


def test_tiny_step_oracle_roundtrip():
    w = workloads.make("tiny")
    st = Step(w)
    kc, vc = st.oracle_caches()
    out = st.oracle_out(kc, vc)
    assert np.isfinite(out).all()
    # the poisoned slots are exactly the ones no token uses after the step
    used = st.ref.used_slot_mask()
    kb = kc.view(np.uint16).transpose(0, 2, 1, 3)
    assert (kb[~used] == 0x7E00).all() and not (kb[used] == 0x7E00).any()
    compare(out.astype(np.float16), out)
