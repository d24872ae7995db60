"""Register budgets of the kernels that split their registers between
warpgroups (setmaxnreg).

Such a kernel is launched with threads x R registers per CTA.  Its warpgroups
then lower and raise their per-thread counts, and the shares must add up to no
more than that pool, or a raising warpgroup would wait forever.  The host
refuses at run time a kernel whose compiled count is not the R its split was
sized for.  This test checks the same at build time, from the counts ptxas
reports (-Xptxas -v), for every split kernel.  It also checks that the
single-token decode kernels spill nothing: their consumers were given the
producers' registers for that purpose.  It needs nvcc but no GPU."""
import os
import re
import shutil
import subprocess
import tempfile
from concurrent.futures import ThreadPoolExecutor

import pytest

from paged_kv_cache_12_gb300 import build as B

NVCC = None
try:
    NVCC = B.nvcc()
except RuntimeError:  # pragma: no cover
    pass

pytestmark = pytest.mark.skipif(NVCC is None, reason="nvcc not available")

UNITS = ("decode.cu", "decode_bf16.cu", "decode_fp8.cu", "prefill.cu")


def ptxas_report(unit: str, out_dir: str) -> dict:
    """{mangled kernel name: (registers, spill store bytes, spill load bytes)}"""
    cmd = [NVCC, *B.ARCH, "-O3", "-std=c++17", "-Xptxas", "-v", "-I", B.INCLUDE, "-I", B.CSRC, "-c",
           os.path.join(B.CSRC, unit), "-o", os.path.join(out_dir, unit + ".o")]
    res = subprocess.run(cmd, capture_output=True, text=True)
    assert res.returncode == 0, res.stderr
    kernels, name, spills = {}, None, (0, 0)
    for line in res.stderr.splitlines():
        m = re.search(r"Function properties for (\S+)", line)
        if m:
            name = m.group(1)
            continue
        m = re.search(r"(\d+) bytes spill stores, (\d+) bytes spill loads", line)
        if m and name:
            spills = (int(m.group(1)), int(m.group(2)))
            continue
        m = re.search(r"Used (\d+) registers", line)
        if m and name:
            kernels[name] = (int(m.group(1)),) + spills
            name, spills = None, (0, 0)
    return kernels


@pytest.fixture(scope="module")
def reports():
    out = tempfile.mkdtemp(prefix="pa_regs_")
    try:
        with ThreadPoolExecutor(max_workers=len(UNITS)) as ex:
            got = dict(zip(UNITS, ex.map(lambda u: ptxas_report(u, out), UNITS)))
    finally:
        shutil.rmtree(out, ignore_errors=True)
    return got


def find(kernels: dict, pattern: str) -> list:
    hits = [(k, v) for k, v in kernels.items() if re.search(pattern, k)]
    assert hits, f"no kernel matching {pattern}"
    return hits


@pytest.mark.parametrize("unit", ["decode.cu", "decode_bf16.cu", "decode_fp8.cu"])
def test_single_token_decode_split(unit, reports):
    # decode_kernel<128, 1, false, KV>: 256 threads, two CTAs per SM, so 128
    # registers a thread at launch; producers 80 + consumers 176 = 2 x 128
    for name, (regs, st, ld) in find(reports[unit], r"decode_kernelILi128ELi1ELb0ELi\dE"):
        assert regs == 128, (name, regs)
        assert st == 0 and ld == 0, (name, st, ld)


def test_two_tile_prefill_split(reports):
    # prefill2_kernel<KV>: 384 threads, one CTA per SM: 168 at launch, split
    # 128 x 104 (producer warpgroup) + 256 x 200 (softmax) = 64,512 = 384 x 168
    for name, (regs, _, _) in find(reports["prefill.cu"], r"prefill2_kernelILi\dE"):
        assert regs == 168, (name, regs)


def test_fp8_one_tile_prefill_split(reports):
    # prefill_kernel<FP8, MODE>: 384 threads: 168 at launch, split 128 x 232
    # (softmax) + 256 x 136 (the other two warpgroups) = 64,512 = 384 x 168
    for name, (regs, _, _) in find(reports["prefill.cu"], r"prefill_kernelILi2ELi\dE"):
        assert regs == 168, (name, regs)
