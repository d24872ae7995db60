"""The C-ABI library loads on a machine without a GPU and exports every symbol
include/*.h declares; host-only calls behave as documented."""
import ctypes
import glob
import os
import re

import pytest

import paged_kv_cache_12_gb300 as pa
from conftest import ROOT


def declared_symbols():
    names = set()
    for h in glob.glob(os.path.join(ROOT, "include", "*.h")):
        text = open(h).read()
        names |= set(re.findall(r"^PA_API[^;(]*?\b(pa_\w+)\s*\(", text, flags=re.M))
    return names


def test_header_declares_the_binding_exports():
    assert declared_symbols() == set(pa.EXPORTS)


def test_every_declared_symbol_is_exported():
    lib = ctypes.CDLL(pa.LIB_PATH)
    for name in declared_symbols():
        assert hasattr(lib, name), name


def test_status_strings_and_version():
    assert pa.pa_version() == 1
    for code in range(-7, 1):
        assert pa.pa_status_string(code) and pa.pa_status_string(code) != "unknown status"
    assert pa.pa_status_string(-99) == "unknown status"


def test_workspace_size_is_a_host_bound():
    small = pa.pa_decode_workspace_size(4, 4, 2, 64, 100)
    big = pa.pa_decode_workspace_size(100, 64, 8, 128, 8192)
    # header + offsets + item list; partial results only when a sequence can span partitions
    assert 0 < small < 8192
    # 100 x 8 x 8 partitions of 1024 tokens reach 4096 items: 8 partials per head
    assert big >= 100 * 8 * 64 * 128 * 4 and big < 100 * 16 * 64 * 128 * 4
    assert pa.pa_decode_workspace_size(100, 64, 8, 128, 256) < 100 * 64 * 128 * 4
    # few sequences: shorter partitions (256 tokens) so that the work still spreads
    assert pa.pa_decode_workspace_size(2, 8, 1, 128, 8192) >= 2 * 32 * 8 * 128 * 4
    # groups smaller than 8 aim at 8 / G times as many items: 64 x 32 kv heads x
    # 2048 tokens takes 1024-token partitions at G = 8, 256-token ones at G = 1
    g8 = pa.pa_decode_workspace_size(64, 256, 32, 128, 2048)
    assert 64 * 2 * 256 * 128 * 4 <= g8 < 64 * 3 * 256 * 128 * 4
    g1 = pa.pa_decode_workspace_size(64, 32, 32, 128, 2048)
    assert 64 * 8 * 32 * 128 * 4 <= g1 < 64 * 9 * 32 * 128 * 4
    assert pa.lib().pa_decode_workspace_size(1, 8, 0, 128, 10) == 0
    # multi-token form: a partial row per query row and partition (400 rows x 8
    # partitions of 1024), and the narrow kernel's merge scratch (160 CTAs x two
    # item parities x four quarters' 128 x 32 fp32 O and 32 (m, l) pairs)
    spec = pa.pa_attention_causal_workspace_size(100, 400, 64, 8, 128, 8192)
    scratch = 160 * 2 * 4 * (128 * 32 * 4 + 32 * 8)
    assert 400 * 8 * 64 * 128 * 4 + scratch <= spec < 400 * 9 * 64 * 128 * 4 + scratch
    assert pa.lib().pa_attention_causal_workspace_size(1, 4, 6, 4, 128, 10) == 0


def test_host_checks_fail_before_any_launch():
    L = pa.lib()
    nul = None
    # unsupported head_dim / block size / group size: rejected on the host
    assert L.pa_decode(nul, nul, nul, nul, nul, nul, 1, 8, 1, 96, 16, 10, 1, 16, 0.1, nul, 0, nul) == pa.PA_ERR_UNSUPPORTED
    assert L.pa_decode(nul, nul, nul, nul, nul, nul, 1, 8, 1, 128, 64, 10, 1, 16, 0.1, nul, 0, nul) == pa.PA_ERR_UNSUPPORTED
    assert L.pa_decode(nul, nul, nul, nul, nul, nul, 1, 32, 1, 128, 16, 10, 1, 16, 0.1, nul, 0, nul) == pa.PA_ERR_UNSUPPORTED
    assert L.pa_decode(nul, nul, nul, nul, nul, nul, 1, 6, 4, 128, 16, 10, 1, 16, 0.1, nul, 0, nul) == pa.PA_ERR_INVALID_ARG
    # missing pointers
    assert L.pa_decode(nul, nul, nul, nul, nul, nul, 1, 8, 1, 128, 16, 10, 1, 16, 0.1, nul, 0, nul) == pa.PA_ERR_INVALID_ARG
    assert L.pa_kv_write(nul, nul, nul, nul, nul, 3, 8, 128, 16, 10, nul) == pa.PA_ERR_INVALID_ARG
    assert L.pa_block_copy(nul, nul, nul, 2, 8, 128, 16, 10, nul) == pa.PA_ERR_INVALID_ARG
    assert L.pa_kv_write(nul, nul, nul, nul, nul, 1, 8, 100, 16, 10, nul) == pa.PA_ERR_INVALID_ARG  # head_dim % 8
    # empty work is valid and launches nothing
    assert L.pa_kv_write(nul, nul, nul, nul, nul, 0, 8, 128, 16, 10, nul) == pa.PA_OK
    assert L.pa_block_copy(nul, nul, nul, 0, 8, 128, 16, 10, nul) == pa.PA_OK
    assert L.pa_decode(nul, nul, nul, nul, nul, nul, 0, 8, 1, 128, 16, 10, 1, 16, 0.1, nul, 0, nul) == pa.PA_OK
    assert L.pa_decode(nul, nul, nul, nul, nul, nul, 1, 8, 1, 128, 16, 10, 1, 16, -0.1, nul, 0, nul) == pa.PA_ERR_INVALID_ARG
    # the variant without a workspace checks its arguments as pa_decode does
    # and only then its scratch size (fake aligned addresses: never read)
    S = L.pa_decode_static_ws
    fake = ctypes.c_void_p(1 << 20)
    assert S(nul, nul, nul, nul, nul, nul, 1, 8, 1, 96, 16, 10, 1, 16, 0.1, nul) == pa.PA_ERR_UNSUPPORTED
    assert S(nul, nul, nul, nul, nul, nul, 1, 32, 1, 128, 16, 10, 1, 16, 0.1, nul) == pa.PA_ERR_UNSUPPORTED
    assert S(nul, nul, nul, nul, nul, nul, 1, 6, 4, 128, 16, 10, 1, 16, 0.1, nul) == pa.PA_ERR_INVALID_ARG
    assert S(nul, nul, nul, nul, nul, nul, 1, 8, 1, 128, 16, 0, 1, 16, 0.1, nul) == pa.PA_ERR_INVALID_ARG
    assert S(nul, nul, nul, nul, nul, nul, 1, 8, 1, 128, 16, 10, 1, 16, float("nan"), nul) == pa.PA_ERR_INVALID_ARG
    assert S(nul, nul, nul, nul, nul, nul, 1, 8, 1, 128, 16, 10, 1, 16, 0.1, nul) == pa.PA_ERR_INVALID_ARG
    assert S(nul, nul, nul, nul, nul, nul, 0, 8, 1, 128, 16, 10, 1, 16, 0.1, nul) == pa.PA_OK
    assert S(fake, fake, fake, fake, fake, fake, 4096, 64, 8, 128, 16, 10, 1, 32768, 0.1, nul) == pa.PA_ERR_WORKSPACE
    assert L.pa_decode_static_ws_status(nul, nul) == pa.PA_ERR_INVALID_ARG
    # the multi-token form: same shape rules; no query rows launches nothing; rows need sequences
    C = L.pa_attention_causal
    assert C(nul, nul, nul, nul, nul, nul, nul, 1, 4, 8, 1, 96, 16, 10, 1, 16, 0.1, nul, 0, nul) == pa.PA_ERR_UNSUPPORTED
    assert C(nul, nul, nul, nul, nul, nul, nul, 1, 4, 8, 1, 128, 16, 10, 1, 16, 0.1, nul, 0, nul) == pa.PA_ERR_INVALID_ARG
    assert C(nul, nul, nul, nul, nul, nul, nul, 0, 4, 8, 1, 128, 16, 10, 1, 16, 0.1, nul, 0, nul) == pa.PA_ERR_INVALID_ARG
    assert C(nul, nul, nul, nul, nul, nul, nul, 3, 0, 8, 1, 128, 16, 10, 1, 16, 0.1, nul, 0, nul) == pa.PA_OK
    assert C(nul, nul, nul, nul, nul, nul, nul, 1, 4, 8, 3, 128, 16, 10, 1, 16, 0.1, nul, 0, nul) == pa.PA_ERR_INVALID_ARG
