"""Paged KV cache decode path for GB300 (sm_103a).

A thin ctypes binding over libpa.so, the C-ABI library declared in
``include/pa.h``.  The functions keep the C names and only marshal arguments:
tensors are passed as raw pointers, the stream is the caller's (default: the
current torch stream), and every step of the computation runs in the
library's CUDA kernels.  There is no fallback: if libpa.so is missing or a
call fails, a ``PAError`` is raised.

Device tensors are torch CUDA tensors (torch is used for device memory and
streams only):
  caches    fp16 [num_blocks, num_kv_heads, block_size, head_dim]
  query/out fp16 [num_seqs, num_heads, head_dim]
  key/value fp16 [num_tokens, num_kv_heads, head_dim]
"""
from __future__ import annotations

import ctypes
import os

import numpy as np

_HERE = os.path.dirname(os.path.abspath(__file__))
LIB_PATH = os.path.join(_HERE, "libpa.so")

PA_OK = 0
PA_ERR_INVALID_ARG = -1
PA_ERR_OUT_OF_BLOCKS = -2
PA_ERR_STATE = -3
PA_ERR_WORKSPACE = -4
PA_ERR_CUDA = -5
PA_ERR_UNSUPPORTED = -6
PA_ERR_TIMEOUT = -7

# every symbol include/pa.h declares
EXPORTS = (
    "pa_status_string", "pa_version", "pa_kv_write", "pa_block_copy", "pa_decode_workspace_size", "pa_decode",
    "pa_workspace_status", "pa_alloc_create", "pa_alloc_destroy", "pa_alloc_add_seq", "pa_alloc_append",
    "pa_alloc_fork", "pa_alloc_free_seq", "pa_alloc_seq_len", "pa_alloc_block_tables", "pa_alloc_refcount",
    "pa_alloc_stats", "pa_decode_static_ws", "pa_alloc_free_queue", "pa_alloc_enable_prefix_cache",
    "pa_alloc_match_prefix", "pa_alloc_append_ids", "pa_alloc_block_hash", "pa_alloc_prefix_stats", "pa_sha256",
    "pa_decode_shared_prefix_workspace_size", "pa_decode_shared_prefix", "pa_selftest_wait_timeout",
    "pa_attention_causal_workspace_size", "pa_attention_causal", "pa_kv_write_fp8", "pa_block_copy_typed",
    "pa_decode_typed", "pa_attention_causal_typed", "pa_decode_static_ws_status",
)

# cache element types (PA_KV_* in pa.h)
PA_KV_F16, PA_KV_BF16, PA_KV_FP8_E4M3 = 0, 1, 2

# bytes of the library's built-in scratch array used by pa_decode_static_ws
PA_DECODE_STATIC_WS_BYTES = 64 << 20

_lib = None


class PAError(RuntimeError):
    def __init__(self, code: int, where: str):
        super().__init__(f"{where}: {status_text(code)} ({code})")
        self.code = code


class AllocStats(ctypes.Structure):
    _fields_ = [(n, ctypes.c_int64) for n in
                ("num_blocks", "free_blocks", "used_blocks", "shared_blocks", "num_seqs", "logical_tokens")]


def lib():
    """The loaded libpa.so (raises if it has not been built)."""
    global _lib
    if _lib is None:
        if not os.path.exists(LIB_PATH):
            raise RuntimeError(f"{LIB_PATH} is missing: build it with `python -m paged_kv_cache_12_gb300.build`")
        L = ctypes.CDLL(LIB_PATH)
        vp, i32, i64, sz = ctypes.c_void_p, ctypes.c_int, ctypes.c_int64, ctypes.c_size_t
        sig = {
            "pa_status_string": ([i32], ctypes.c_char_p),
            "pa_version": ([], i32),
            "pa_kv_write": ([vp, vp, vp, vp, vp, i32, i32, i32, i32, i64, vp], i32),
            "pa_block_copy": ([vp, vp, vp, i32, i32, i32, i32, i64, vp], i32),
            "pa_decode_workspace_size": ([i32, i32, i32, i32, i32], sz),
            "pa_decode": ([vp, vp, vp, vp, vp, vp, i32, i32, i32, i32, i32, i64, i32, i32, ctypes.c_float, vp, sz, vp],
                          i32),
            "pa_workspace_status": ([vp, ctypes.POINTER(i32), vp], i32),
            "pa_alloc_create": ([i64, i32, vp, ctypes.POINTER(vp)], i32),
            "pa_alloc_destroy": ([vp], i32),
            "pa_alloc_add_seq": ([vp, i64], i32),
            "pa_alloc_append": ([vp, i32, vp, vp, vp, vp, i32, ctypes.POINTER(i32)], i32),
            "pa_alloc_fork": ([vp, i64, i64], i32),
            "pa_alloc_free_seq": ([vp, i64], i32),
            "pa_alloc_seq_len": ([vp, i64, ctypes.POINTER(i64)], i32),
            "pa_alloc_block_tables": ([vp, i32, vp, vp, i32, vp], i32),
            "pa_alloc_refcount": ([vp, i64, ctypes.POINTER(ctypes.c_int32)], i32),
            "pa_alloc_stats": ([vp, ctypes.POINTER(AllocStats)], i32),
            "pa_decode_static_ws": ([vp, vp, vp, vp, vp, vp, i32, i32, i32, i32, i32, i64, i32, i32,
                                     ctypes.c_float, vp], i32),
            "pa_decode_static_ws_status": ([ctypes.POINTER(i32), vp], i32),
            "pa_alloc_free_queue": ([vp, vp, i64, ctypes.POINTER(i64)], i32),
            "pa_alloc_enable_prefix_cache": ([vp], i32),
            "pa_alloc_match_prefix": ([vp, i64, vp, i32, ctypes.c_uint64, ctypes.POINTER(i32)], i32),
            "pa_alloc_append_ids": ([vp, i32, vp, vp, vp, vp, vp, i32, ctypes.POINTER(i32)], i32),
            "pa_alloc_block_hash": ([vp, i64, vp, ctypes.POINTER(i32)], i32),
            "pa_alloc_prefix_stats": ([vp, ctypes.POINTER(i64), ctypes.POINTER(i64), ctypes.POINTER(i64)], i32),
            "pa_sha256": ([vp, sz, vp], i32),
            "pa_decode_shared_prefix_workspace_size": ([i32, i32, i32, i32, i32], sz),
            "pa_selftest_wait_timeout": ([ctypes.c_longlong, vp, vp], i32),
            "pa_decode_shared_prefix": ([vp, vp, vp, vp, vp, vp, vp, vp, i32, i32, i32, i32, i32, i64, i32, i32,
                                         ctypes.c_float, vp, sz, vp], i32),
            "pa_attention_causal_workspace_size": ([i32, i32, i32, i32, i32, i32], sz),
            "pa_kv_write_fp8": ([vp, vp, vp, vp, vp, i32, i32, i32, i32, i64, ctypes.c_float, ctypes.c_float, vp],
                                i32),
            "pa_block_copy_typed": ([vp, vp, vp, i32, i32, i32, i32, i64, i32, vp], i32),
            "pa_decode_typed": ([vp, vp, vp, vp, vp, vp, i32, i32, i32, i32, i32, i64, i32, i32, ctypes.c_float, i32,
                                 ctypes.c_float, ctypes.c_float, vp, sz, vp], i32),
            "pa_attention_causal_typed": ([vp, vp, vp, vp, vp, vp, vp, i32, i32, i32, i32, i32, i32, i64, i32, i32,
                                           ctypes.c_float, i32, ctypes.c_float, ctypes.c_float, vp, sz, vp], i32),
            "pa_attention_causal": ([vp, vp, vp, vp, vp, vp, vp, i32, i32, i32, i32, i32, i32, i64, i32, i32,
                                     ctypes.c_float, vp, sz, vp], i32),
        }
        for name, (args, res) in sig.items():
            f = getattr(L, name)
            f.argtypes = args
            f.restype = res
        _lib = L
    return _lib


def status_text(code: int) -> str:
    try:
        return lib().pa_status_string(int(code)).decode()
    except Exception:  # the library itself may be what failed to load
        return "status"


def pa_version() -> int:
    return lib().pa_version()


def pa_status_string(code: int) -> str:
    return lib().pa_status_string(int(code)).decode()


def _check(rc: int, where: str):
    if rc != PA_OK:
        raise PAError(rc, where)


# ---------------------------------------------------------------- device calls

def _stream(stream):
    import torch
    if stream is None:
        stream = torch.cuda.current_stream()
    return ctypes.c_void_p(stream.cuda_stream if hasattr(stream, "cuda_stream") else int(stream))


def _need(t, dtype, ndim, name):
    import torch
    if not isinstance(t, torch.Tensor) or not t.is_cuda or t.dtype != dtype or t.dim() != ndim or not t.is_contiguous():
        raise ValueError(f"{name}: expected a contiguous CUDA {dtype} tensor with {ndim} dims")


def pa_kv_write(key, value, slot_mapping, k_cache, v_cache, stream=None):
    """Store key[t], value[t] at slot slot_mapping[t] of the caches (slot < 0:
    skipped); fp16 rows into fp16 caches or bf16 rows into bf16 caches (a copy
    of 16-bit elements either way)."""
    import torch
    dt = torch.bfloat16 if k_cache.dtype == torch.bfloat16 else torch.float16
    _need(k_cache, dt, 4, "k_cache")
    _need(v_cache, dt, 4, "v_cache")
    _need(key, dt, 3, "key")
    _need(value, dt, 3, "value")
    _need(slot_mapping, torch.int64, 1, "slot_mapping")
    nb, hkv, bs, d = k_cache.shape
    if v_cache.shape != k_cache.shape or key.shape != value.shape or key.shape[1:] != (hkv, d) \
            or slot_mapping.shape[0] != key.shape[0]:
        raise ValueError("pa_kv_write: shape mismatch")
    _check(lib().pa_kv_write(key.data_ptr(), value.data_ptr(), slot_mapping.data_ptr(), k_cache.data_ptr(),
                             v_cache.data_ptr(), key.shape[0], hkv, d, bs, nb, _stream(stream)), "pa_kv_write")


def kv_dtype_of(cache) -> int:
    """PA_KV_* of a cache tensor: float16, bfloat16, or one-byte E4M3 codes
    (uint8 or torch.float8_e4m3fn)."""
    import torch
    if cache.dtype == torch.float16:
        return PA_KV_F16
    if cache.dtype == torch.bfloat16:
        return PA_KV_BF16
    if cache.dtype == torch.uint8 or cache.dtype == getattr(torch, "float8_e4m3fn", None):
        return PA_KV_FP8_E4M3
    raise ValueError(f"unsupported cache dtype {cache.dtype}")


def _need_cache(t, name, kv):
    import torch
    want = {PA_KV_F16: (torch.float16,), PA_KV_BF16: (torch.bfloat16,),
            PA_KV_FP8_E4M3: (torch.uint8, getattr(torch, "float8_e4m3fn", torch.uint8))}[kv]
    if not isinstance(t, torch.Tensor) or not t.is_cuda or t.dtype not in want or t.dim() != 4 \
            or not t.is_contiguous():
        raise ValueError(f"{name}: expected a contiguous 4-d CUDA cache tensor of {want[0]}")


def pa_block_copy(k_cache, v_cache, pairs, stream=None):
    """Copy every (src, dst) block pair of int64 ``pairs`` [n, 2], K and V
    (caches of fp16, bf16 or fp8 codes)."""
    import torch
    kv = kv_dtype_of(k_cache)
    _need_cache(k_cache, "k_cache", kv)
    _need_cache(v_cache, "v_cache", kv)
    _need(pairs, torch.int64, 2, "pairs")
    nb, hkv, bs, d = k_cache.shape
    if v_cache.shape != k_cache.shape or pairs.shape[1] != 2:
        raise ValueError("pa_block_copy: shape mismatch")
    if kv == PA_KV_F16:
        _check(lib().pa_block_copy(k_cache.data_ptr(), v_cache.data_ptr(), pairs.data_ptr(), pairs.shape[0], hkv, d,
                                   bs, nb, _stream(stream)), "pa_block_copy")
    else:
        _check(lib().pa_block_copy_typed(k_cache.data_ptr(), v_cache.data_ptr(), pairs.data_ptr(), pairs.shape[0],
                                         hkv, d, bs, nb, kv, _stream(stream)), "pa_block_copy_typed")


def pa_kv_write_fp8(key, value, slot_mapping, k_cache, v_cache, k_scale, v_scale, stream=None):
    """Quantise fp16 key/value rows into caches of FP8 E4M3 codes (uint8 or
    float8_e4m3fn tensors): code = E4M3(fl32(x * fl32(1 / scale))), nearest
    value, ties to even, saturating at 448."""
    import torch
    _need_cache(k_cache, "k_cache", PA_KV_FP8_E4M3)
    _need_cache(v_cache, "v_cache", PA_KV_FP8_E4M3)
    _need(key, torch.float16, 3, "key")
    _need(value, torch.float16, 3, "value")
    _need(slot_mapping, torch.int64, 1, "slot_mapping")
    nb, hkv, bs, d = k_cache.shape
    if v_cache.shape != k_cache.shape or key.shape != value.shape or key.shape[1:] != (hkv, d) \
            or slot_mapping.shape[0] != key.shape[0]:
        raise ValueError("pa_kv_write_fp8: shape mismatch")
    _check(lib().pa_kv_write_fp8(key.data_ptr(), value.data_ptr(), slot_mapping.data_ptr(), k_cache.data_ptr(),
                                 v_cache.data_ptr(), key.shape[0], hkv, d, bs, nb, float(k_scale), float(v_scale),
                                 _stream(stream)), "pa_kv_write_fp8")


def pa_decode_typed(out, query, k_cache, v_cache, block_tables, context_lens, scale, max_context_len, workspace,
                    k_scale=1.0, v_scale=1.0, stream=None):
    """pa_decode over a cache of fp16, bf16 (bf16 query/out) or fp8 E4M3 codes
    (fp16 query/out; a code stands for its value times k_scale or v_scale).
    Workspace: pa_decode_workspace_size."""
    import torch
    kv = kv_dtype_of(k_cache)
    qdt = torch.bfloat16 if kv == PA_KV_BF16 else torch.float16
    _need_cache(k_cache, "k_cache", kv)
    _need_cache(v_cache, "v_cache", kv)
    for t, dt, nd, nm in ((out, qdt, 3, "out"), (query, qdt, 3, "query"),
                          (block_tables, torch.int32, 2, "block_tables"), (context_lens, torch.int32, 1, "context_lens"),
                          (workspace, torch.uint8, 1, "workspace")):
        _need(t, dt, nd, nm)
    nb, hkv, bs, d = k_cache.shape
    B, hq, d2 = query.shape
    if out.shape != query.shape or d2 != d or v_cache.shape != k_cache.shape or block_tables.shape[0] != B \
            or context_lens.shape[0] != B:
        raise ValueError("pa_decode_typed: shape mismatch")
    _check(lib().pa_decode_typed(out.data_ptr(), query.data_ptr(), k_cache.data_ptr(), v_cache.data_ptr(),
                                 block_tables.data_ptr(), context_lens.data_ptr(), B, hq, hkv, d, bs, nb,
                                 block_tables.shape[1], int(max_context_len), float(scale), kv, float(k_scale),
                                 float(v_scale), workspace.data_ptr(), workspace.numel(), _stream(stream)),
           "pa_decode_typed")


def pa_attention_causal_typed(out, query, k_cache, v_cache, block_tables, context_lens, query_start, scale,
                              max_context_len, workspace, k_scale=1.0, v_scale=1.0, stream=None):
    """pa_attention_causal over a cache of fp16, bf16 or fp8 E4M3 codes (as
    pa_decode_typed).  Workspace: pa_attention_causal_workspace_size."""
    import torch
    kv = kv_dtype_of(k_cache)
    qdt = torch.bfloat16 if kv == PA_KV_BF16 else torch.float16
    _need_cache(k_cache, "k_cache", kv)
    _need_cache(v_cache, "v_cache", kv)
    for t, dt, nd, nm in ((out, qdt, 3, "out"), (query, qdt, 3, "query"),
                          (block_tables, torch.int32, 2, "block_tables"), (context_lens, torch.int32, 1, "context_lens"),
                          (query_start, torch.int32, 1, "query_start"), (workspace, torch.uint8, 1, "workspace")):
        _need(t, dt, nd, nm)
    nb, hkv, bs, d = k_cache.shape
    nq, hq, d2 = query.shape
    B = context_lens.shape[0]
    if out.shape != query.shape or d2 != d or v_cache.shape != k_cache.shape or block_tables.shape[0] != B \
            or query_start.shape[0] != B + 1:
        raise ValueError("pa_attention_causal_typed: shape mismatch")
    _check(lib().pa_attention_causal_typed(out.data_ptr(), query.data_ptr(), k_cache.data_ptr(), v_cache.data_ptr(),
                                           block_tables.data_ptr(), context_lens.data_ptr(), query_start.data_ptr(),
                                           B, nq, hq, hkv, d, bs, nb, block_tables.shape[1], int(max_context_len),
                                           float(scale), kv, float(k_scale), float(v_scale), workspace.data_ptr(),
                                           workspace.numel(), _stream(stream)), "pa_attention_causal_typed")


def pa_decode_workspace_size(num_seqs, num_heads, num_kv_heads, head_dim, max_context_len) -> int:
    n = lib().pa_decode_workspace_size(int(num_seqs), int(num_heads), int(num_kv_heads), int(head_dim),
                                       int(max_context_len))
    if n == 0 and num_seqs >= 0:
        raise PAError(PA_ERR_INVALID_ARG, "pa_decode_workspace_size")
    return n


def pa_decode(out, query, k_cache, v_cache, block_tables, context_lens, scale, max_context_len, workspace,
              stream=None):
    """Paged decode attention: out[i][h] = softmax(scale q K^T) V over sequence i's blocks."""
    import torch
    for t, dt, nd, nm in ((out, torch.float16, 3, "out"), (query, torch.float16, 3, "query"),
                          (k_cache, torch.float16, 4, "k_cache"), (v_cache, torch.float16, 4, "v_cache"),
                          (block_tables, torch.int32, 2, "block_tables"), (context_lens, torch.int32, 1, "context_lens"),
                          (workspace, torch.uint8, 1, "workspace")):
        _need(t, dt, nd, nm)
    nb, hkv, bs, d = k_cache.shape
    B, hq, d2 = query.shape
    if out.shape != query.shape or d2 != d or v_cache.shape != k_cache.shape or block_tables.shape[0] != B \
            or context_lens.shape[0] != B:
        raise ValueError("pa_decode: shape mismatch")
    _check(lib().pa_decode(out.data_ptr(), query.data_ptr(), k_cache.data_ptr(), v_cache.data_ptr(),
                           block_tables.data_ptr(), context_lens.data_ptr(), B, hq, hkv, d, bs, nb,
                           block_tables.shape[1], int(max_context_len), float(scale), workspace.data_ptr(),
                           workspace.numel(), _stream(stream)), "pa_decode")


def pa_decode_static_ws(out, query, k_cache, v_cache, block_tables, context_lens, scale, max_context_len,
                        stream=None):
    """pa_decode without a workspace argument, for callers that cannot allocate
    device memory: the library's own fixed scratch array (64 MiB, shared by all
    calls on a device) stands in for it.  Calls that overlap on the GPU must not
    share it; sizes needing more scratch raise PAError(PA_ERR_WORKSPACE)."""
    import torch
    for t, dt, nd, nm in ((out, torch.float16, 3, "out"), (query, torch.float16, 3, "query"),
                          (k_cache, torch.float16, 4, "k_cache"), (v_cache, torch.float16, 4, "v_cache"),
                          (block_tables, torch.int32, 2, "block_tables"), (context_lens, torch.int32, 1, "context_lens")):
        _need(t, dt, nd, nm)
    nb, hkv, bs, d = k_cache.shape
    B, hq, d2 = query.shape
    if out.shape != query.shape or d2 != d or v_cache.shape != k_cache.shape or block_tables.shape[0] != B \
            or context_lens.shape[0] != B:
        raise ValueError("pa_decode_static_ws: shape mismatch")
    _check(lib().pa_decode_static_ws(out.data_ptr(), query.data_ptr(), k_cache.data_ptr(), v_cache.data_ptr(),
                                     block_tables.data_ptr(), context_lens.data_ptr(), B, hq, hkv, d, bs, nb,
                                     block_tables.shape[1], int(max_context_len), float(scale), _stream(stream)),
           "pa_decode_static_ws")


def pa_decode_static_ws_status(stream=None) -> int:
    """The error word the last pa_decode_static_ws call on the current device
    left in the library's scratch array (PA_OK or PA_ERR_TIMEOUT); synchronises
    the stream."""
    st = ctypes.c_int(0)
    _check(lib().pa_decode_static_ws_status(ctypes.byref(st), _stream(stream)), "pa_decode_static_ws_status")
    return st.value


def pa_decode_shared_prefix_workspace_size(num_seqs, num_heads, num_kv_heads, head_dim, max_context_len) -> int:
    n = lib().pa_decode_shared_prefix_workspace_size(int(num_seqs), int(num_heads), int(num_kv_heads),
                                                     int(head_dim), int(max_context_len))
    if n == 0:
        raise PAError(PA_ERR_INVALID_ARG, "pa_decode_shared_prefix_workspace_size")
    return n


def pa_decode_shared_prefix(out, query, k_cache, v_cache, block_tables, context_lens, group_leader, shared_len,
                            scale, max_context_len, workspace, stream=None):
    """pa_decode where runs of sequences share the blocks of a common prefix:
    group_leader[i] = first sequence of i's group, shared_len[leader] = tokens
    shared (int32 device tensors of num_seqs)."""
    import torch
    for t, dt, nd, nm in ((out, torch.float16, 3, "out"), (query, torch.float16, 3, "query"),
                          (k_cache, torch.float16, 4, "k_cache"), (v_cache, torch.float16, 4, "v_cache"),
                          (block_tables, torch.int32, 2, "block_tables"), (context_lens, torch.int32, 1, "context_lens"),
                          (group_leader, torch.int32, 1, "group_leader"), (shared_len, torch.int32, 1, "shared_len"),
                          (workspace, torch.uint8, 1, "workspace")):
        _need(t, dt, nd, nm)
    nb, hkv, bs, d = k_cache.shape
    B, hq, d2 = query.shape
    if out.shape != query.shape or d2 != d or v_cache.shape != k_cache.shape or block_tables.shape[0] != B \
            or context_lens.shape[0] != B or group_leader.shape[0] != B or shared_len.shape[0] != B:
        raise ValueError("pa_decode_shared_prefix: shape mismatch")
    _check(lib().pa_decode_shared_prefix(out.data_ptr(), query.data_ptr(), k_cache.data_ptr(), v_cache.data_ptr(),
                                         block_tables.data_ptr(), context_lens.data_ptr(), group_leader.data_ptr(),
                                         shared_len.data_ptr(), B, hq, hkv, d, bs, nb, block_tables.shape[1],
                                         int(max_context_len), float(scale), workspace.data_ptr(), workspace.numel(),
                                         _stream(stream)), "pa_decode_shared_prefix")


def pa_attention_causal_workspace_size(num_seqs, num_query_tokens, num_heads, num_kv_heads, head_dim,
                                       max_context_len) -> int:
    n = lib().pa_attention_causal_workspace_size(int(num_seqs), int(num_query_tokens), int(num_heads),
                                                 int(num_kv_heads), int(head_dim), int(max_context_len))
    if n == 0:
        raise PAError(PA_ERR_INVALID_ARG, "pa_attention_causal_workspace_size")
    return n


def pa_attention_causal(out, query, k_cache, v_cache, block_tables, context_lens, query_start, scale,
                        max_context_len, workspace, stream=None):
    """Several new tokens per sequence (chunked prefill, speculative tokens):
    query rows query_start[i] .. query_start[i+1]-1 are sequence i's last new
    tokens, each attending to the positions up to its own."""
    import torch
    for t, dt, nd, nm in ((out, torch.float16, 3, "out"), (query, torch.float16, 3, "query"),
                          (k_cache, torch.float16, 4, "k_cache"), (v_cache, torch.float16, 4, "v_cache"),
                          (block_tables, torch.int32, 2, "block_tables"), (context_lens, torch.int32, 1, "context_lens"),
                          (query_start, torch.int32, 1, "query_start"), (workspace, torch.uint8, 1, "workspace")):
        _need(t, dt, nd, nm)
    nb, hkv, bs, d = k_cache.shape
    nq, hq, d2 = query.shape
    B = context_lens.shape[0]
    if out.shape != query.shape or d2 != d or v_cache.shape != k_cache.shape or block_tables.shape[0] != B \
            or query_start.shape[0] != B + 1:
        raise ValueError("pa_attention_causal: shape mismatch")
    _check(lib().pa_attention_causal(out.data_ptr(), query.data_ptr(), k_cache.data_ptr(), v_cache.data_ptr(),
                                     block_tables.data_ptr(), context_lens.data_ptr(), query_start.data_ptr(), B, nq,
                                     hq, hkv, d, bs, nb, block_tables.shape[1], int(max_context_len), float(scale),
                                     workspace.data_ptr(), workspace.numel(), _stream(stream)), "pa_attention_causal")


def pa_selftest_wait_timeout(limit_cycles: int, status, stream=None):
    """Run the bounded-wait self-test; `status` is an int32 CUDA tensor of one element."""
    import torch
    _need(status, torch.int32, 1, "status")
    _check(lib().pa_selftest_wait_timeout(int(limit_cycles), status.data_ptr(), _stream(stream)),
           "pa_selftest_wait_timeout")


def pa_workspace_status(workspace, stream=None) -> int:
    st = ctypes.c_int(0)
    _check(lib().pa_workspace_status(workspace.data_ptr(), ctypes.byref(st), _stream(stream)), "pa_workspace_status")
    return st.value


# ---------------------------------------------------------------- allocator

def _i64(a):
    return np.ascontiguousarray(a, dtype=np.int64)


def pa_sha256(data: bytes) -> bytes:
    """SHA-256 of a byte string, as the prefix cache computes it."""
    out = (ctypes.c_uint8 * 32)()
    buf = bytes(data)
    _check(lib().pa_sha256(buf, len(buf), out), "pa_sha256")
    return bytes(out)


class Allocator:
    """Host block allocator (pa_alloc_* calls)."""

    def __init__(self, num_blocks: int, block_size: int, free_order=None, prefix_cache: bool = False):
        self._h = ctypes.c_void_p()
        self.num_blocks, self.block_size = int(num_blocks), int(block_size)
        order = None if free_order is None else np.ascontiguousarray(free_order, dtype=np.int32)
        _check(lib().pa_alloc_create(self.num_blocks, self.block_size,
                                     None if order is None else order.ctypes.data, ctypes.byref(self._h)),
               "pa_alloc_create")
        if prefix_cache:
            _check(lib().pa_alloc_enable_prefix_cache(self._h), "pa_alloc_enable_prefix_cache")

    def close(self):
        if self._h:
            lib().pa_alloc_destroy(self._h)
            self._h = ctypes.c_void_p()

    def __del__(self):
        try:
            self.close()
        except Exception:
            pass

    def add_seq(self, seq_id: int):
        _check(lib().pa_alloc_add_seq(self._h, int(seq_id)), "pa_alloc_add_seq")

    def append(self, seq_ids, counts):
        """Reserve slots; returns (slots int64 [sum(counts)], pairs int64 [n, 2])."""
        ids = _i64(seq_ids)
        cnt = np.ascontiguousarray(counts, dtype=np.int32)
        slots = np.empty(max(0, int(cnt[cnt > 0].sum())), dtype=np.int64)
        pairs = np.empty((max(1, len(ids)), 2), dtype=np.int64)
        n = ctypes.c_int(0)
        _check(lib().pa_alloc_append(self._h, len(ids), ids.ctypes.data, cnt.ctypes.data, slots.ctypes.data,
                                     pairs.ctypes.data, pairs.shape[0], ctypes.byref(n)), "pa_alloc_append")
        return slots, pairs[: n.value].copy()

    def append_ids(self, seq_ids, counts, token_ids):
        """append() with the appended tokens' ids (concatenated in sequence order)."""
        ids = _i64(seq_ids)
        cnt = np.ascontiguousarray(counts, dtype=np.int32)
        toks = np.ascontiguousarray(token_ids, dtype=np.int32)
        slots = np.empty(max(0, int(cnt[cnt > 0].sum())), dtype=np.int64)
        pairs = np.empty((max(1, len(ids)), 2), dtype=np.int64)
        n = ctypes.c_int(0)
        _check(lib().pa_alloc_append_ids(self._h, len(ids), ids.ctypes.data, cnt.ctypes.data, toks.ctypes.data,
                                         slots.ctypes.data, pairs.ctypes.data, pairs.shape[0], ctypes.byref(n)),
               "pa_alloc_append_ids")
        return slots, pairs[: n.value].copy()

    def match_prefix(self, seq_id: int, tokens, extra_key: int = 0) -> int:
        """Start seq_id on a prompt, reusing cached full blocks; returns the tokens covered."""
        toks = np.ascontiguousarray(tokens, dtype=np.int32)
        got = ctypes.c_int(0)
        _check(lib().pa_alloc_match_prefix(self._h, int(seq_id), toks.ctypes.data, len(toks),
                                           ctypes.c_uint64(int(extra_key) & (2 ** 64 - 1)), ctypes.byref(got)),
               "pa_alloc_match_prefix")
        return got.value

    def free_queue(self):
        n = ctypes.c_int64(0)
        lib().pa_alloc_free_queue(self._h, None, 0, ctypes.byref(n))
        out = np.empty(n.value, dtype=np.int32)
        _check(lib().pa_alloc_free_queue(self._h, out.ctypes.data, len(out), ctypes.byref(n)), "pa_alloc_free_queue")
        return out.tolist()

    def block_hash(self, block: int):
        h = (ctypes.c_uint8 * 32)()
        c = ctypes.c_int(0)
        _check(lib().pa_alloc_block_hash(self._h, int(block), h, ctypes.byref(c)), "pa_alloc_block_hash")
        return bytes(h), bool(c.value)

    def prefix_stats(self) -> dict:
        c, q, h = ctypes.c_int64(0), ctypes.c_int64(0), ctypes.c_int64(0)
        _check(lib().pa_alloc_prefix_stats(self._h, ctypes.byref(c), ctypes.byref(q), ctypes.byref(h)),
               "pa_alloc_prefix_stats")
        return {"cached_blocks": c.value, "queries": q.value, "hits": h.value}

    def fork(self, parent: int, child: int):
        _check(lib().pa_alloc_fork(self._h, int(parent), int(child)), "pa_alloc_fork")

    def free_seq(self, seq_id: int):
        _check(lib().pa_alloc_free_seq(self._h, int(seq_id)), "pa_alloc_free_seq")

    def seq_len(self, seq_id: int) -> int:
        n = ctypes.c_int64(0)
        _check(lib().pa_alloc_seq_len(self._h, int(seq_id), ctypes.byref(n)), "pa_alloc_seq_len")
        return n.value

    def block_tables(self, seq_ids, max_blocks: int):
        """int32 [n, max_blocks] tables (unused -1) and int32 [n] lengths."""
        ids = _i64(seq_ids)
        tab = np.empty((len(ids), int(max_blocks)), dtype=np.int32)
        lens = np.empty(len(ids), dtype=np.int32)
        _check(lib().pa_alloc_block_tables(self._h, len(ids), ids.ctypes.data, tab.ctypes.data, int(max_blocks),
                                           lens.ctypes.data), "pa_alloc_block_tables")
        return tab, lens

    def refcount(self, block: int) -> int:
        c = ctypes.c_int32(0)
        _check(lib().pa_alloc_refcount(self._h, int(block), ctypes.byref(c)), "pa_alloc_refcount")
        return c.value

    def stats(self) -> dict:
        s = AllocStats()
        _check(lib().pa_alloc_stats(self._h, ctypes.byref(s)), "pa_alloc_stats")
        return {n: getattr(s, n) for n, _ in AllocStats._fields_}
