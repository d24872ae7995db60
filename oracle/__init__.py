"""The oracle: a plain, slow, obviously correct CPU statement of the paged decode path.

TEST INFRASTRUCTURE ONLY.  Only ``tests/``, ``__graft_entry__.smoke()`` and the
CPU-baseline leg of ``bench.py`` may import this package.  It shares no code
with ``paged_kv_cache_12_gb300`` (neither imports the other); the only module
both sides use is the seeded input generator, which holds none of the method's
arithmetic.

Contents, each with the passage it follows:

* ``kv_bytes_per_token`` -- the KV-size formula of "PagedAttention de vLLM :
  comment la gestion de la VRAM soutient l'inference des grands modeles"
  (deepsonar.com.cn), section 2.1.
* ``OracleAllocator`` -- fixed-size blocks, per-sequence block table and
  allocation on demand (deepsonar page section 2.2 and section VII steps 1-3;
  "PagedAttention : comment optimiser la memoire GPU lors de l'inference des
  LLM" (deeplearn.tn), section "Un exemple concret d'allocation"), reference
  counts with copy-on-write (deepsonar page section 2.3), free queue handing out
  from the head and taking freed blocks back at the tail (deepsonar page
  section 2.4).
* prefix caching in ``OracleAllocator`` (deepsonar page section 2.4 and
  section VII step 5): chained block hashes sha256(parent hash, block tokens,
  extra key), a hash -> block map, the free queue as eviction order, prefix
  matching block by block with the last prompt token always recomputed.
* ``kv_write`` / ``block_copy`` -- the new token's K/V go into the free slot of
  the sequence's current block (deeplearn.tn page, same section); a writer that
  finds a shared block copies it first (deepsonar page section 2.3).
* ``paged_decode`` / ``paged_decode_split`` -- fp64 attention over the gathered
  history, in C (``oracle.c``), see that file's header for the passages.
* ``paged_attention_causal`` -- several new query tokens per sequence, each
  attending causally to the positions up to its own (deepsonar page section
  2.5: chunked prefill and speculative tokens), in C.
* ``paged_attention_typed`` / ``kv_write_fp8`` / ``e4m3_encode`` -- the same
  attention over caches of bf16 or fp8 E4M3 codes with one scale for K and one
  for V, and the quantising write into an fp8 cache.  The pages keep the cache
  in fp16 (deepsonar page section 2.1, two bytes per element); these follow
  the formats' definitions, and the quantiser is the reading recorded with it.

Readings where the pages are silent are listed with each function.
"""
from __future__ import annotations

import ctypes
import hashlib
import os
import struct
import subprocess
import threading
from collections import OrderedDict
from concurrent.futures import ThreadPoolExecutor

import numpy as np

_HERE = os.path.dirname(os.path.abspath(__file__))
_SRC = os.path.join(_HERE, "oracle.c")
_BUILD_DIR = os.path.join(_HERE, "_build")
_LIB_PATH = os.path.join(_BUILD_DIR, "liboracle.so")

_lib = None
_lib_lock = threading.Lock()


def build(force: bool = False) -> str:
    """Compile oracle.c into a shared library with the host C compiler."""
    os.makedirs(_BUILD_DIR, exist_ok=True)
    if force or not os.path.exists(_LIB_PATH) or os.path.getmtime(_LIB_PATH) < os.path.getmtime(_SRC):
        tmp = _LIB_PATH + f".tmp{os.getpid()}"
        subprocess.check_call(["gcc", "-O2", "-std=c99", "-fPIC", "-shared", "-o", tmp, _SRC, "-lm"])
        os.replace(tmp, _LIB_PATH)
    return _LIB_PATH


def _load():
    global _lib
    with _lib_lock:
        if _lib is None:
            lib = ctypes.CDLL(build())
            i32, i64, dbl, vp = ctypes.c_int, ctypes.c_int64, ctypes.c_double, ctypes.c_void_p
            lib.or_half_to_double.argtypes = [ctypes.c_uint16]
            lib.or_half_to_double.restype = dbl
            common = [vp, vp, vp, vp, vp, vp, i32, i32, i32, i32, i32, i32, i64, i64, i64, dbl]
            lib.or_paged_decode.argtypes = common + [i32, i32]
            lib.or_paged_decode.restype = i32
            lib.or_paged_decode_split.argtypes = common + [i32, i32, i32]
            lib.or_paged_decode_split.restype = i32
            lib.or_paged_attention_causal.argtypes = [vp, vp, vp, vp, vp, vp, vp, i32, i32, i32, i32, i32, i32,
                                                      i64, i64, i64, dbl, i32, i32]
            lib.or_paged_attention_causal.restype = i32
            lib.or_bf16_to_double.argtypes = [ctypes.c_uint16]
            lib.or_bf16_to_double.restype = dbl
            lib.or_e4m3_to_double.argtypes = [ctypes.c_uint8]
            lib.or_e4m3_to_double.restype = dbl
            lib.or_paged_attention_typed.argtypes = [vp, vp, i32, vp, vp, i32, dbl, dbl, vp, vp, vp, i32, i32, i32,
                                                     i32, i32, i32, i64, i64, i64, dbl, i32, i32]
            lib.or_paged_attention_typed.restype = i32
            _lib = lib
    return _lib


def half_to_double(bits: int) -> float:
    """The C oracle's own binary16 -> double conversion, for pinning it."""
    return _load().or_half_to_double(int(bits) & 0xFFFF)


def bf16_to_double(bits: int) -> float:
    """The C oracle's bfloat16 -> double conversion."""
    return _load().or_bf16_to_double(int(bits) & 0xFFFF)


def e4m3_to_double(code: int) -> float:
    """The C oracle's FP8 E4M3 code -> double conversion."""
    return _load().or_e4m3_to_double(int(code) & 0xFF)


KV_F16, KV_BF16, KV_FP8_E4M3 = 0, 1, 2


def e4m3_encode(x) -> np.ndarray:
    """float32 values -> FP8 E4M3 codes, rounding to the nearest representable
    value, ties to the even code, magnitudes beyond the largest finite value
    (448) saturating to it, NaN to the NaN code; the sign is kept (so -0 and
    negative values that round to zero give 0x80).  Written as a search over
    the format's 127 finite non-negative values (``e4m3_to_double`` of codes
    0x00 .. 0x7E), which is the definition of rounding to nearest."""
    x = np.asarray(x, dtype=np.float32)
    values = np.array([e4m3_to_double(c) for c in range(0x7F)])     # increasing
    a = np.abs(x.astype(np.float64))
    hi = np.clip(np.searchsorted(values, a, side="left"), 0, 0x7E)  # first value >= a
    lo = np.clip(hi - 1, 0, 0x7E)
    d_hi = values[hi] - a
    d_lo = a - values[lo]
    take_lo = (d_lo < d_hi) | ((d_lo == d_hi) & (lo % 2 == 0))
    code = np.where(take_lo, lo, hi)
    code = np.where(a >= values[0x7E], 0x7E, code)                  # saturate (also +-inf)
    code = np.where(np.isnan(a), 0x7F, code).astype(np.uint8)
    sign = np.signbit(x).astype(np.uint8) << 7
    return code | sign


def fp8_quantise(x, scale: float) -> np.ndarray:
    """Codes of fp16 values x for an fp8 cache with dequantisation scale
    `scale` (a stored code c stands for e4m3(c) * scale).  Reading (the pages
    keep fp16): in float32 arithmetic, code = e4m3_encode(fl32(x) * inv) with
    inv = fl32(1 / fl32(scale)) -- one reciprocal per cache, one product per
    element, each rounded to float32."""
    inv = np.float32(1.0) / np.float32(scale)
    return e4m3_encode(np.asarray(x).astype(np.float32) * inv)


# ---------------------------------------------------------------------------
# KV-size formula
# ---------------------------------------------------------------------------

def kv_bytes_per_token(num_layers: int, num_kv_heads: int, head_dim: int, bytes_per_elem: int) -> int:
    """KV-cache bytes per token = 2 (K and V) x layers x KV heads x head dim x
    bytes per element (deepsonar page, section 2.1)."""
    return 2 * num_layers * num_kv_heads * head_dim * bytes_per_elem


# ---------------------------------------------------------------------------
# Block allocator
# ---------------------------------------------------------------------------

class OracleError(Exception):
    def __init__(self, code: str):
        super().__init__(code)
        self.code = code


ZERO_HASH = bytes(32)


def block_hash(parent: bytes, tokens, extra_key: int) -> bytes:
    """Chained block hash: sha256(parent hash || token ids as little-endian
    int32 || extra key as little-endian uint64); parent = 32 zero bytes for a
    sequence's first block (deepsonar page section 2.4: hash of the parent
    block, the block's tokens and an extra key)."""
    data = parent + struct.pack("<%di" % len(tokens), *[int(t) for t in tokens]) + \
        struct.pack("<Q", int(extra_key) & (2 ** 64 - 1))
    return hashlib.sha256(data).digest()


class OracleAllocator:
    """Plain Python block allocator.

    * Blocks hold ``block_size`` tokens; a sequence's token t sits in logical
      block t // block_size at offset t % block_size; its slot number is
      physical_block * block_size + offset (the block-16 layout of the
      chester-dev.com page, section "PagedAttention transforme l'historique en
      blocs reutilisables": A -> blocks 7, 2, 19, 4).
    * A new block is taken only when the token to write starts a block, i.e.
      the previous block is full (allocation on demand, left to right).
    * The free queue hands out from its head and takes released blocks back at
      its tail.  Reading taken where the pages are silent: a released
      sequence's blocks are returned in table order, logical block 0 first.
    * ``fork`` shares every block of the parent with the child (reference count
      + 1 each).  Writing a token into a block whose count is above one first
      takes a fresh block, records the pair (shared, fresh) for the caller to
      copy, and drops the shared block's count by one (copy-on-write).
    * A call that runs out of blocks raises ``OracleError('OUT_OF_BLOCKS')``
      and leaves the state as it was.
    * With ``prefix_cache``: a full block whose tokens are known is hashed
      (``block_hash``, chained from its predecessor) and entered in a map
      unless the map already has that hash.  Released blocks keep their entry
      while free; a block taken from the queue head drops it.
      ``match_prefix`` starts a sequence by taking, in order, the cached
      blocks of its prompt's full blocks within all but the last token,
      stopping at the first miss.
    """

    def __init__(self, num_blocks: int, block_size: int, free_order=None, prefix_cache: bool = False):
        if num_blocks <= 0 or block_size <= 0:
            raise OracleError("INVALID_ARG")
        self.num_blocks = int(num_blocks)
        self.block_size = int(block_size)
        order = list(range(num_blocks)) if free_order is None else [int(b) for b in free_order]
        if sorted(order) != list(range(num_blocks)):
            raise OracleError("INVALID_ARG")
        self.free = OrderedDict((b, None) for b in order)   # head first
        self.ref = [0] * num_blocks
        self.seqs: dict = {}
        self.prefix_cache = bool(prefix_cache)
        self.hash_of: dict = {}       # block -> hash recorded for it
        self.cached: dict = {}        # hash -> block
        self.queries = 0
        self.hits = 0

    # -- free queue ---------------------------------------------------------
    def _pop_free(self):
        b, _ = self.free.popitem(last=False)
        h = self.hash_of.pop(b, None)
        if h is not None and self.cached.get(h) == b:
            del self.cached[h]
        return b

    # -- sequences --------------------------------------------------------
    def _new_seq(self):
        return {"len": 0, "blocks": [], "ids": [], "chain": [], "extra": 0}

    def add_seq(self, seq_id: int):
        if seq_id in self.seqs:
            raise OracleError("INVALID_ARG")
        self.seqs[seq_id] = self._new_seq()

    def _blocks_needed(self, seq, n):
        bs = self.block_size
        length = seq["len"]
        new_blocks = -(-(length + n) // bs) - (-(-length // bs))
        cow = 0
        if n > 0 and length % bs != 0 and self.ref[seq["blocks"][-1]] > 1:
            cow = 1
        return new_blocks + cow

    def append_tokens(self, seq_id: int, n: int):
        """Reserve slots for the next n tokens of a sequence.

        Returns (slots, pairs): slots[k] is the slot of token len+k; pairs is a
        list of (src_block, dst_block) copies that must run before the K/V of
        those tokens are written."""
        return self.append_batch([seq_id], [n])

    def append_batch(self, seq_ids, counts, token_ids=None):
        """Same as append_tokens for several sequences, in the order given.
        All-or-nothing: if the blocks needed by the whole call exceed the free
        queue, nothing changes.  ``token_ids`` (concatenated, sequence by
        sequence) lets completed blocks be hashed when prefix caching is on."""
        if len(seq_ids) != len(counts):
            raise OracleError("INVALID_ARG")
        for s, n in zip(seq_ids, counts):
            if s not in self.seqs or n < 0:
                raise OracleError("INVALID_ARG")
        if len(set(seq_ids)) != len(seq_ids):
            raise OracleError("INVALID_ARG")
        need = sum(self._blocks_needed(self.seqs[s], n) for s, n in zip(seq_ids, counts))
        if need > len(self.free):
            raise OracleError("OUT_OF_BLOCKS")
        bs = self.block_size
        slots, pairs = [], []
        w = 0
        for s, n in zip(seq_ids, counts):
            seq = self.seqs[s]
            if token_ids is None:
                seq["ids"] = None
            for _ in range(n):
                t = seq["len"]
                off = t % bs
                if off == 0:
                    b = self._pop_free()
                    self.ref[b] = 1
                    seq["blocks"].append(b)
                else:
                    tail = seq["blocks"][-1]
                    if self.ref[tail] > 1:
                        nb = self._pop_free()
                        self.ref[nb] = 1
                        self.ref[tail] -= 1
                        seq["blocks"][-1] = nb
                        pairs.append((tail, nb))
                slots.append(seq["blocks"][t // bs] * bs + off)
                if token_ids is not None and seq["ids"] is not None:
                    seq["ids"].append(int(token_ids[w]))
                w += 1
                seq["len"] = t + 1
                self._maybe_hash(seq, t)
        return slots, pairs

    def _maybe_hash(self, seq, t):
        bs = self.block_size
        if not self.prefix_cache or seq["ids"] is None or (t + 1) % bs != 0:
            return
        j = t // bs
        if len(seq["chain"]) != j:
            return
        parent = seq["chain"][j - 1] if j else ZERO_HASH
        h = block_hash(parent, seq["ids"][j * bs:(j + 1) * bs], seq["extra"])
        seq["chain"].append(h)
        b = seq["blocks"][j]
        if b not in self.hash_of:
            self.hash_of[b] = h
            self.cached.setdefault(h, b)

    def match_prefix(self, seq_id: int, tokens, extra_key: int = 0) -> int:
        """Start ``seq_id`` on a prompt; returns the tokens covered by cached blocks."""
        if not self.prefix_cache or seq_id in self.seqs:
            raise OracleError("INVALID_ARG")
        bs = self.block_size
        tokens = [int(x) for x in tokens]
        seq = self._new_seq()
        seq["extra"] = int(extra_key)
        candidates = (len(tokens) - 1) // bs if tokens else 0
        for j in range(candidates):
            parent = seq["chain"][j - 1] if j else ZERO_HASH
            h = block_hash(parent, tokens[j * bs:(j + 1) * bs], extra_key)
            self.queries += 1
            if h not in self.cached:
                break
            self.hits += 1
            b = self.cached[h]
            if b in self.free:
                del self.free[b]
            self.ref[b] += 1
            seq["blocks"].append(b)
            seq["chain"].append(h)
            seq["ids"].extend(tokens[j * bs:(j + 1) * bs])
            seq["len"] += bs
        self.seqs[seq_id] = seq
        return seq["len"]

    def fork(self, parent: int, child: int):
        if parent not in self.seqs or child in self.seqs:
            raise OracleError("INVALID_ARG")
        p = self.seqs[parent]
        for b in p["blocks"]:
            self.ref[b] += 1
        self.seqs[child] = {"len": p["len"], "blocks": list(p["blocks"]),
                            "ids": None if p["ids"] is None else list(p["ids"]),
                            "chain": list(p["chain"]), "extra": p["extra"]}

    def free_seq(self, seq_id: int):
        if seq_id not in self.seqs:
            raise OracleError("INVALID_ARG")
        seq = self.seqs[seq_id]
        uses: dict = {}
        for b in seq["blocks"]:
            uses[b] = uses.get(b, 0) + 1
            if uses[b] > self.ref[b]:
                raise OracleError("STATE")
        del self.seqs[seq_id]
        for b in seq["blocks"]:
            self.ref[b] -= 1
            if self.ref[b] == 0:
                self.free[b] = None

    # -- views --------------------------------------------------------------
    def block_table(self, seq_id: int):
        return list(self.seqs[seq_id]["blocks"])

    def seq_len(self, seq_id: int) -> int:
        return self.seqs[seq_id]["len"]

    def slot_of(self, seq_id: int, t: int) -> int:
        seq = self.seqs[seq_id]
        return seq["blocks"][t // self.block_size] * self.block_size + t % self.block_size

    def stats(self):
        used = sum(1 for r in self.ref if r > 0)
        shared = sum(1 for r in self.ref if r > 1)
        return {
            "num_blocks": self.num_blocks,
            "free_blocks": len(self.free),
            "used_blocks": used,
            "shared_blocks": shared,
            "num_seqs": len(self.seqs),
            "logical_tokens": sum(s["len"] for s in self.seqs.values()),
        }

    def prefix_stats(self):
        return {"cached_blocks": len(self.cached), "queries": self.queries, "hits": self.hits}

    def used_slot_mask(self):
        """Boolean [num_blocks, block_size]: True where some sequence holds a
        token.  Used by tests to poison every other slot."""
        mask = np.zeros((self.num_blocks, self.block_size), dtype=bool)
        for seq in self.seqs.values():
            for t in range(seq["len"]):
                mask[seq["blocks"][t // self.block_size], t % self.block_size] = True
        return mask

    def tables(self, seq_ids, max_blocks: int):
        """int32 [len(seq_ids)][max_blocks] block tables (unused entries -1)
        and int32 context lengths."""
        tab = np.full((len(seq_ids), max_blocks), -1, dtype=np.int32)
        lens = np.zeros(len(seq_ids), dtype=np.int32)
        for i, s in enumerate(seq_ids):
            blocks = self.seqs[s]["blocks"]
            tab[i, : len(blocks)] = blocks
            lens[i] = self.seqs[s]["len"]
        return tab, lens


# ---------------------------------------------------------------------------
# KV write and block copy
# ---------------------------------------------------------------------------

def kv_write(k_cache, v_cache, key, value, slot_mapping, block_size):
    """Return copies of the caches with token t's K/V rows stored at slot
    slot_mapping[t] (block slot // block_size, offset slot % block_size).
    Caches are indexed [block, kv_head, offset, dim]; key/value are
    [tokens, kv_heads, dim].  Negative slots are padding and are skipped."""
    kc, vc = k_cache.copy(), v_cache.copy()
    for t, slot in enumerate(np.asarray(slot_mapping).tolist()):
        if slot < 0:
            continue
        b, o = divmod(int(slot), block_size)
        kc[b, :, o, :] = key[t]
        vc[b, :, o, :] = value[t]
    return kc, vc


def kv_write_fp8(k_cache, v_cache, key, value, slot_mapping, block_size, k_scale, v_scale):
    """kv_write into caches of fp8 codes (uint8 [block, kv_head, offset, dim]):
    each new fp16 row is quantised with its cache's scale (``fp8_quantise``)."""
    return kv_write(k_cache, v_cache, fp8_quantise(key, k_scale), fp8_quantise(value, v_scale), slot_mapping,
                    block_size)


def block_copy(k_cache, v_cache, pairs):
    """Return copies of the caches where each dst block holds what its src
    block held before the call (all K and V of every kv head and offset)."""
    kc, vc = k_cache.copy(), v_cache.copy()
    for src, dst in np.asarray(pairs, dtype=np.int64).reshape(-1, 2).tolist():
        kc[dst] = k_cache[src]
        vc[dst] = v_cache[src]
    return kc, vc


# ---------------------------------------------------------------------------
# Decode attention (fp64, C)
# ---------------------------------------------------------------------------

def default_threads() -> int:
    try:
        return len(os.sched_getaffinity(0))
    except AttributeError:  # pragma: no cover
        return os.cpu_count() or 1


def _decode_call(split_tokens, query, k_cache, v_cache, block_tables, context_lens,
                 num_kv_heads, block_size, scale, threads, seq_range):
    lib = _load()
    q = np.ascontiguousarray(query).view(np.uint16)
    if q.ndim != 3:
        raise ValueError("query must be [num_seqs, num_heads, head_dim]")
    num_seqs, num_heads, head_dim = q.shape
    kc = np.asarray(k_cache).view(np.uint16)
    vc = np.asarray(v_cache).view(np.uint16)
    if kc.ndim != 4 or kc.strides != vc.strides or kc.shape != vc.shape:
        raise ValueError("caches must be 4-d [block, kv_head, offset, dim] views with equal strides")
    if kc.strides[3] != 2:
        raise ValueError("the dim axis of the caches must be unit-stride")
    if kc.shape[1] != num_kv_heads or kc.shape[2] != block_size or kc.shape[3] != head_dim:
        raise ValueError("cache shape does not match the arguments")
    sb, sh, st = (s // 2 for s in kc.strides[:3])
    tab = np.ascontiguousarray(block_tables, dtype=np.int32)
    lens = np.ascontiguousarray(context_lens, dtype=np.int32)
    max_blocks = tab.shape[1]
    out = np.zeros((num_seqs, num_heads, head_dim), dtype=np.float64)
    # pointers to the start of the (possibly strided) cache views
    kptr = kc.__array_interface__["data"][0]
    vptr = vc.__array_interface__["data"][0]
    lo, hi = seq_range if seq_range is not None else (0, num_seqs)
    threads = max(1, min(threads or default_threads(), hi - lo))

    def run(a, b):
        args = [out.ctypes.data, q.ctypes.data, kptr, vptr, tab.ctypes.data, lens.ctypes.data,
                num_seqs, num_heads, num_kv_heads, head_dim, block_size, max_blocks, sb, sh, st,
                float(scale)]
        if split_tokens is None:
            rc = lib.or_paged_decode(*args, a, b)
        else:
            rc = lib.or_paged_decode_split(*args, int(split_tokens), a, b)
        if rc != 0:
            raise RuntimeError("oracle decode failed")

    bounds = np.linspace(lo, hi, threads + 1).astype(int)
    if threads == 1:
        run(lo, hi)
    else:
        with ThreadPoolExecutor(max_workers=threads) as ex:
            list(ex.map(lambda ab: run(*ab), zip(bounds[:-1], bounds[1:])))
    return out


def paged_decode(query, k_cache, v_cache, block_tables, context_lens, num_kv_heads, block_size,
                 scale, threads=None, seq_range=None):
    """fp64 decode attention (see oracle.c).  Caches are [block, kv_head,
    offset, dim] numpy views (fp16 or their uint16 bits); any strides with a
    unit-stride dim axis.  Returns float64 [num_seqs, num_heads, head_dim];
    rows outside ``seq_range`` stay zero."""
    return _decode_call(None, query, k_cache, v_cache, block_tables, context_lens,
                        num_kv_heads, block_size, scale, threads, seq_range)


def paged_decode_split(query, k_cache, v_cache, block_tables, context_lens, num_kv_heads,
                       block_size, scale, partition_tokens, threads=None, seq_range=None):
    """fp64 split-context decode with the log-sum-exp merge (see oracle.c)."""
    return _decode_call(int(partition_tokens), query, k_cache, v_cache, block_tables, context_lens,
                        num_kv_heads, block_size, scale, threads, seq_range)


def paged_attention_causal(query, k_cache, v_cache, block_tables, context_lens, query_start, num_kv_heads,
                           block_size, scale, threads=None):
    """fp64 causal attention of query rows [num_query_tokens, Hq, D]: sequence
    i owns rows query_start[i] .. query_start[i+1] - 1, its last T_i context
    positions; row j of it sees positions 0 .. L_i - T_i + j."""
    lib = _load()
    q = np.ascontiguousarray(query).view(np.uint16)
    nq, num_heads, head_dim = q.shape
    kc = np.asarray(k_cache).view(np.uint16)
    vc = np.asarray(v_cache).view(np.uint16)
    if kc.ndim != 4 or kc.strides != vc.strides or kc.strides[3] != 2:
        raise ValueError("caches must be 4-d [block, kv_head, offset, dim] views with a unit-stride dim")
    sb, sh, st = (s // 2 for s in kc.strides[:3])
    tab = np.ascontiguousarray(block_tables, dtype=np.int32)
    lens = np.ascontiguousarray(context_lens, dtype=np.int32)
    qs = np.ascontiguousarray(query_start, dtype=np.int32)
    B = len(lens)
    if len(qs) != B + 1 or qs[-1] != nq:
        raise ValueError("query_start must have num_seqs + 1 entries ending at the query row count")
    out = np.zeros((nq, num_heads, head_dim), dtype=np.float64)
    kptr = kc.__array_interface__["data"][0]
    vptr = vc.__array_interface__["data"][0]
    threads = max(1, min(threads or default_threads(), B))

    def run(a, b):
        rc = lib.or_paged_attention_causal(out.ctypes.data, q.ctypes.data, kptr, vptr, tab.ctypes.data,
                                           lens.ctypes.data, qs.ctypes.data, B, num_heads, num_kv_heads, head_dim,
                                           block_size, tab.shape[1], sb, sh, st, float(scale), a, b)
        if rc != 0:
            raise RuntimeError("oracle causal attention failed")

    bounds = np.linspace(0, B, threads + 1).astype(int)
    with ThreadPoolExecutor(max_workers=threads) as ex:
        list(ex.map(lambda ab: run(*ab), zip(bounds[:-1], bounds[1:])))
    return out


def paged_attention_typed(query, k_cache, v_cache, block_tables, context_lens, query_start, num_kv_heads, block_size,
                          scale, kv_dtype, k_scale=1.0, v_scale=1.0, threads=None):
    """fp64 attention over caches of element type kv_dtype (KV_F16, KV_BF16
    with bf16 query rows, KV_FP8_E4M3 with fp16 query rows): element e of the
    K cache stands for value(e) * k_scale, of the V cache for value(e) *
    v_scale.  query_start None: one query row per sequence (the decode, a zero
    row for an empty context); else the causal multi-token form.  query and
    the caches are arrays of 16-bit patterns (uint16/float16) or, for fp8,
    uint8 codes; the caches are 4-d [block, kv_head, offset, dim] views."""
    lib = _load()
    q = np.ascontiguousarray(query)
    q_dtype = KV_BF16 if kv_dtype == KV_BF16 else KV_F16
    nq, num_heads, head_dim = q.shape
    kc = np.asarray(k_cache)
    vc = np.asarray(v_cache)
    esz = 1 if kv_dtype == KV_FP8_E4M3 else 2
    if kc.ndim != 4 or kc.strides != vc.strides or kc.strides[3] != esz or kc.itemsize != esz:
        raise ValueError("caches must be 4-d [block, kv_head, offset, dim] views with a unit-stride dim")
    sb, sh, st = (s // esz for s in kc.strides[:3])
    tab = np.ascontiguousarray(block_tables, dtype=np.int32)
    lens = np.ascontiguousarray(context_lens, dtype=np.int32)
    B = len(lens)
    if query_start is None:
        qs, qs_ptr = None, None
        if nq != B:
            raise ValueError("one query row per sequence")
    else:
        qs = np.ascontiguousarray(query_start, dtype=np.int32)
        if len(qs) != B + 1 or qs[-1] != nq:
            raise ValueError("query_start must have num_seqs + 1 entries ending at the query row count")
        qs_ptr = qs.ctypes.data
    out = np.zeros((nq, num_heads, head_dim), dtype=np.float64)
    kptr = kc.__array_interface__["data"][0]
    vptr = vc.__array_interface__["data"][0]
    threads = max(1, min(threads or default_threads(), B))

    def run(a, b):
        rc = lib.or_paged_attention_typed(out.ctypes.data, q.ctypes.data, q_dtype, kptr, vptr, int(kv_dtype),
                                          float(k_scale), float(v_scale), tab.ctypes.data, lens.ctypes.data, qs_ptr,
                                          B, num_heads, num_kv_heads, head_dim, block_size, tab.shape[1], sb, sh, st,
                                          float(scale), a, b)
        if rc != 0:
            raise RuntimeError("oracle typed attention failed")

    bounds = np.linspace(0, B, threads + 1).astype(int)
    with ThreadPoolExecutor(max_workers=threads) as ex:
        list(ex.map(lambda ab: run(*ab), zip(bounds[:-1], bounds[1:])))
    return out
