"""Seeded synthetic workloads for the paged decode path.

This module draws inputs only: shapes, context lengths, the order in which the
free queue hands out physical blocks, and fp16 values.  It computes nothing
the method computes (no slots, no block tables, no attention); the tests,
the benchmark and the oracle all build those from what is drawn here.

Every array comes from NumPy's PCG64 seeded with ``1000 + k`` (k = the
workload's index below), values N(0, 1) (Box-Muller over float32
uniforms) rounded to fp16 (round to nearest even).  Each array has its own child stream of that seed (and each chunk of
2^22 values its own grandchild stream), so any one of them can be drawn
without drawing the others, by any number of threads.

Workloads (shaped like the pages' examples; sizes named by what they are):

* ``tiny``    -- 4 sequences, 4 query / 2 KV heads, head_dim 64, block 16,
  context U{1..100}, a pool of 64 blocks handed out in a random order.
* ``mha7b``   -- 64 sequences, 32 = 32 heads, head_dim 128, block 16, context
  U{512..2048}, one new token per sequence written this step.
* ``gqa72b``  -- 100 sequences, 64 query / 8 KV heads, head_dim 128, block 16,
  context 8192 each (the 80-layer, 8-KV-head, dim-128 model of the deepsonar
  page, section 2.1: 8k context, 100 concurrent requests).
* ``mix``     -- 256 sequences, 32 / 8 heads, head_dim 128, block 16, context
  log-uniform in [64, 32768]; sequences 0, 1, 2 are set to 600, 12000 and
  18000 tokens (the chat / legal-summary sizes of the chester-dev.com page,
  first section).  One new token per sequence.
* ``cow16`` / ``cow32`` -- 32 prompts x 8 samples (parallel sampling, deepsonar
  page section 2.3), 32 / 8 heads, head_dim 128, block 16 or 32; a 2048-token
  prompt shared by all 8 samples (``prompt_extra`` > 0 adds 1..block-1 tokens
  so the shared tail block is partial), then U{0..512} private tokens per
  sample already generated, plus this step's token.
* ``spec72b`` -- the gqa72b shapes with 4 new tokens per sequence in the step
  (speculative candidates, deepsonar page section 2.5): 100 sequences of 8192
  positions, the last 4 computed together.
* ``chunked`` -- 64 sequences, 32 / 8 heads, head_dim 128, block 16, in one
  step (deepsonar page section 2.5: prefill chunks mixed into the decode
  batch): sequence 0 computes the last 2048-token chunk of a 12000-token
  prompt, sequence 1 a whole 600-token prompt (the chester-dev.com page's
  legal-summary and chat sizes), sequences 2..63 one decode token each over
  log-uniform [64, 32768] contexts.

Steps with several new tokens per sequence also draw ``query_multi``: one
query row per new token, sequences in order.
"""
from __future__ import annotations

import math
import os
from concurrent.futures import ThreadPoolExecutor
from dataclasses import dataclass, field

import numpy as np

WORKLOADS = ("tiny", "mha7b", "gqa72b", "mix", "cow16", "cow32", "spec72b", "chunked")

# child-stream indices, one per drawn array
_S_LENGTHS, _S_ORDER, _S_QUERY, _S_KPOOL, _S_VPOOL, _S_NEWK, _S_NEWV, _S_EXTRA, _S_QMULTI = range(9)


_CHUNK = 1 << 22     # values per independently seeded chunk


def _rng(seed: int, stream: int, chunk: int | None = None) -> np.random.Generator:
    key = (stream,) if chunk is None else (stream, chunk)
    return np.random.Generator(np.random.PCG64(np.random.SeedSequence(seed, spawn_key=key)))


def _normal_chunk(rng: np.random.Generator, n: int) -> np.ndarray:
    """n N(0, 1) float32 values by the Box-Muller transform (Box and Muller,
    1958): from uniforms u1 in (0, 1] and u2 in [0, 1), r = sqrt(-2 ln u1)
    gives the pair r cos(2 pi u2), r sin(2 pi u2)."""
    m = (n + 1) // 2
    u1 = np.float32(1.0) - rng.random(m, dtype=np.float32)
    ang = rng.random(m, dtype=np.float32) * np.float32(2.0 * np.pi)
    r = np.sqrt(np.float32(-2.0) * np.log(u1))
    out = np.empty(2 * m, dtype=np.float32)
    np.multiply(r, np.cos(ang), out=out[0::2])
    np.multiply(r, np.sin(ang), out=out[1::2])
    return out[:n]


def normal_fp16(seed: int, stream: int, shape) -> np.ndarray:
    """N(0, 1) values rounded to fp16.  Chunk c of _CHUNK values is drawn from
    child stream (stream, c) of ``seed``, so the result does not depend on how
    many threads draw it."""
    n = int(np.prod(shape))
    out = np.empty(n, dtype=np.float16)

    def fill(c):
        a = c * _CHUNK
        b = min(n, a + _CHUNK)
        out[a:b] = _normal_chunk(_rng(seed, stream, c), b - a).astype(np.float16)

    chunks = range(-(-n // _CHUNK))
    if n <= _CHUNK:
        for c in chunks:
            fill(c)
    else:
        with ThreadPoolExecutor(max_workers=min(32, os.cpu_count() or 1)) as ex:
            list(ex.map(fill, chunks))
    return out.reshape(shape)


@dataclass
class Workload:
    name: str
    seed: int
    num_seqs: int
    num_heads: int
    num_kv_heads: int
    head_dim: int
    block_size: int
    num_blocks: int
    context_lens: np.ndarray          # int32 [num_seqs]: tokens attended this step, new token included
    history_lens: np.ndarray          # int32 [num_seqs]: tokens already in the cache before this step
    free_order: np.ndarray            # int32 [num_blocks]: order in which free blocks are handed out
    # parallel sampling structure (cow workloads only)
    num_prompts: int = 0
    samples_per_prompt: int = 0
    prompt_len: int = 0
    divergent: np.ndarray | None = None   # int32 [num_seqs]: private tokens generated before this step
    # several new tokens per sequence are computed in this step (each written
    # token is a query row); otherwise one query per sequence (the decode)
    multi: bool = False
    _cache: dict = field(default_factory=dict, repr=False)

    @property
    def group(self) -> int:
        return self.num_heads // self.num_kv_heads

    @property
    def scale(self) -> float:
        return 1.0 / math.sqrt(self.head_dim)

    @property
    def new_counts(self) -> np.ndarray:
        """Tokens written into the cache by this step, per sequence."""
        return (self.context_lens - self.history_lens).astype(np.int32)

    @property
    def num_new_tokens(self) -> int:
        return int(self.new_counts.sum())

    @property
    def max_context_len(self) -> int:
        return int(self.context_lens.max()) if self.num_seqs else 0

    @property
    def max_blocks_per_seq(self) -> int:
        return max(1, -(-self.max_context_len // self.block_size))

    def _get(self, key, stream, shape):
        if key not in self._cache:
            self._cache[key] = normal_fp16(self.seed, stream, shape)
        return self._cache[key]

    @property
    def query(self) -> np.ndarray:
        """fp16 [num_seqs, num_heads, head_dim]"""
        return self._get("q", _S_QUERY, (self.num_seqs, self.num_heads, self.head_dim))

    @property
    def query_multi(self) -> np.ndarray:
        """fp16 [num_new_tokens, num_heads, head_dim]: a query row for every
        token written this step, sequences in order."""
        return self._get("qm", _S_QMULTI, (self.num_new_tokens, self.num_heads, self.head_dim))

    @property
    def query_start(self) -> np.ndarray:
        """int32 [num_seqs + 1]: first query_multi row of every sequence."""
        return np.concatenate([[0], np.cumsum(self.new_counts)]).astype(np.int32)

    @property
    def k_pool(self) -> np.ndarray:
        """fp16 [num_blocks, num_kv_heads, block_size, head_dim]: initial K content of every
        physical slot (the history already in the cache)."""
        return self._get("k", _S_KPOOL, (self.num_blocks, self.num_kv_heads, self.block_size, self.head_dim))

    @property
    def v_pool(self) -> np.ndarray:
        return self._get("v", _S_VPOOL, (self.num_blocks, self.num_kv_heads, self.block_size, self.head_dim))

    @property
    def new_key(self) -> np.ndarray:
        """fp16 [num_new_tokens, num_kv_heads, head_dim], sequences in order."""
        return self._get("nk", _S_NEWK, (self.num_new_tokens, self.num_kv_heads, self.head_dim))

    @property
    def new_value(self) -> np.ndarray:
        return self._get("nv", _S_NEWV, (self.num_new_tokens, self.num_kv_heads, self.head_dim))

    def drop_arrays(self):
        self._cache.clear()


def _order(seed, num_blocks):
    return _rng(seed, _S_ORDER).permutation(num_blocks).astype(np.int32)


def _spare_pool(context_lens, block_size, spare):
    return int(sum(-(-int(L) // block_size) for L in context_lens)) + spare


def custom(name="custom", seed=7, num_seqs=4, num_heads=4, num_kv_heads=2, head_dim=64, block_size=16,
           context_lens=None, new_tokens=1, num_blocks=None, spare_blocks=None, permute=True, multi=None) -> Workload:
    """A workload with given shapes and lengths (edge cases in tests);
    new_tokens: tokens written this step, one count or one per sequence;
    multi: each of them is a query row (default: when any count is not 1)."""
    lens = np.asarray(context_lens if context_lens is not None else [1] * num_seqs, dtype=np.int32)
    hist = np.maximum(lens - np.asarray(new_tokens, dtype=np.int32), 0).astype(np.int32)
    spare = num_seqs if spare_blocks is None else spare_blocks
    nb = num_blocks if num_blocks is not None else max(1, _spare_pool(lens, block_size, spare))
    order = _order(seed, nb) if permute else np.arange(nb, dtype=np.int32)
    if multi is None:
        multi = bool(np.any(np.asarray(new_tokens) != 1))
    return Workload(name, seed, len(lens), num_heads, num_kv_heads, head_dim, block_size, nb, lens, hist, order,
                    multi=bool(multi))


def make(name: str, prompt_extra: int | None = None, spec_tokens: int = 4) -> Workload:
    """The named workload.  For cow16/cow32, ``prompt_extra`` = None draws the
    partial-tail variant's extra tokens r in 1..block-1 from the seed;
    ``prompt_extra=0`` gives the whole-block 2048-token prompt.  For spec72b,
    ``spec_tokens`` is the number of new (speculative) tokens per sequence."""
    k = WORKLOADS.index(name)
    seed = 1000 + k
    rl = _rng(seed, _S_LENGTHS)
    if name == "tiny":
        lens = rl.integers(1, 100, size=4, endpoint=True).astype(np.int32)
        return Workload(name, seed, 4, 4, 2, 64, 16, 64, lens, lens - 1, _order(seed, 64))
    if name == "mha7b":
        lens = rl.integers(512, 2048, size=64, endpoint=True).astype(np.int32)
        nb = _spare_pool(lens, 16, 64)
        return Workload(name, seed, 64, 32, 32, 128, 16, nb, lens, lens - 1, _order(seed, nb))
    if name == "gqa72b":
        lens = np.full(100, 8192, dtype=np.int32)
        nb = _spare_pool(lens, 16, 100)
        return Workload(name, seed, 100, 64, 8, 128, 16, nb, lens, lens - 1, _order(seed, nb))
    if name == "mix":
        u = rl.uniform(math.log(64), math.log(32768), size=256)
        lens = np.rint(np.exp(u)).astype(np.int32)
        lens[:3] = (600, 12000, 18000)
        nb = _spare_pool(lens, 16, 256)
        return Workload(name, seed, 256, 32, 8, 128, 16, nb, lens, lens - 1, _order(seed, nb))
    if name in ("cow16", "cow32"):
        bs = 16 if name == "cow16" else 32
        prompts, samples = 32, 8
        if prompt_extra is None:
            prompt_extra = int(_rng(seed, _S_EXTRA).integers(1, bs - 1, endpoint=True))
        plen = 2048 + int(prompt_extra)
        div = rl.integers(0, 512, size=prompts * samples, endpoint=True).astype(np.int32)
        lens = (plen + div + 1).astype(np.int32)
        hist = np.full(prompts * samples, plen, dtype=np.int32)
        # blocks: one copy of each prompt, every sample's private tail, one copy per CoW, spare
        nb = prompts * (-(-plen // bs)) + int(sum(-(-(int(d) + 1) // bs) + 1 for d in div)) + prompts * samples
        w = Workload(name, seed, prompts * samples, 32, 8, 128, bs, nb, lens, hist, _order(seed, nb),
                     num_prompts=prompts, samples_per_prompt=samples, prompt_len=plen, divergent=div)
        return w
    if name == "spec72b":
        lens = np.full(100, 8192, dtype=np.int32)
        nb = _spare_pool(lens, 16, 100)
        return Workload(name, seed, 100, 64, 8, 128, 16, nb, lens, lens - int(spec_tokens), _order(seed, nb),
                        multi=True)
    if name == "chunked":
        u = rl.uniform(math.log(64), math.log(32768), size=64)
        lens = np.rint(np.exp(u)).astype(np.int32)
        lens[:2] = (12000, 600)
        hist = lens - 1
        hist[:2] = (12000 - 2048, 0)
        nb = _spare_pool(lens, 16, 64)
        return Workload(name, seed, 64, 32, 8, 128, 16, nb, lens, hist.astype(np.int32), _order(seed, nb),
                        multi=True)
    raise KeyError(name)
