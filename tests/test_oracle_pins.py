"""Pins for the oracle: what the pages and the mathematics fix, independent of
the oracle's own code.  CPU only.

* every binary16 bit pattern converts as NumPy's independent float16 says;
* the KV-size formula reproduces the deepsonar page's printed numbers
  (section 2.1);
* the paged decode equals a NumPy brute force over contiguous arrays that this
  file builds itself (no block table involved), for MHA and GQA;
* the output does not change, bit for bit, when the physical placement, the
  block size or the cache layout changes;
* closed forms: one token gives its V row; a zero query or identical keys give
  the mean of V; a score boosted by 64 selects its V row; zero length gives 0;
* the split-context form with the log-sum-exp merge equals the unsplit form;
* the multi-token causal form equals a masked brute force and, with one token
  per sequence, the decode;
* bf16 and fp8 E4M3 elements decode to the values their formats define
  (every bf16 pattern through float32, the E4M3 values of the OCP definition),
  E4M3 rounding takes ties to the even code and saturates at 448, and the
  typed attention equals a brute force over the decoded values, with the K
  scale on the scores and the V scale on the output.
"""
import json
import math
import os

import numpy as np
import pytest

import oracle
from paged_kv_cache_12_gb300 import workloads

RNG = np.random.default_rng(12345)


def rand_fp16(*shape, rng=RNG):
    return rng.standard_normal(shape).astype(np.float16)


def page_sequences(Ks, Vs, block_size, rng, num_blocks=None, layout="bhod"):
    """Place each sequence's contiguous K/V [L, Hkv, D] into a paged cache at
    randomly chosen physical blocks.  Returns (k_cache, v_cache, tables, lens)
    with caches as [block, kv_head, offset, dim] views of the chosen layout;
    every slot that holds no token is NaN."""
    hkv, d = Ks[0].shape[1], Ks[0].shape[2]
    need = sum(-(-len(k) // block_size) for k in Ks)
    nb = num_blocks or need + 3
    phys = rng.permutation(nb)[:need]
    if layout == "bhod":
        kc = np.full((nb, hkv, block_size, d), np.nan, dtype=np.float16)
        vc = np.full_like(kc, np.nan)
        kview, vview = kc, vc
    else:  # block, offset, kv_head, dim storage; viewed as block, kv_head, offset, dim
        kc = np.full((nb, block_size, hkv, d), np.nan, dtype=np.float16)
        vc = np.full_like(kc, np.nan)
        kview, vview = kc.transpose(0, 2, 1, 3), vc.transpose(0, 2, 1, 3)
    maxb = max(1, max(-(-len(k) // block_size) for k in Ks))
    tables = np.full((len(Ks), maxb), -1, dtype=np.int32)
    lens = np.array([len(k) for k in Ks], dtype=np.int32)
    j = 0
    for i, (K, V) in enumerate(zip(Ks, Vs)):
        for lb in range(-(-len(K) // block_size)):
            tables[i, lb] = phys[j]
            t0, t1 = lb * block_size, min(len(K), (lb + 1) * block_size)
            kview[phys[j], :, : t1 - t0, :] = K[t0:t1].transpose(1, 0, 2)
            vview[phys[j], :, : t1 - t0, :] = V[t0:t1].transpose(1, 0, 2)
            j += 1
    return kview, vview, tables, lens


def brute_force(q, Ks, Vs, num_kv_heads, scale):
    """softmax(q K^T * scale) V per sequence and head, NumPy fp64, contiguous."""
    B, H, D = q.shape
    G = H // num_kv_heads
    out = np.zeros((B, H, D))
    for i in range(B):
        K = Ks[i].astype(np.float64)
        V = Vs[i].astype(np.float64)
        if len(K) == 0:
            continue
        for h in range(H):
            s = scale * (K[:, h // G, :] @ q[i, h].astype(np.float64))
            w = np.exp(s - s.max())
            w /= w.sum()
            out[i, h] = w @ V[:, h // G, :]
    return out


def make_case(lens, H, Hkv, D, rng=RNG):
    q = rand_fp16(len(lens), H, D, rng=rng)
    Ks = [rand_fp16(L, Hkv, D, rng=rng) for L in lens]
    Vs = [rand_fp16(L, Hkv, D, rng=rng) for L in lens]
    return q, Ks, Vs


# ---------------------------------------------------------------------------

def test_half_to_double_every_bit_pattern():
    bits = np.arange(1 << 16, dtype=np.uint32)
    ref = bits.astype(np.uint16).view(np.float16).astype(np.float64)
    got = np.array([oracle.half_to_double(int(b)) for b in bits])
    nan = np.isnan(ref)
    assert np.array_equal(np.isnan(got), nan)
    assert np.array_equal(got[~nan], ref[~nan])
    # a few values fixed by the binary16 format itself
    assert oracle.half_to_double(0x3C00) == 1.0
    assert oracle.half_to_double(0xC000) == -2.0
    assert oracle.half_to_double(0x7BFF) == 65504.0
    assert oracle.half_to_double(0x0001) == 2.0 ** -24
    assert oracle.half_to_double(0x7C00) == math.inf


def test_kv_size_formula_matches_page(golden_dir):
    g = json.load(open(os.path.join(golden_dir, "kv_size_deepsonar_s2_1.json")))
    per_tok = oracle.kv_bytes_per_token(g["layers"], g["kv_heads"], g["head_dim"], g["bytes_per_elem"])
    assert per_tok == g["bytes_per_token"] == 327680
    assert per_tok * g["context_tokens"] == g["bytes_per_request_gib"] * 2 ** 30
    assert per_tok * g["context_tokens"] * g["requests"] == g["bytes_all_requests_gib"] * 2 ** 30
    # per layer and token, the figure the byte accounting of one decode layer uses
    assert oracle.kv_bytes_per_token(1, 8, 128, 2) == 4096
    # without GQA every one of the 64 query heads would need its own KV head
    mha = oracle.kv_bytes_per_token(g["layers"], g["query_heads"], g["head_dim"], g["bytes_per_elem"])
    assert mha == g["mha_factor"] * per_tok


@pytest.mark.parametrize("H,Hkv,D,bs", [(4, 4, 64, 16), (8, 2, 64, 8), (16, 2, 128, 32), (6, 3, 32, 4)])
def test_decode_equals_bruteforce(H, Hkv, D, bs):
    lens = [1, 5, bs, bs + 1, 3 * bs - 1, 97]
    q, Ks, Vs = make_case(lens, H, Hkv, D)
    kc, vc, tab, ln = page_sequences(Ks, Vs, bs, RNG)
    scale = 1.0 / math.sqrt(D)
    got = oracle.paged_decode(q, kc, vc, tab, ln, Hkv, bs, scale, threads=2)
    ref = brute_force(q, Ks, Vs, Hkv, scale)
    assert np.max(np.abs(got - ref)) <= 1e-12


def test_gqa_grouping_is_contiguous():
    # heads 0,1 read kv head 0; heads 2,3 read kv head 1 (G = 2).  Make the two
    # kv heads' V constant and different, so each output row shows which it read.
    L, Hkv, D = 9, 2, 16
    q = rand_fp16(1, 4, D)
    K = rand_fp16(L, Hkv, D)
    V = np.zeros((L, Hkv, D), dtype=np.float16)
    V[:, 0, :] = 1.0
    V[:, 1, :] = -3.0
    kc, vc, tab, ln = page_sequences([K], [V], 4, RNG)
    out = oracle.paged_decode(q, kc, vc, tab, ln, Hkv, 4, 0.25)
    assert np.allclose(out[0, :2], 1.0, atol=1e-12)
    assert np.allclose(out[0, 2:], -3.0, atol=1e-12)


def test_invariant_under_physical_placement():
    lens = [33, 1, 70, 16]
    q, Ks, Vs = make_case(lens, 4, 2, 64)
    outs = []
    for seed in (1, 2, 3):
        kc, vc, tab, ln = page_sequences(Ks, Vs, 16, np.random.default_rng(seed), num_blocks=40)
        outs.append(oracle.paged_decode(q, kc, vc, tab, ln, 2, 16, 0.125))
    assert np.array_equal(outs[0], outs[1]) and np.array_equal(outs[0], outs[2])


def test_invariant_under_block_size_and_layout():
    lens = [100, 7, 64, 65]
    q, Ks, Vs = make_case(lens, 8, 2, 64)
    outs = []
    for bs in (8, 16, 32):
        for layout in ("bhod", "bohd"):
            kc, vc, tab, ln = page_sequences(Ks, Vs, bs, RNG, layout=layout)
            outs.append(oracle.paged_decode(q, kc, vc, tab, ln, 2, bs, 0.125))
    for o in outs[1:]:
        assert np.array_equal(outs[0], o)


def test_closed_forms():
    D, Hkv, H, bs = 64, 2, 4, 16
    scale = 1.0 / 8.0
    # one token: the output is that token's V row, exactly
    q, Ks, Vs = make_case([1], H, Hkv, D)
    kc, vc, tab, ln = page_sequences(Ks, Vs, bs, RNG)
    out = oracle.paged_decode(q, kc, vc, tab, ln, Hkv, bs, scale)
    for h in range(H):
        assert np.array_equal(out[0, h], Vs[0][0, h // 2].astype(np.float64))
    # zero query: uniform weights, the mean of V
    q, Ks, Vs = make_case([37], H, Hkv, D)
    q[:] = 0
    kc, vc, tab, ln = page_sequences(Ks, Vs, bs, RNG)
    out = oracle.paged_decode(q, kc, vc, tab, ln, Hkv, bs, scale)
    for h in range(H):
        assert np.max(np.abs(out[0, h] - Vs[0][:, h // 2].astype(np.float64).mean(0))) < 1e-13
    # identical keys: also the mean of V
    q, Ks, Vs = make_case([23], H, Hkv, D)
    Ks[0][:] = Ks[0][0]
    kc, vc, tab, ln = page_sequences(Ks, Vs, bs, RNG)
    out = oracle.paged_decode(q, kc, vc, tab, ln, Hkv, bs, scale)
    for h in range(H):
        assert np.max(np.abs(out[0, h] - Vs[0][:, h // 2].astype(np.float64).mean(0))) < 1e-13
    # one key scores 64 above all others: its V row, to within e^-64
    L, star = 50, 31
    q = np.zeros((1, H, D), dtype=np.float16)
    q[0, :, 0] = 8.0
    K = np.zeros((L, Hkv, D), dtype=np.float16)
    K[:, :, 1:] = rand_fp16(L, Hkv, D - 1)
    K[star, :, 0] = 64.0          # score = scale * 8 * 64 = 64; every other score is 0
    V = rand_fp16(L, Hkv, D)
    kc, vc, tab, ln = page_sequences([K], [V], bs, RNG)
    out = oracle.paged_decode(q, kc, vc, tab, ln, Hkv, bs, scale)
    for h in range(H):
        assert np.max(np.abs(out[0, h] - V[star, h // 2].astype(np.float64))) < 1e-12
    # zero length: a zero row
    q, Ks, Vs = make_case([5, 0], H, Hkv, D)
    kc, vc, tab, ln = page_sequences(Ks, Vs, bs, RNG)
    out = oracle.paged_decode(q, kc, vc, tab, ln, Hkv, bs, scale)
    assert np.array_equal(out[1], np.zeros((H, D)))


def test_mha_is_group_of_one():
    # G = 1 reduces to standard multi-head attention: head h reads kv head h.
    lens = [19, 40]
    q, Ks, Vs = make_case(lens, 3, 3, 32)
    kc, vc, tab, ln = page_sequences(Ks, Vs, 8, RNG)
    out = oracle.paged_decode(q, kc, vc, tab, ln, 3, 8, 0.3)
    for i, L in enumerate(lens):
        for h in range(3):
            K = Ks[i][:, h, :].astype(np.float64)
            V = Vs[i][:, h, :].astype(np.float64)
            s = 0.3 * K @ q[i, h].astype(np.float64)
            p = np.exp(s - s.max()) / np.exp(s - s.max()).sum()
            assert np.max(np.abs(out[i, h] - p @ V)) < 1e-12


@pytest.mark.parametrize("part", [1, 7, 16, 100, 512])
def test_split_merge_identity(part):
    lens = [1, 15, 16, 17, 250, 513]
    q, Ks, Vs = make_case(lens, 4, 2, 64)
    kc, vc, tab, ln = page_sequences(Ks, Vs, 16, RNG)
    a = oracle.paged_decode(q, kc, vc, tab, ln, 2, 16, 0.125)
    b = oracle.paged_decode_split(q, kc, vc, tab, ln, 2, 16, 0.125, part)
    assert np.max(np.abs(a - b)) <= 1e-12


def test_decode_threads_and_ranges_agree():
    w = workloads.make("tiny")
    rng = np.random.default_rng(5)
    q, Ks, Vs = make_case(list(w.context_lens), 4, 2, 64, rng=rng)
    kc, vc, tab, ln = page_sequences(Ks, Vs, 16, rng)
    one = oracle.paged_decode(q, kc, vc, tab, ln, 2, 16, w.scale, threads=1)
    many = oracle.paged_decode(q, kc, vc, tab, ln, 2, 16, w.scale, threads=4)
    assert np.array_equal(one, many)
    part = oracle.paged_decode(q, kc, vc, tab, ln, 2, 16, w.scale, seq_range=(1, 3))
    assert np.array_equal(part[1:3], one[1:3]) and not part[0].any() and not part[3].any()


def test_kv_write_and_block_copy_by_hand():
    kc = np.arange(3 * 2 * 4 * 2, dtype=np.float16).reshape(3, 2, 4, 2)
    vc = -kc
    key = np.array([[[100, 101], [102, 103]], [[200, 201], [202, 203]]], dtype=np.float16)
    val = -key
    # token 0 -> slot 5 = block 1 offset 1; token 1 is padding
    k2, v2 = oracle.kv_write(kc, vc, key, val, [5, -1], 4)
    exp_k = kc.copy()
    exp_k[1, 0, 1] = [100, 101]
    exp_k[1, 1, 1] = [102, 103]
    assert np.array_equal(k2, exp_k) and np.array_equal(v2, -exp_k)
    assert np.array_equal(kc, np.arange(48, dtype=np.float16).reshape(3, 2, 4, 2))  # input untouched
    # copy block 0 -> 2 and 0 -> 1: both destinations get block 0's old content
    k3, v3 = oracle.block_copy(kc, vc, [(0, 2), (0, 1)])
    assert np.array_equal(k3[1], kc[0]) and np.array_equal(k3[2], kc[0]) and np.array_equal(k3[0], kc[0])
    assert np.array_equal(v3[2], vc[0])


def test_causal_attention_pins():
    """Multi-token causal attention: one query token per sequence is the
    decode; several equal a brute force with the causal mask over contiguous
    arrays; the last query token of a chunk sees the whole context."""
    H, Hkv, D, bs = 8, 2, 64, 16
    lens = [1, 40, 97, 130, 16]
    T = [1, 3, 7, 0, 16]
    q_all, Ks, Vs = make_case(lens, H, Hkv, D)
    kc, vc, tab, ln = page_sequences(Ks, Vs, bs, RNG)
    qs = np.concatenate([[0], np.cumsum(T)]).astype(np.int32)
    query = rand_fp16(int(qs[-1]), H, D)
    scale = 0.125
    got = oracle.paged_attention_causal(query, kc, vc, tab, ln, qs, Hkv, bs, scale, threads=2)
    for i, (L, t) in enumerate(zip(lens, T)):
        K = Ks[i].astype(np.float64)
        V = Vs[i].astype(np.float64)
        for j in range(t):
            visible = L - t + j + 1
            for h in range(H):
                s = scale * (K[:visible, h // 4, :] @ query[qs[i] + j, h].astype(np.float64))
                p = np.exp(s - s.max())
                p /= p.sum()
                assert np.max(np.abs(got[qs[i] + j, h] - p @ V[:visible, h // 4, :])) < 1e-12
    # one token per sequence: exactly the decode oracle
    qs1 = np.arange(len(lens) + 1, dtype=np.int32)
    q1 = rand_fp16(len(lens), H, D)
    a = oracle.paged_attention_causal(q1, kc, vc, tab, ln, qs1, Hkv, bs, scale)
    b = oracle.paged_decode(q1, kc, vc, tab, ln, Hkv, bs, scale)
    assert np.array_equal(a, b)


# ------------------------------------------------- bf16 and fp8 E4M3 caches

def test_bf16_every_bit_pattern():
    # bfloat16 is the top half of an IEEE binary32: reinterpret through float32
    bits = np.arange(1 << 16, dtype=np.uint32)
    with np.errstate(invalid="ignore"):          # signalling NaN patterns
        ref = (bits << 16).view(np.float32).astype(np.float64)
    got = np.array([oracle.bf16_to_double(int(b)) for b in bits])
    nan = np.isnan(ref)
    assert np.array_equal(np.isnan(got), nan) and np.array_equal(got[~nan], ref[~nan])
    assert oracle.bf16_to_double(0x3F80) == 1.0 and oracle.bf16_to_double(0xC000) == -2.0
    assert oracle.bf16_to_double(0x0001) == 2.0 ** -133 and oracle.bf16_to_double(0x7F80) == math.inf
    assert oracle.bf16_to_double(0x7F7F) == (2 - 2 ** -7) * 2.0 ** 127


def test_e4m3_values_of_the_format():
    v = oracle.e4m3_to_double
    # values the OCP FP8 E4M3 definition fixes (S.EEEE.MMM, bias 7, no infinities)
    assert v(0x38) == 1.0 and v(0xB8) == -1.0 and v(0x40) == 2.0 and v(0x3C) == 1.5
    assert v(0x7E) == 448.0 and v(0xFE) == -448.0                   # largest finite: S.1111.110
    assert v(0x08) == 2.0 ** -6 and v(0x07) == 0.875 * 2.0 ** -6    # smallest normal, largest subnormal
    assert v(0x01) == 2.0 ** -9 and v(0x00) == 0.0                  # smallest subnormal
    assert math.copysign(1.0, v(0x80)) == -1.0 and v(0x80) == 0.0
    assert v(0x77) == 240.0 and v(0x78) == 256.0 and v(0x7D) == 416.0
    assert math.isnan(v(0x7F)) and math.isnan(v(0xFF))
    vals = [v(c) for c in range(0x7F)]
    assert all(b > a for a, b in zip(vals, vals[1:]))                # codes 0 .. 0x7E increase
    assert all(v(0x80 | c) == -v(c) for c in range(1, 0x7F))


def test_e4m3_rounding_ties_and_saturation():
    enc = lambda x: int(oracle.e4m3_encode(np.float32(x)))
    assert enc(1.0) == 0x38 and enc(-1.0) == 0xB8 and enc(448.0) == 0x7E and enc(-448.0) == 0xFE
    for big in (449.0, 464.0, 500.0, 1e6, np.inf):
        assert enc(big) == 0x7E and enc(-big) == 0xFE
    assert enc(np.nan) == 0x7F
    assert enc(0.0) == 0x00 and enc(-0.0) == 0x80
    # ties go to the even code
    assert enc(2.0 ** -10) == 0x00            # halfway between 0 and 2^-9
    assert enc(3 * 2.0 ** -10) == 0x02        # halfway between 2^-9 (0x01) and 2^-8 (0x02)
    assert enc(1.0625) == 0x38 and enc(1.1875) == 0x3A
    assert enc(1.0624) == 0x38 and enc(1.0626) == 0x39
    assert enc(2.0 ** -11) == 0x00 and enc(-(2.0 ** -11)) == 0x80
    # every finite code survives a round trip
    codes = np.array([c for c in range(256) if (c & 0x7F) != 0x7F], dtype=np.uint8)
    vals = np.array([oracle.e4m3_to_double(int(c)) for c in codes], dtype=np.float32)
    assert np.array_equal(oracle.e4m3_encode(vals), codes)
    # random values land on the nearest representable value (brute force)
    x = RNG.uniform(-460, 460, size=4000).astype(np.float32)
    c = oracle.e4m3_encode(x)
    table = np.array([oracle.e4m3_to_double(k) for k in range(0x7F)])
    got = np.array([oracle.e4m3_to_double(int(k)) for k in c])
    best = np.min(np.abs(np.abs(x.astype(np.float64))[:, None] - table[None, :]), axis=1)
    assert np.all(np.abs(np.abs(got) - np.minimum(np.abs(x), 448.0)) <= best + 1e-12)


def test_fp8_quantise_is_exact_on_representable_values():
    codes = np.array([c for c in range(256) if (c & 0x7F) != 0x7F], dtype=np.uint8)
    vals = np.array([oracle.e4m3_to_double(int(c)) for c in codes])
    for scale in (1.0, 0.25, 8.0):                     # powers of two: x = value * scale is exact in fp16/fp32
        x = (vals * scale).astype(np.float32)
        ok = np.abs(x) <= 65504                         # fp16 inputs
        assert np.array_equal(oracle.fp8_quantise(x[ok].astype(np.float16), scale), codes[ok])


def _typed_case(kv_dtype, lens, T, H, Hkv, D, bs, rng):
    """Contiguous per-sequence K/V values and the same data paged in a cache of
    the given element type; returns (query, caches, tables, lens, qs, Kv, Vv)."""
    q_bits = rand_fp16(sum(T), H, D, rng=rng)
    if kv_dtype == oracle.KV_BF16:
        q_bits = (q_bits.astype(np.float32).view(np.uint32) >> 16).astype(np.uint16)
        q_val = (q_bits.astype(np.uint32) << 16).view(np.float32).astype(np.float64)
    else:
        q_val = q_bits.astype(np.float64)
    Kraw, Vraw, Kv, Vv = [], [], [], []
    for L in lens:
        if kv_dtype == oracle.KV_FP8_E4M3:
            k = rng.integers(0, 256, size=(L, Hkv, D)).astype(np.uint8)
            v = rng.integers(0, 256, size=(L, Hkv, D)).astype(np.uint8)
            k[(k & 0x7F) == 0x7F] = 0x30          # no NaN codes in real data
            v[(v & 0x7F) == 0x7F] = 0x30
            # values decoded by hand from the format: sign, 4-bit exponent (bias 7), 3-bit fraction
            dec = lambda c: np.where((c >> 3) & 15, (8 + (c & 7)) * 2.0 ** (((c >> 3) & 15).astype(np.int64) - 10),
                                     (c & 7) * 2.0 ** -9) * np.where(c >> 7, -1.0, 1.0)
            Kv.append(dec(k)), Vv.append(dec(v))
        elif kv_dtype == oracle.KV_BF16:
            k = (rng.standard_normal((L, Hkv, D)).astype(np.float32).view(np.uint32) >> 16).astype(np.uint16)
            v = (rng.standard_normal((L, Hkv, D)).astype(np.float32).view(np.uint32) >> 16).astype(np.uint16)
            Kv.append((k.astype(np.uint32) << 16).view(np.float32).astype(np.float64))
            Vv.append((v.astype(np.uint32) << 16).view(np.float32).astype(np.float64))
        else:
            k, v = rand_fp16(L, Hkv, D, rng=rng), rand_fp16(L, Hkv, D, rng=rng)
            Kv.append(k.astype(np.float64)), Vv.append(v.astype(np.float64))
        Kraw.append(k), Vraw.append(v)
    # page with a fill pattern that is NaN in every format (unused slots)
    fill = {oracle.KV_F16: np.float16(np.nan), oracle.KV_BF16: np.uint16(0x7FC0), oracle.KV_FP8_E4M3: np.uint8(0x7F)}
    need = sum(-(-L // bs) for L in lens)
    nb = need + 2
    phys = rng.permutation(nb)[:need]
    kc = np.full((nb, Hkv, bs, D), fill[kv_dtype], dtype=Kraw[0].dtype)
    vc = np.full_like(kc, fill[kv_dtype])
    tab = np.full((len(lens), max(1, max(-(-L // bs) for L in lens))), -1, dtype=np.int32)
    j = 0
    for i, L in enumerate(lens):
        for lb in range(-(-L // bs)):
            tab[i, lb] = phys[j]
            t0, t1 = lb * bs, min(L, (lb + 1) * bs)
            kc[phys[j], :, : t1 - t0] = Kraw[i][t0:t1].transpose(1, 0, 2)
            vc[phys[j], :, : t1 - t0] = Vraw[i][t0:t1].transpose(1, 0, 2)
            j += 1
    qs = np.concatenate([[0], np.cumsum(T)]).astype(np.int32)
    return q_bits, q_val, kc, vc, tab, np.array(lens, dtype=np.int32), qs, Kv, Vv


@pytest.mark.parametrize("kv_dtype", [0, 1, 2])
def test_typed_attention_equals_masked_bruteforce(kv_dtype):
    H, Hkv, D, bs = 8, 2, 32, 8
    lens, T = [1, 9, 30, 17], [1, 3, 5, 0]
    rng = np.random.default_rng(77 + kv_dtype)
    q_bits, q_val, kc, vc, tab, ln, qs, Kv, Vv = _typed_case(kv_dtype, lens, T, H, Hkv, D, bs, rng)
    ks, vs = (0.02, 0.5) if kv_dtype == oracle.KV_FP8_E4M3 else (1.0, 1.0)
    scale = 0.2
    got = oracle.paged_attention_typed(q_bits, kc, vc, tab, ln, qs, Hkv, bs, scale, kv_dtype, ks, vs, threads=2)
    for i, (L, t) in enumerate(zip(lens, T)):
        for j in range(t):
            vis = L - t + j + 1
            for h in range(H):
                s = scale * (Kv[i][:vis, h // 4, :] * ks) @ q_val[qs[i] + j, h]
                p = np.exp(s - s.max())
                p /= p.sum()
                assert np.max(np.abs(got[qs[i] + j, h] - p @ (Vv[i][:vis, h // 4, :] * vs))) < 1e-12


def test_typed_attention_reduces_to_fp16_forms_and_scales():
    lens = [40, 7, 100]
    q, Ks, Vs = make_case(lens, 8, 2, 64)
    kc, vc, tab, ln = page_sequences(Ks, Vs, 16, RNG)
    a = oracle.paged_attention_typed(q, kc, vc, tab, ln, None, 2, 16, 0.125, oracle.KV_F16)
    assert np.array_equal(a, oracle.paged_decode(q, kc, vc, tab, ln, 2, 16, 0.125))
    qm = rand_fp16(6, 8, 64)
    qs = np.array([0, 2, 3, 6], dtype=np.int32)
    b = oracle.paged_attention_typed(qm, kc, vc, tab, ln, qs, 2, 16, 0.125, oracle.KV_F16)
    assert np.array_equal(b, oracle.paged_attention_causal(qm, kc, vc, tab, ln, qs, 2, 16, 0.125))
    # k_scale multiplies every score, v_scale the output (closed forms)
    c = oracle.paged_attention_typed(q, kc, vc, tab, ln, None, 2, 16, 0.125, oracle.KV_F16, 2.0, 3.0)
    d = oracle.paged_attention_typed(q, kc, vc, tab, ln, None, 2, 16, 0.25, oracle.KV_F16)
    assert np.max(np.abs(c - 3.0 * d)) < 1e-12
