"""Caches of bf16 and of fp8 E4M3 codes.

* pa_kv_write_fp8 must store, bit for bit, the oracle's codes (float32
  product with the reciprocal scale, nearest E4M3 value, ties to even,
  saturation at 448); pa_block_copy moves one-byte blocks whole.
* pa_decode_typed / pa_attention_causal_typed must give the oracle's
  attention over the decoded values (code x scale) within the path's
  tolerance.  fp8 codes are exact fp16 values, so the fp8 path keeps the
  fp16 bar (max abs 2e-3, normwise relative 1e-2).  bf16 carries 8
  significant bits: its P weights and outputs are rounded to bf16 (relative
  2^-9 each), so the absolute bar is 2^-7 of the row's largest value (at
  least 2e-3) and the normwise relative bar stays 1e-2.
"""
import numpy as np
import pytest

import oracle
import paged_kv_cache_12_gb300 as pa
from paged_kv_cache_12_gb300 import workloads
from scenario import build_allocators, step_allocation, NAN16

torch = pytest.importorskip("torch")
pytestmark = pytest.mark.gpu

if not torch.cuda.is_available():  # pragma: no cover
    pytest.skip("no CUDA device", allow_module_level=True)

KS, VS = 1.0 / 64, 1.0 / 32      # fp8 scales: N(0, 1) data spans about +-5, i.e. +-320 / +-160 in codes


def t(a):
    return torch.from_numpy(np.ascontiguousarray(a)).cuda()


def to_bf16_bits(x):
    """fp16/float values -> bf16 bit patterns (truncation of the float32; any
    fixed mapping serves as input data)."""
    return (np.asarray(x, dtype=np.float32).view(np.uint32) >> 16).astype(np.uint16)


def compare(g, o, kv):
    g = np.asarray(g, dtype=np.float64)
    assert np.isfinite(g).all(), "non-finite values in the GPU output"
    err = np.abs(g - o).reshape(-1, o.shape[-1])
    rowmax = np.abs(o).reshape(-1, o.shape[-1]).max(axis=1)
    if kv == pa.PA_KV_BF16:
        bound = np.maximum(2e-3, 2.0 ** -7 * rowmax)[:, None]
        assert (err <= bound).all(), f"max abs error {err.max():.3e} over the bf16 bound"
    else:
        assert err.max() <= 2e-3, f"max abs error {err.max():.3e}"
    rel = (err.max(axis=1) / np.maximum(rowmax, 1e-6)).max()
    assert rel <= 1e-2, f"normwise rel error {rel:.3e}"


def fp8_pool(w, pool, scale, stream):
    """Codes of a cache pool: the oracle's quantiser of the fp16 pool; for pools
    too large for it to finish quickly, seeded random finite codes instead
    (any codes serve as cache content)."""
    if pool.size <= 1 << 25:
        return oracle.fp8_quantise(pool, scale)
    rng = np.random.default_rng([w.seed, stream])
    c = rng.integers(0, 256, size=pool.shape, dtype=np.uint8)
    c[(c & 0x7F) == 0x7F] = 0x38               # no NaN codes
    return c


class TypedStep:
    """One step (history, block copies, KV writes, attention) over a cache of
    element type kv, on the GPU and in the oracle."""

    def __init__(self, w, kv):
        self.w, self.kv = w, kv
        ref, dut, used = build_allocators(w)
        self.slots, self.pairs = step_allocation(w, ref, dut)
        ids = list(range(w.num_seqs))
        self.tables, self.lens = dut.block_tables(ids, w.max_blocks_per_seq)
        unused = ~used
        if kv == pa.PA_KV_FP8_E4M3:
            k0, v0 = fp8_pool(w, w.k_pool, KS, 1), fp8_pool(w, w.v_pool, VS, 2)
            nanc = np.uint8(0x7F)
            self.q = w.query
            self.qm = w.query_multi
            self.nk, self.nv = w.new_key, w.new_value
        elif kv == pa.PA_KV_BF16:
            k0, v0 = to_bf16_bits(w.k_pool), to_bf16_bits(w.v_pool)
            nanc = np.uint16(0x7FC0)
            self.q, self.qm = to_bf16_bits(w.query), to_bf16_bits(w.query_multi)
            self.nk, self.nv = to_bf16_bits(w.new_key), to_bf16_bits(w.new_value)
        else:
            k0, v0 = w.k_pool.view(np.uint16).copy(), w.v_pool.view(np.uint16).copy()
            nanc = NAN16
            self.q, self.qm = w.query, w.query_multi
            self.nk, self.nv = w.new_key.view(np.uint16), w.new_value.view(np.uint16)   # bit patterns, as the caches
        k0.transpose(0, 2, 1, 3)[unused] = nanc
        v0.transpose(0, 2, 1, 3)[unused] = nanc
        self.k0, self.v0 = k0, v0

    def torch_dtype(self):
        return {pa.PA_KV_F16: torch.float16, pa.PA_KV_BF16: torch.bfloat16, pa.PA_KV_FP8_E4M3: torch.uint8}[self.kv]

    def run_gpu(self):
        dt = self.torch_dtype()
        qdt = torch.bfloat16 if self.kv == pa.PA_KV_BF16 else torch.float16
        v = lambda a, d: t(a).view(d)
        self.d = d = {"k": v(self.k0, dt), "v": v(self.v0, dt), "tables": t(self.tables), "lens": t(self.lens),
                      "slots": t(self.slots), "pairs": t(self.pairs)}
        pa.pa_block_copy(d["k"], d["v"], d["pairs"])
        if self.kv == pa.PA_KV_FP8_E4M3:
            pa.pa_kv_write_fp8(t(self.nk), t(self.nv), d["slots"], d["k"], d["v"], KS, VS)
        else:
            pa.pa_kv_write(v(self.nk, qdt), v(self.nv, qdt), d["slots"], d["k"], d["v"])
        d["q"], d["qm"] = v(self.q, qdt), v(self.qm, qdt)
        torch.cuda.synchronize()

    def oracle_caches(self):
        w = self.w
        kc, vc = oracle.block_copy(self.k0, self.v0, self.pairs)
        if self.kv == pa.PA_KV_FP8_E4M3:
            return oracle.kv_write_fp8(kc, vc, self.nk, self.nv, self.slots, w.block_size, KS, VS)
        return oracle.kv_write(kc, vc, self.nk, self.nv, self.slots, w.block_size)

    def scales(self):
        return (KS, VS) if self.kv == pa.PA_KV_FP8_E4M3 else (1.0, 1.0)

    def decode(self):
        w, d = self.w, self.d
        out = torch.full_like(d["q"], float("nan"))
        ws = torch.zeros(pa.pa_decode_workspace_size(w.num_seqs, w.num_heads, w.num_kv_heads, w.head_dim,
                                                     w.max_context_len), dtype=torch.uint8, device="cuda")
        pa.pa_decode_typed(out, d["q"], d["k"], d["v"], d["tables"], d["lens"], w.scale, w.max_context_len, ws,
                           *self.scales())
        torch.cuda.synchronize()
        assert pa.pa_workspace_status(ws) == pa.PA_OK
        return out

    def causal(self):
        w, d = self.w, self.d
        out = torch.full_like(d["qm"], float("nan"))
        ws = torch.zeros(pa.pa_attention_causal_workspace_size(w.num_seqs, w.num_new_tokens, w.num_heads,
                                                               w.num_kv_heads, w.head_dim, w.max_context_len),
                         dtype=torch.uint8, device="cuda")
        pa.pa_attention_causal_typed(out, d["qm"], d["k"], d["v"], d["tables"], d["lens"], t(self.w.query_start),
                                     w.scale, w.max_context_len, ws, *self.scales())
        torch.cuda.synchronize()
        assert pa.pa_workspace_status(ws) == pa.PA_OK
        return out


def as_f64(out, kv):
    if kv == pa.PA_KV_BF16:
        return out.float().cpu().numpy().astype(np.float64)
    return out.cpu().numpy().astype(np.float64)


# --------------------------------------------------------------- fp8 writes

def test_kv_write_fp8_codes_bit_exact():
    rng = np.random.default_rng(5)
    T, Hkv, D, bs, nb = 300, 4, 128, 16, 40
    x = (rng.standard_normal((2, T, Hkv, D)) * rng.choice([0.01, 1, 30, 600], size=(2, T, Hkv, 1))).astype(np.float16)
    special = np.array([0.0, -0.0, 1.0625, 1.1875, 2.0 ** -10, 3 * 2.0 ** -10, 448, 449, 464, 465, 1000, -1000,
                        np.inf, -np.inf, 2.0 ** -14, 65504], dtype=np.float16)
    x[0, 0, 0, : len(special)] = special
    x[1, 0, 0, : len(special)] = -special
    slots = rng.permutation(nb * bs)[:T].astype(np.int64)
    slots[::37] = -1                                   # padding rows are skipped
    for scale in (1.0, 1.0 / 64, 0.3):
        k0 = np.zeros((nb, Hkv, bs, D), dtype=np.uint8)
        v0 = np.full_like(k0, 0x55)
        kc, vc = t(k0), t(v0)
        pa.pa_kv_write_fp8(t(x[0]), t(x[1]), t(slots), kc, vc, scale, 2 * scale)
        rk, rv = oracle.kv_write_fp8(k0, v0, x[0], x[1], slots, bs, scale, 2 * scale)
        assert np.array_equal(kc.cpu().numpy(), rk), scale
        assert np.array_equal(vc.cpu().numpy(), rv), scale


def test_block_copy_one_byte_blocks():
    rng = np.random.default_rng(6)
    k0 = rng.integers(0, 256, size=(12, 2, 16, 128), dtype=np.uint8)
    v0 = rng.integers(0, 256, size=(12, 2, 16, 128), dtype=np.uint8)
    pairs = np.array([[0, 5], [3, 7], [3, 11]], dtype=np.int64)
    kc, vc = t(k0), t(v0)
    pa.pa_block_copy(kc, vc, t(pairs))
    rk, rv = oracle.block_copy(k0, v0, pairs)
    assert np.array_equal(kc.cpu().numpy(), rk) and np.array_equal(vc.cpu().numpy(), rv)


# -------------------------------------------------------- typed attention

CASES = [(8, 8, 128, 16), (64, 8, 128, 16), (32, 4, 128, 32), (16, 2, 128, 8), (16, 1, 128, 16)]


@pytest.mark.parametrize("kv", [pa.PA_KV_BF16, pa.PA_KV_FP8_E4M3])
@pytest.mark.parametrize("H,Hkv,D,bs", CASES + [(8, 2, 64, 16), (32, 2, 64, 32)])
def test_decode_typed_against_oracle(kv, H, Hkv, D, bs):
    if kv == pa.PA_KV_FP8_E4M3 and D != 128:
        pytest.skip("fp8 caches are built for head_dim 128")
    lens = [1, 2, 15, 16, 17, 31, 32, 33, 47, 100, 511, 512, 513, 1025, 2100, 3000]
    w = workloads.custom(seed=H + bs + D + kv, num_seqs=len(lens), num_heads=H, num_kv_heads=Hkv, head_dim=D,
                         block_size=bs, context_lens=lens)
    st = TypedStep(w, kv)
    st.run_gpu()
    kc, vc = st.oracle_caches()
    assert np.array_equal(st.d["k"].view(torch.uint8).cpu().numpy().view(kc.dtype), kc)
    assert np.array_equal(st.d["v"].view(torch.uint8).cpu().numpy().view(vc.dtype), vc)
    out = st.decode()
    ref = oracle.paged_attention_typed(st.q, kc, vc, st.tables, st.lens, None, Hkv, bs, w.scale, kv, *st.scales())
    compare(as_f64(out, kv), ref, kv)
    again = st.decode()
    assert torch.equal(out.view(torch.int16), again.view(torch.int16))


@pytest.mark.parametrize("kv", [pa.PA_KV_BF16, pa.PA_KV_FP8_E4M3])
@pytest.mark.parametrize("H,Hkv,D,bs", [(64, 8, 128, 16), (16, 1, 128, 16), (8, 2, 128, 32)])
def test_causal_typed_against_oracle(kv, H, Hkv, D, bs):
    lens = [1, 5, 40, 300, 1030, 2100, 700]
    T = [1, 5, 16, 7, 20, 150, 0]
    w = workloads.custom(seed=3 * H + bs + kv, num_seqs=len(lens), num_heads=H, num_kv_heads=Hkv, head_dim=D,
                         block_size=bs, context_lens=lens, new_tokens=T)
    st = TypedStep(w, kv)
    st.run_gpu()
    kc, vc = st.oracle_caches()
    out = st.causal()
    ref = oracle.paged_attention_typed(st.qm, kc, vc, st.tables, st.lens, w.query_start, Hkv, bs, w.scale, kv,
                                       *st.scales())
    compare(as_f64(out, kv), ref, kv)


def test_fp16_through_the_typed_entry_is_the_plain_decode():
    lens = [3, 700, 1500, 64]
    w = workloads.custom(seed=8, num_seqs=len(lens), num_heads=32, num_kv_heads=8, head_dim=128, block_size=16,
                         context_lens=lens)
    st = TypedStep(w, pa.PA_KV_F16)
    st.run_gpu()
    d = st.d
    typed = st.decode()
    out = torch.empty_like(typed)
    ws = torch.zeros(pa.pa_decode_workspace_size(w.num_seqs, 32, 8, 128, w.max_context_len), dtype=torch.uint8,
                     device="cuda")
    pa.pa_decode(out, d["q"], d["k"], d["v"], d["tables"], d["lens"], w.scale, w.max_context_len, ws)
    torch.cuda.synchronize()
    assert torch.equal(out.view(torch.int16), typed.view(torch.int16))


def test_fp8_scales_act_as_stated():
    # doubling k_scale is doubling the softmax scale; doubling v_scale doubles the output
    lens = [50, 900]
    w = workloads.custom(seed=12, num_seqs=2, num_heads=16, num_kv_heads=2, head_dim=128, block_size=16,
                         context_lens=lens)
    st = TypedStep(w, pa.PA_KV_FP8_E4M3)
    st.run_gpu()
    d = st.d
    ws = torch.zeros(pa.pa_decode_workspace_size(2, 16, 2, 128, w.max_context_len), dtype=torch.uint8, device="cuda")

    def run(scale, ks, vs):
        o = torch.empty_like(d["q"])
        pa.pa_decode_typed(o, d["q"], d["k"], d["v"], d["tables"], d["lens"], scale, w.max_context_len, ws, ks, vs)
        torch.cuda.synchronize()
        return o.double().cpu().numpy()

    a = run(w.scale, 2 * KS, VS)
    b = run(2 * w.scale, KS, VS)
    assert np.max(np.abs(a - b)) <= 2e-3
    c = run(w.scale, KS, 2 * VS)
    e = run(w.scale, KS, VS)
    assert np.max(np.abs(c - 2 * e)) <= 4e-3


@pytest.mark.slow
def test_fp8_full_size_sampled():
    w = workloads.make("gqa72b")
    st = TypedStep(w, pa.PA_KV_FP8_E4M3)
    st.run_gpu()
    out = st.decode().cpu().numpy()
    assert np.isfinite(out).all()
    kc, vc = st.oracle_caches()
    idx = np.array([0, 41, 99])
    ref = oracle.paged_attention_typed(st.q[idx], kc, vc, st.tables[idx], st.lens[idx], None, w.num_kv_heads,
                                       w.block_size, w.scale, pa.PA_KV_FP8_E4M3, KS, VS)
    compare(out[idx].astype(np.float64), ref, pa.PA_KV_FP8_E4M3)
