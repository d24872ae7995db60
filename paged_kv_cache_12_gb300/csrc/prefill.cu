// Paged causal attention for long runs of new tokens (a prompt chunk) on the
// 5th-generation tensor cores.
//
// What is computed is the multi-token form of decode.cu (deepsonar page,
// section 2.5: a request may compute a chunk of its prompt in one step): new
// token j of sequence i (query row query_start[i] + j) attends to positions
// t <= L_i - T_i + j through the block table.  When a sequence brings many new
// tokens the work is a dense contraction -- 128 query rows against every KV
// tile -- so it runs here on tcgen05 rather than on the decode pipeline.
//
// A work tile is (sequence, kv head, 128 query rows): 128 / G consecutive new
// tokens times the G query heads of the kv head (rows token-major), so a K/V
// tile read from HBM serves all of them.  One CTA per SM, persistent over a
// static list of tiles ordered longest first; six warps:
//   warps 0-1  producers of K and of V: per 128-token KV tile, TMA copies of
//              the block rows (gathered through the block table, one lane per
//              block) into 3-stage rings;
//   warp 2     MMA issuer (one thread): S = Q K^T into one of two tensor
//              memory buffers (M 128, N 128, K 128), then O += P V (M 128,
//              N 128, K 128) into a tensor-memory accumulator, both with the
//              A operand (Q, P) in tensor memory and B (K, V) in shared
//              memory; completions are committed to mbarriers;
//   warps 3-6  softmax (one query row per thread, the row's tensor-memory
//              lane): store the Q row into tensor memory, read the row of S,
//              mask past the row's position, online softmax in fp32 with the
//              running maximum rescaled only when it grows by more than 2^8
//              (then O is rescaled in tensor memory), store P (fp16/bf16) into
//              tensor memory for the PV product, and at the end divide O by
//              the row sum and store the output row.
// Q and P live in tensor memory so that shared memory holds only K/V rings,
// three stages deep: a 32 KB K or V tile takes about 2 us to arrive from L2,
// and with two stages that latency, not the tensor or exponential work, set
// the time per KV tile.
// S for the next KV tile is computed while the softmax works on this one.
// FP8 E4M3 caches: the producer warps stage the one-byte codes by TMA and turn
// them into exact fp16 tiles of the same layout (two stages), the K scale
// folded into the softmax scale and the V scale into the output.
// Every wait is bounded and every warp-collective instruction (tensor-memory
// loads and stores, votes) runs in warp-uniform control flow; tensor memory
// is released on every path.

#include <cmath>
#include <mutex>

#include "prefill_common.cuh"

namespace pa {
namespace {

// Shared memory per cache type: the K and V rings the MMAs read (16-bit
// tiles; R stages each) and, for an FP8 cache, the rings its codes are staged
// in by TMA (S8 stages each) before the producer warps turn them into fp16
// tiles of the same layout.
template <int KV>
struct PfL {
    static constexpr bool F8 = KV == PA_KV_FP8_E4M3;
    static constexpr int R = F8 ? 2 : PST;
    static constexpr int S8 = F8 ? 3 : 0;
    static constexpr int OFF_K = 0;
    static constexpr int OFF_V = R * KV_BYTES;
    static constexpr int OFF_K8 = 2 * R * KV_BYTES;
    static constexpr int OFF_V8 = OFF_K8 + S8 * F8_BYTES;
    static constexpr int OFF_CTRL = OFF_V8 + S8 * F8_BYTES;
    static constexpr int SMEM = OFF_CTRL + CTRL_BYTES + 1024;   // + alignment slack
    // 16-bit caches: warps 0 / 1 produce K / V, 2 issues the MMAs, 3-6 run
    // the softmax.  FP8 caches: warp 0 issues the copies of the codes, 2 the
    // MMAs, 4-7 run the softmax and 8-11 convert (two per cache, one on each
    // SM sub-partition), with a register split (CONV_REGS / SOFT_REGS).
    static constexpr int THREADS = (F8 ? 12 : 7) * 32;
    static constexpr int SOFT_WARP0 = F8 ? 4 : 3;
    static constexpr int SOFT_REGS = 232, CONV_REGS = 136, LAUNCH_REGS = 168;   // FP8: 65536 / 384 at launch
    static_assert(!F8 || 128 * SOFT_REGS + 256 * CONV_REGS <= THREADS * LAUNCH_REGS, "register split");
    static_assert(R <= MAXST && S8 <= MAXST, "ring stages");
    static_assert(SMEM <= 227 * 1024, "shared memory of one CTA");
};
// tensor memory: S0 [0, PN), S1 [PN, 2 PN), O (128 fp32 columns), Q (128 dims,
// two fp16/bf16 per column), P (PN tokens, two per column)
constexpr int TMEM_COLS = 512;
constexpr int TM_O = 2 * PN;
constexpr int TM_Q = TM_O + PD;
constexpr int TM_P = TM_Q + PD / 2;
static_assert(TM_P + PN / 2 <= TMEM_COLS, "tensor-memory columns");
static_assert(PN == 64 || PN == 128, "KV tile of 64 or 128 tokens");
static_assert(8 * (8 * MAXST + 11) + 8 <= CTRL_BAD && CTRL_ABORT + 4 <= CTRL_BYTES, "control block layout");

struct PfBars {
    // pfull / pvdone: one per PV-number parity, so that a softmax warp a step
    // ahead of another never adds its arrival to the other step's phase
    // k8full / v8full: FP8 codes staged (TMA bytes landed); k8empty / v8empty:
    // the staged codes converted (the staging slot may be refilled)
    BarRing kfull, kempty, vfull, vempty, k8full, v8full, k8empty, v8empty;   // MAXST each
    BarRing sfull, sfree, pfull, pvdone;                                      // 2 each
    uint32_t qfull, tmem_slot, flags;   // shared addresses
};

__device__ __forceinline__ PfBars pf_bars(uint8_t *smem, int off_ctrl) {
    uint32_t a = smem_u32(smem + off_ctrl);
    PfBars b;
    BarRing *rings[8] = {&b.kfull, &b.kempty, &b.vfull, &b.vempty, &b.k8full, &b.v8full, &b.k8empty, &b.v8empty};
    for (int r = 0; r < 8; ++r) rings[r]->base = a, a += 8 * MAXST;
    b.sfull.base = a, a += 16;
    b.sfree.base = a, a += 16;
    b.pfull.base = a, a += 16;
    b.pvdone.base = a, a += 16;
    b.qfull = a, a += 8;
    b.tmem_slot = a, a += 8;
    b.flags = a;   // barriers and slots end at byte 8 (8 MAXST + 11) + 8 = 288 <= CTRL_BAD
    return b;
}


template <int KV, int MODE>
__device__ void pf_producer(uint8_t *smem, const CUtensorMap *map, const PrefillArgs &a, const PfBars &bb,
                            volatile int *abort_flag, int total, int kv) {
    using L = PfL<KV>;
    const int off[1] = {kv ? L::OFF_V : L::OFF_K};
    const BarRing full[1] = {kv ? bb.vfull : bb.kfull};
    const BarRing empty[1] = {kv ? bb.vempty : bb.kempty};
    const CUtensorMap *maps[1] = {map};
    pf_stream<L::R, false, 1>(smem, off, L::OFF_CTRL, full, empty, maps, a, abort_flag, total, [&](int item) {
                        const PfTile t = pf_item<MODE>(a, item);
                        return PfRange{t.seq, t.kvh, t.nkv, t.L, t.kv0};
                    });
}

// FP8 cache of the one-tile kernel: the converting warps of one cache.
__device__ void pf_convert_fp8(uint8_t *smem, const PrefillArgs &a, const PfBars &bb, volatile int *abort_flag,
                               int total, int kv, int half) {
    using L = PfL<PA_KV_FP8_E4M3>;
    pf_convert_ring<L::R, L::S8, 2>(smem + (kv ? L::OFF_V8 : L::OFF_K8), smem + (kv ? L::OFF_V : L::OFF_K),
                                 kv ? bb.v8full : bb.k8full, kv ? bb.v8empty : bb.k8empty, kv ? bb.vfull : bb.kfull,
                                 kv ? bb.vempty : bb.kempty, a, abort_flag, total, half,
                                 [&](int item) { return pf_tile(a, item).nkv; });
}

// ----------------------------------------------------------- MMA issuer

template <int KV, int MODE>
__device__ void pf_mma(uint8_t *smem, const PrefillArgs &a, const PfBars &bb, uint32_t tmem, bool bf16,
                       volatile int *abort_flag, int total) {
    using L = PfL<KV>;
    constexpr int PST = L::R;
    constexpr int OFF_K = L::OFF_K, OFF_V = L::OFF_V;
    const uint32_t base = smem_u32(smem);
    const uint32_t id_s = idesc_f16(PM, PN, bf16, false);
    const uint32_t id_o = idesc_f16(PM, PD, bf16, true);
    // descriptors of the shared-memory B tiles; a byte offset o inside shared
    // memory is o / 16 added to the descriptor (its low field is the address / 16)
    const uint64_t dk0 = sw128_desc(base + OFF_K, 16, 1024);
    // V: B operand with N (dims) contiguous: 128-byte rows of 64 dims, one row
    // per token (K); the next 64 dims are the next block of PN rows
    const uint64_t dv0 = sw128_desc(base + OFF_V, PN * 128, 1024);
    int kc = 0, vc = 0, sc = 0, pc = 0, qc = 0;
    bool ok = true;
    auto wait = [&](uint32_t bar, uint32_t parity) {
        if (!ok) return false;
        if (*abort_flag || !mbar_wait_bounded(bar, parity, a.wait_limit)) {
            pf_error(a);
            *abort_flag = 1;
            ok = false;
        }
        return ok;
    };
    // S(next) = Q K^T into tensor-memory buffer sc & 1
    auto issue_s = [&]() {
        const int ks = kc % PST;
        const int b = sc & 1;
        if (!wait(bb.kfull[ks], (kc / PST) & 1)) return;
        if (sc >= 2 && !wait(bb.sfree[b], ((sc >> 1) - 1) & 1)) return;
        tc_fence_after_sync();
        const uint64_t dk = dk0 + (uint64_t)(ks * (KV_BYTES >> 4));
        const uint32_t dst = tmem + b * PN;
#pragma unroll
        for (int k = 0; k < PD / 16; ++k) {
            // K-step k: 16 dims = Q columns 8k .. 8k + 7; K at byte 32 (k % 4) of the 64-dim block k / 4
            umma_f16_ts(dst, tmem + TM_Q + 8 * k, dk + (uint64_t)(((k >> 2) * (PN * 128) + (k & 3) * 32) >> 4), id_s,
                        k > 0 ? 1u : 0u);
        }
        umma_commit(bb.sfull[b]);
        umma_commit(bb.kempty[ks]);
        ++kc;
        ++sc;
    };
    for (int item = blockIdx.x; item < total && ok; item += gridDim.x) {
        const PfTile t = pf_item<MODE>(a, item);
        if (!wait(bb.qfull, qc & 1)) break;
        ++qc;
        issue_s();
        for (int n = 0; n < t.nkv && ok; ++n) {
            if (n + 1 < t.nkv) issue_s();
            const int pb = pc & 1;   // barrier parity of PV number pc
            if (!wait(bb.pfull[pb], (pc >> 1) & 1)) break;
            ++pc;
            const int vs = vc % PST;
            if (!wait(bb.vfull[vs], (vc / PST) & 1)) break;
            tc_fence_after_sync();
            const uint64_t dv = dv0 + (uint64_t)(vs * (KV_BYTES >> 4));
#pragma unroll
            for (int k = 0; k < PN / 16; ++k)   // K-step k: 16 tokens = P columns 8k .. 8k + 7, V row 16 k
                umma_f16_ts(tmem + TM_O, tmem + TM_P + 8 * k, dv + (uint64_t)((k * 16 * 128) >> 4), id_o,
                            (n > 0 || k > 0) ? 1u : 0u);
            umma_commit(bb.pvdone[pb]);
            umma_commit(bb.vempty[vs]);
            ++vc;
        }
    }
}

// ------------------------------------------------------------- softmax

template <int KV, int MODE>
__device__ void pf_softmax(uint8_t *smem, const PrefillArgs &a, const PfBars &bb, uint32_t tmem,
                           volatile int *abort_flag, int total) {
    using L = PfL<KV>;
    constexpr int PST = L::R;
    constexpr int OFF_V = L::OFF_V, OFF_CTRL = L::OFF_CTRL;
    const int tid = threadIdx.x - 32 * L::SOFT_WARP0;   // 0 .. 127
    const int lane = threadIdx.x & 31;
    const int quarter = (threadIdx.x >> 5) & 3;    // tensor-memory lanes 32 quarter .. + 31
    const int m = quarter * 32 + lane;             // this thread's query row in the tile
    const uint32_t trow = tmem + ((uint32_t)(quarter * 32) << 16);
    const float sl2 = a.scale_log2;
    // g: P tiles written so far (P tile g feeds PV number g; one P buffer, so
    // P tile g is stored once PV number g - 1 is done); pvdone[b] completes
    // for PV numbers b, b + 2, ... in order
    int sc = 0, g = 0, vcount = 0;
    bool ok = true;
    // every thread of the warp takes the same decision, so warp-collective
    // tensor-memory loads and stores are never reached by part of a warp
    auto wait = [&](uint32_t bar, uint32_t parity) {
        if (!ok) return false;
        const bool got = !*abort_flag && mbar_wait_bounded(bar, parity, a.wait_limit);
        if (!__all_sync(0xffffffffu, got)) {
            if (lane == 0) pf_error(a);
            *abort_flag = 1;
            ok = false;
        }
        return ok;
    };
    const int tok = m / a.G, hh = m - tok * a.G;   // new token (or member) and head of this row
    // ---- an item's Q rows into this thread's lane of the tensor-memory A
    // tile, two dims per column (zeros past the item's rows).  The next item's
    // rows are stored as soon as this item's last PV is done (every product
    // that read Q is then done too), before this item's epilogue, so that the
    // next item's first S product overlaps the epilogue.
    auto store_q = [&](const PfTile &tq) {
        const bool v = tok < tq.ntok;
        const uint4 *src = reinterpret_cast<const uint4 *>(
            a.query + ((long long)(tq.q0 + tq.row0 + tok) * a.Hq + tq.kvh * a.G + hh) * PD);
#pragma unroll
        for (int h = 0; h < 2; ++h) {
            uint32_t r[32];
#pragma unroll
            for (int c = 0; c < 8; ++c) {
                const uint4 x = v ? __ldg(src + 8 * h + c) : make_uint4(0, 0, 0, 0);
                r[4 * c] = x.x;
                r[4 * c + 1] = x.y;
                r[4 * c + 2] = x.z;
                r[4 * c + 3] = x.w;
            }
            tmem_st32(trow + TM_Q + 32 * h, r);
        }
        tmem_wait_st();
        tc_fence_before_sync();
        mbar_arrive(bb.qfull);
    };
    if ((int)blockIdx.x < total) store_q(pf_item<MODE>(a, blockIdx.x));
    for (int item = blockIdx.x; item < total && ok; item += gridDim.x) {
        const PfTile t = pf_item<MODE>(a, item);
        const bool valid = tok < t.ntok;
        const long long qrow = ((long long)(t.q0 + t.row0 + tok) * a.Hq + t.kvh * a.G + hh) * PD;
        // positions of the range this row sees: causally up to its own new
        // token, or (a shared range) all of them
        const int vis = !valid ? 1 : MODE == PF_SHARED ? t.L : t.C + t.row0 + tok;
        float mrun = -INFINITY, l = 0.f;
        for (int n = 0; n < t.nkv && ok; ++n) {
            // ---- S row of this KV tile
            const int b = sc & 1;
            if (!wait(bb.sfull[b], (sc >> 1) & 1)) break;
            ++sc;
            tc_fence_after_sync();
            float s[PN];
#pragma unroll
            for (int q = 0; q < PN / 32; ++q) {
                uint32_t r[32];
                tmem_ld32(trow + b * PN + 32 * q, r);
#pragma unroll
                for (int c = 0; c < 32; ++c) s[32 * q + c] = __uint_as_float(r[c]);
            }
            tmem_wait_ld();
            tc_fence_before_sync();
            mbar_arrive(bb.sfree[b]);
            const int t0 = n * PN;
            if (t0 + PN > vis) {   // the tile reaches past this row's position
#pragma unroll
                for (int c = 0; c < PN; ++c) s[c] = t0 + c < vis ? s[c] : -INFINITY;
            }
            // row maximum of the raw scores (scale > 0), eight partial maxima
            float mp[8];
#pragma unroll
            for (int j = 0; j < 8; ++j) mp[j] = s[j];
#pragma unroll
            for (int c = 8; c < PN; ++c) mp[c & 7] = fmaxf(mp[c & 7], s[c]);
            const float mx = fmaxf(fmaxf(fmaxf(mp[0], mp[1]), fmaxf(mp[2], mp[3])),
                                   fmaxf(fmaxf(mp[4], mp[5]), fmaxf(mp[6], mp[7]))) * sl2;
            // Whether to rescale is decided per row, but the tensor-memory round
            // trip of O and the wait before it are warp-collective: when any
            // row of the warp grows, every lane takes the branch, and a lane
            // whose own row does not grow scales by exactly 1 (its bits stay).
            // A branch taken by part of a warp would run tcgen05.ld/st and the
            // vote of the bounded wait in divergent code, which can hang the
            // warp outside any bounded wait.
            const bool grow = mx > mrun + RESCALE_THRESHOLD;
            if (__any_sync(0xffffffffu, grow)) {
                const float nm = grow ? fmaxf(mrun, mx) : mrun;
                const float alpha = grow ? fast_exp2(mrun - nm) : 1.f;
                if (n > 0) {   // O holds PV up to number g - 1: rescale it in tensor memory
                    if (!wait(bb.pvdone[(g - 1) & 1], ((g - 1) >> 1) & 1)) break;
                    tc_fence_after_sync();
#pragma unroll 1
                    for (int c4 = 0; c4 < PD / 32; ++c4) {
                        uint32_t o[32];
                        tmem_ld32(trow + TM_O + c4 * 32, o);
                        tmem_wait_ld();
#pragma unroll
                        for (int c = 0; c < 32; ++c) o[c] = __float_as_uint(__uint_as_float(o[c]) * alpha);
                        tmem_st32(trow + TM_O + c4 * 32, o);
                    }
                    tmem_wait_st();
                }
                l *= alpha;
                mrun = nm;
            }
            // ---- the last KV tile: V rows past the context are zeroed (P is 0 there)
            const int vs = vcount % PST;
            const int vphase = (vcount / PST) & 1;
            ++vcount;
            const bool zero_v = t0 + PN > t.L;
            if (zero_v) {
                if (!wait(bb.vfull[vs], vphase)) break;
                const int first = t.L - t0;    // rows first .. PN-1 of both 64-dim blocks
                uint8_t *vt = smem + OFF_V + vs * KV_BYTES;
                for (int k = tid; k < 2 * PN * 8; k += 128) {
                    const int h = k / (PN * 8), rr = (k / 8) % PN, cc = k % 8;
                    if (rr >= first)
                        *reinterpret_cast<uint4 *>(vt + h * (PN * 128) + rr * 128 + cc * 16) = make_uint4(0, 0, 0, 0);
                }
            }
            // ---- p = 2^(s scale log2(e) - m), packed two per column into this
            // thread's lane of the tensor-memory P tile (64 tokens per store),
            // and the row sum in eight partial sums
            float lp[8];
#pragma unroll
            for (int j = 0; j < 8; ++j) lp[j] = 0.f;
            auto pack64 = [&](int h, uint32_t (&r)[32]) {
#pragma unroll
                for (int c = 0; c < 8; ++c) {   // tokens 64 h + 8 c .. + 7
                    float p[8];
#pragma unroll
                    for (int j = 0; j < 8; ++j) {
                        p[j] = fast_exp2(fmaf(s[64 * h + 8 * c + j], sl2, -mrun));
                        lp[j] += p[j];
                    }
                    r[4 * c] = pack_p<KV>(p[0], p[1]);
                    r[4 * c + 1] = pack_p<KV>(p[2], p[3]);
                    r[4 * c + 2] = pack_p<KV>(p[4], p[5]);
                    r[4 * c + 3] = pack_p<KV>(p[6], p[7]);
                }
            };
            {
                uint32_t r[32];
                pack64(0, r);
                // one P buffer: PV g - 1 (which reads P tile g - 1) is done first
                if (g >= 1 && !wait(bb.pvdone[(g - 1) & 1], ((g - 1) >> 1) & 1)) break;
                tmem_st32(trow + TM_P, r);
            }
            if constexpr (PN == 128) {
                uint32_t r[32];
                pack64(1, r);
                tmem_st32(trow + TM_P + 32, r);
            }
            l += ((lp[0] + lp[1]) + (lp[2] + lp[3])) + ((lp[4] + lp[5]) + (lp[6] + lp[7]));
            tmem_wait_st();
            if (zero_v) fence_proxy_async_smem();   // the zeroed V rows, for the tensor cores
            tc_fence_before_sync();
            mbar_arrive(bb.pfull[g & 1]);
            ++g;
        }
        if (!ok) break;
        // ---- epilogue: O / l once the tile's last PV (number g - 1) is done;
        // the next item's Q first
        if (!wait(bb.pvdone[(g - 1) & 1], ((g - 1) >> 1) & 1)) break;
        tc_fence_after_sync();
        if (item + (int)gridDim.x < total) store_q(pf_item<MODE>(a, item + gridDim.x));
        const bool bad = *pf_bad_slot(smem, OFF_CTRL, pf_local(item)) == pf_local(item) + 1;
        if constexpr (MODE == PF_SHARED) {
            // the member's partial row of this shared range: unnormalised O,
            // and (m, l) -- the decode kernel's partial format -- at the
            // canonical row part_off[member] + the range's partition index
            const float qnan = __int_as_float(0x7fc00000);
            const long long wrow = valid ? ((long long)a.part_off[t.q0 + tok] + t.kv0 / a.pt) * a.Hq +
                                               t.kvh * a.G + hh
                                         : 0;
            float *prow = a.ws_o + wrow * PD;
#pragma unroll 1
            for (int c4 = 0; c4 < PD / 32; ++c4) {
                uint32_t o[32];
                tmem_ld32(trow + TM_O + c4 * 32, o);
                tmem_wait_ld();
                if (valid) {
#pragma unroll
                    for (int c = 0; c < 32; c += 4)
                        *reinterpret_cast<float4 *>(prow + c4 * 32 + c) =
                            bad ? make_float4(qnan, qnan, qnan, qnan)
                                : make_float4(__uint_as_float(o[c]) * a.v_scale, __uint_as_float(o[c + 1]) * a.v_scale,
                                              __uint_as_float(o[c + 2]) * a.v_scale,
                                              __uint_as_float(o[c + 3]) * a.v_scale);
                }
            }
            if (valid) a.ws_ml[wrow] = bad ? make_float2(qnan, qnan) : make_float2(mrun, l);
            tc_fence_before_sync();
            continue;
        }
        const float inv = bad ? __int_as_float(0x7fc00000) : a.v_scale / l;
        uint16_t *orow = a.out + qrow;
#pragma unroll 1
        for (int c4 = 0; c4 < PD / 32; ++c4) {
            uint32_t o[32];
            tmem_ld32(trow + TM_O + c4 * 32, o);
            tmem_wait_ld();
            if (valid) {
#pragma unroll
                for (int c = 0; c < 32; c += 8) {
                    uint4 v;
                    v.x = (uint32_t)out_bits<KV>(__uint_as_float(o[c]) * inv) |
                          ((uint32_t)out_bits<KV>(__uint_as_float(o[c + 1]) * inv) << 16);
                    v.y = (uint32_t)out_bits<KV>(__uint_as_float(o[c + 2]) * inv) |
                          ((uint32_t)out_bits<KV>(__uint_as_float(o[c + 3]) * inv) << 16);
                    v.z = (uint32_t)out_bits<KV>(__uint_as_float(o[c + 4]) * inv) |
                          ((uint32_t)out_bits<KV>(__uint_as_float(o[c + 5]) * inv) << 16);
                    v.w = (uint32_t)out_bits<KV>(__uint_as_float(o[c + 6]) * inv) |
                          ((uint32_t)out_bits<KV>(__uint_as_float(o[c + 7]) * inv) << 16);
                    *reinterpret_cast<uint4 *>(orow + c4 * 32 + c) = v;
                }
            }
        }
        tc_fence_before_sync();
    }
}

template <int KV, int MODE>
__global__ void __launch_bounds__(PfL<KV>::THREADS, 1) prefill_kernel(const __grid_constant__ CUtensorMap tmk,
                                                                 const __grid_constant__ CUtensorMap tmv,
                                                                 const PrefillArgs a) {
    extern __shared__ uint8_t smem_raw[];
    uint8_t *smem = reinterpret_cast<uint8_t *>((reinterpret_cast<uintptr_t>(smem_raw) + 1023) & ~uintptr_t(1023));
    using L = PfL<KV>;
    const PfBars bb = pf_bars(smem, L::OFF_CTRL);
    volatile int *abort_flag = reinterpret_cast<volatile int *>(smem + L::OFF_CTRL + CTRL_ABORT);
    const int warp = threadIdx.x >> 5;
    const int total = *reinterpret_cast<volatile int *>(&a.hdr->pf_items);   // written by the prep kernel
    if ((int)blockIdx.x >= total) return;   // no work item for this CTA (the whole CTA leaves)
    if (threadIdx.x == 0) {
        constexpr uint32_t fill = L::F8 ? 2 : 1;   // FP8: two converting warps per ring
        for (int s = 0; s < L::R; ++s) {
            mbar_init(bb.kfull[s], fill);
            mbar_init(bb.kempty[s], 1);
            mbar_init(bb.vfull[s], fill);
            mbar_init(bb.vempty[s], 1);
        }
        for (int s = 0; s < L::S8; ++s) {
            mbar_init(bb.k8full[s], 1);
            mbar_init(bb.v8full[s], 1);
            mbar_init(bb.k8empty[s], 2);
            mbar_init(bb.v8empty[s], 2);
        }
        mbar_init(bb.sfull[0], 1);
        mbar_init(bb.sfull[1], 1);
        mbar_init(bb.sfree[0], 128);
        mbar_init(bb.sfree[1], 128);
        mbar_init(bb.pfull[0], 128);
        mbar_init(bb.pfull[1], 128);
        mbar_init(bb.pvdone[0], 1);
        mbar_init(bb.pvdone[1], 1);
        mbar_init(bb.qfull, 128);
        mbar_init(bb.flags, 1);            // all MMAs completed (before tensor memory is freed)
        for (int k = 0; k < BAD_SLOTS; ++k) *pf_bad_slot(smem, L::OFF_CTRL, k) = 0;
        *abort_flag = 0;
        fence_mbar_init();
    }
    if (warp == 2) {   // this warp owns the tensor memory
        tmem_alloc(bb.tmem_slot, TMEM_COLS);
        tmem_relinquish();
    }
    tc_fence_before_sync();
    __syncthreads();
    tc_fence_after_sync();
    const uint32_t tmem = *reinterpret_cast<volatile uint32_t *>(smem + (bb.tmem_slot - smem_u32(smem)));
    auto mma = [&]() {
        if ((threadIdx.x & 31) == 0) {
            pf_mma<KV, MODE>(smem, a, bb, tmem, KV == PA_KV_BF16, abort_flag, total);
            // every MMA issued has completed before tensor memory is released
            umma_commit(bb.flags);
            mbar_wait_bounded(bb.flags, 0, WAIT_LIMIT);
        }
        __syncwarp();
    };
    if constexpr (L::F8) {
        // register split: the softmax warpgroup (warps 4-7) gets SOFT_REGS
        // registers, the others CONV_REGS (the host checks the launch count)
        if (warp >= 4 && warp < 8) {
            regs_increase<L::SOFT_REGS>();
            pf_softmax<KV, MODE>(smem, a, bb, tmem, abort_flag, total);
        } else {
            regs_decrease<L::CONV_REGS>();
            if (warp == 0) {   // the codes of K and V into the staging rings
                const int off[2] = {L::OFF_K8, L::OFF_V8};
                const BarRing full[2] = {bb.k8full, bb.v8full};
                const BarRing empty[2] = {bb.k8empty, bb.v8empty};
                const CUtensorMap *maps[2] = {&tmk, &tmv};
                pf_stream<L::S8, true, 2>(smem, off, L::OFF_CTRL, full, empty, maps, a, abort_flag, total,
                                          [&](int item) {
                                              const PfTile t = pf_tile(a, item);
                                              return PfRange{t.seq, t.kvh, t.nkv, t.L, t.kv0};
                                          });
            } else if (warp == 2) {
                mma();
            } else if (warp >= 8) {   // 8, 9: K; 10, 11: V; each half of the rows
                pf_convert_fp8(smem, a, bb, abort_flag, total, (warp - 8) >> 1, warp & 1);
            }
        }
    } else {
        if (warp < 2)
            pf_producer<KV, MODE>(smem, warp ? &tmv : &tmk, a, bb, abort_flag, total, warp);
        else if (warp == 2)
            mma();
        else
            pf_softmax<KV, MODE>(smem, a, bb, tmem, abort_flag, total);
    }
    tc_fence_before_sync();
    __syncthreads();
    if (warp == 2) {
        tc_fence_after_sync();
        tmem_dealloc(tmem, TMEM_COLS);
    }
}

// ===================================================== two row tiles per CTA
//
// A sequence with a long run of new tokens has many row tiles over nearly the
// same KV range.  Here one CTA takes two neighbouring row tiles of it (tile 0
// the later rows, which see the longer range) and every K/V tile it loads
// feeds both, so L2 delivers half the bytes per FLOP of the one-tile kernel.
// Tensor memory holds S0, S1 (one 128-column buffer per tile), O0 and O1 (all
// 512 columns); each tile's P (fp16/bf16, two per column) is written over the
// first 64 columns of its own S once the softmax has read them, and Q lives
// in shared memory.  So S_x(n + 1) may only be issued after PV_x(n) -- which
// reads P_x(n) from those columns -- and the MMA thread alternates the tiles:
//   PV0(n), S0(n + 1), PV1(n), S1(n + 1), ...
// while tile 1's softmax works on S1(n), tile 0's MMAs run, and the other way
// round.  MMAs issued by one thread complete in issue order, and a commit
// tracks every MMA issued before it: when S_x(n) is complete so is PV_x(n - 1),
// so the softmax may rescale O_x then without waiting for anything else.
// Warps: 0 and 1 produce K and V (3- and 2-stage rings), 2 issues the MMAs,
// 3 idles, 4-7 run tile 0's softmax and 8-11 tile 1's, one row per thread.

constexpr int P2_THREADS = 12 * 32;
constexpr int Q_BYTES = PM * PD * 2;       // one 128-row Q tile, fp16/bf16, 128-byte swizzled K-major
constexpr int P2_RK = 3, P2_RV = 2;        // K and V ring stages
constexpr int P2_OFF_K = 0;
constexpr int P2_OFF_V = P2_RK * KV_BYTES;
constexpr int P2_OFF_Q = P2_OFF_V + P2_RV * KV_BYTES;
constexpr int P2_OFF_CTRL = P2_OFF_Q + 2 * Q_BYTES;
constexpr int P2_SMEM = P2_OFF_CTRL + CTRL_BYTES + 1024;   // + alignment slack
constexpr int TM2_O = 2 * PN;              // O0 at columns 256 .., O1 at 384 ..
constexpr int P2_REGS_LAUNCH = 168;        // per thread at launch: 65536 / 384, rounded down to 8
constexpr int P2_REGS_LOW = 104;           // producers, MMA issuer (warpgroup 0)
constexpr int P2_REGS_HIGH = 200;          // the two softmax warpgroups
static_assert(128 * P2_REGS_LOW + 256 * P2_REGS_HIGH <= P2_THREADS * P2_REGS_LAUNCH,
              "register split within the launch's pool");
static_assert(P2_SMEM <= 227 * 1024, "shared memory of one CTA");
static_assert(TM2_O + 2 * PD <= TMEM_COLS && PN == 128, "tensor-memory columns of the two-tile kernel");

struct P2Bars {
    BarRing kfull, kempty, vfull, vempty;   // P2_RK / P2_RV stages
    BarRing sfull, pfull, pvdone, qfull;    // per tile
    uint32_t tmem_slot, flags;
};
static_assert(8 * (2 * P2_RK + 2 * P2_RV + 8 + 2) <= CTRL_BAD, "control block layout of the two-tile kernel");

__device__ __forceinline__ P2Bars p2_bars(uint8_t *smem) {
    uint32_t a = smem_u32(smem + P2_OFF_CTRL);
    P2Bars b;
    b.kfull.base = a, a += 8 * P2_RK;
    b.kempty.base = a, a += 8 * P2_RK;
    b.vfull.base = a, a += 8 * P2_RV;
    b.vempty.base = a, a += 8 * P2_RV;
    b.sfull.base = a, a += 16;
    b.pfull.base = a, a += 16;
    b.pvdone.base = a, a += 16;
    b.qfull.base = a, a += 16;
    b.tmem_slot = a, a += 8;
    b.flags = a;
    return b;
}

// Work item of the two-tile kernel: tile 0 and, if the pair has one, tile 1
// (nkv of an absent tile 1 is 0).
struct P2Item {
    PfTile t[2];
};

__device__ __forceinline__ P2Item p2_item(const PrefillArgs &a, int item) {
    const int4 rec = a.pairs[item / a.Hkv];
    P2Item p;
    p.t[0] = pf_row_tile(a, rec.x, item % a.Hkv, rec.y);
    if (rec.z >= 0) {
        p.t[1] = pf_row_tile(a, rec.x, item % a.Hkv, rec.z);
    } else {
        p.t[1] = p.t[0];
        p.t[1].nkv = 0;
    }
    return p;
}

template <int KV>
__device__ void p2_mma(uint8_t *smem, const PrefillArgs &a, const P2Bars &bb, uint32_t tmem, volatile int *abort_flag,
                       int total) {
    const bool bf16 = KV == PA_KV_BF16;
    const uint32_t base = smem_u32(smem);
    const uint32_t id_s = idesc_f16(PM, PN, bf16, false);
    const uint32_t id_o = idesc_f16(PM, PD, bf16, true);
    // K-major 128-byte-swizzled A (Q) and B (K) tiles: K-step k (16 dims) is at
    // byte 32 (k % 4) of the 64-dim half k / 4, halves 128 rows x 128 bytes apart
    const uint64_t dk0 = sw128_desc(base + P2_OFF_K, 16, 1024);
    const uint64_t dq0 = sw128_desc(base + P2_OFF_Q, 16, 1024);
    const uint64_t dv0 = sw128_desc(base + P2_OFF_V, PN * 128, 1024);
    int kc = 0, vc = 0, qc[2] = {0, 0}, pc[2] = {0, 0};
    bool ok = true;
    auto wait = [&](uint32_t bar, uint32_t parity) {
        if (!ok) return false;
        if (*abort_flag || !mbar_wait_bounded(bar, parity, a.wait_limit)) {
            pf_error(a);
            *abort_flag = 1;
            ok = false;
        }
        return ok;
    };
    auto issue_s = [&](int x, int ks) {   // S_x = Q_x K^T, K from ring stage ks
        const uint64_t dk = dk0 + (uint64_t)(ks * (KV_BYTES >> 4));
        const uint64_t dq = dq0 + (uint64_t)(x * (Q_BYTES >> 4));
#pragma unroll
        for (int k = 0; k < PD / 16; ++k) {
            const uint64_t off = (uint64_t)((((k >> 2) * (PN * 128)) + (k & 3) * 32) >> 4);
            umma_f16(tmem + x * PN, dq + off, dk + off, id_s, k > 0 ? 1u : 0u);
        }
        umma_commit(bb.sfull[x]);
    };
    auto issue_pv = [&](int x, int vs, int n) {   // O_x += P_x V, P_x in the first 64 columns of S_x
        const uint64_t dv = dv0 + (uint64_t)(vs * (KV_BYTES >> 4));
#pragma unroll
        for (int k = 0; k < PN / 16; ++k)   // K-step k: 16 tokens = P columns 8k .. 8k + 7, V row 16 k
            umma_f16_ts(tmem + TM2_O + x * PD, tmem + x * PN + 8 * k, dv + (uint64_t)((k * 16 * 128) >> 4), id_o,
                        (n > 0 || k > 0) ? 1u : 0u);
        umma_commit(bb.pvdone[x]);
    };
    for (int item = blockIdx.x; item < total && ok; item += gridDim.x) {
        const P2Item p = p2_item(a, item);
        const int nkv0 = p.t[0].nkv, nkv1 = p.t[1].nkv;
        if (!wait(bb.qfull[0], qc[0] & 1)) break;
        ++qc[0];
        if (nkv1 > 0) {
            if (!wait(bb.qfull[1], qc[1] & 1)) break;
            ++qc[1];
        }
        {   // S0(0), S1(0)
            const int ks = kc % P2_RK;
            if (!wait(bb.kfull[ks], (kc / P2_RK) & 1)) break;
            tc_fence_after_sync();
            issue_s(0, ks);
            if (nkv1 > 0) issue_s(1, ks);
            umma_commit(bb.kempty[ks]);
            ++kc;
        }
        for (int n = 0; n < nkv0 && ok; ++n) {
            const int vs = vc % P2_RV;
            const int ks = kc % P2_RK;                 // K tile n + 1
            const bool more0 = n + 1 < nkv0, more1 = n + 1 < nkv1;
            if (!wait(bb.pfull[0], pc[0] & 1)) break;
            ++pc[0];
            if (!wait(bb.vfull[vs], (vc / P2_RV) & 1)) break;
            tc_fence_after_sync();
            issue_pv(0, vs, n);
            if (more0) {
                if (!wait(bb.kfull[ks], (kc / P2_RK) & 1)) break;
                tc_fence_after_sync();
                issue_s(0, ks);
            }
            if (n < nkv1) {
                if (!wait(bb.pfull[1], pc[1] & 1)) break;
                ++pc[1];
                tc_fence_after_sync();
                issue_pv(1, vs, n);
                if (more1) issue_s(1, ks);             // more1 implies more0: K tile n + 1 is in
            }
            umma_commit(bb.vempty[vs]);
            ++vc;
            if (more0) {
                umma_commit(bb.kempty[ks]);
                ++kc;
            }
        }
    }
}

template <int KV>
__device__ void p2_softmax(uint8_t *smem, const PrefillArgs &a, const P2Bars &bb, uint32_t tmem,
                           volatile int *abort_flag, int total, int x) {
    const int lane = threadIdx.x & 31;
    const int quarter = (threadIdx.x >> 5) & 3;    // tensor-memory lanes 32 quarter .. + 31
    const int m = quarter * 32 + lane;             // this thread's query row in its tile
    const int tid = m;                             // 0 .. 127 within the tile's warpgroup
    const uint32_t trow = tmem + ((uint32_t)(quarter * 32) << 16);
    const uint32_t scol = (uint32_t)(x * PN), ocol = (uint32_t)(TM2_O + x * PD);
    uint8_t *qs = smem + P2_OFF_Q + x * Q_BYTES;
    const float sl2 = a.scale_log2;
    int sc = 0, pvc = 0, vcount = 0;   // S_x completed, PV_x issued, V tiles passed (tile 0 zeroes V)
    bool ok = true;
    auto wait = [&](uint32_t bar, uint32_t parity) {
        if (!ok) return false;
        const bool got = !*abort_flag && mbar_wait_bounded(bar, parity, a.wait_limit);
        if (!__all_sync(0xffffffffu, got)) {
            if (lane == 0) pf_error(a);
            *abort_flag = 1;
            ok = false;
        }
        return ok;
    };
    const int tok = m / a.G, hh = m - tok * a.G;
    // ---- an item's Q row into shared memory in the 128-byte-swizzled K-major
    // layout (zeros past the tile's new tokens).  Stored for the next item as
    // soon as this tile's last PV is done (every product that read Q_x is then
    // done), before the epilogue, so that the next S_x overlaps the epilogue.
    int q_item = -1;   // the item whose Q_x is in shared memory
    auto tile_of = [&](int it) {
        const P2Item p = p2_item(a, it);
        return x ? p.t[1] : p.t[0];   // (a run-time index would put the pair in local memory)
    };
    auto store_q = [&](int it, const PfTile &tq) {
        const bool v = tok < tq.ntok;
        const uint4 *src = reinterpret_cast<const uint4 *>(
            a.query + ((long long)(tq.q0 + tq.row0 + tok) * a.Hq + tq.kvh * a.G + hh) * PD);
#pragma unroll
        for (int c = 0; c < 16; ++c) {
            const uint4 q = v ? __ldg(src + c) : make_uint4(0, 0, 0, 0);
            *reinterpret_cast<uint4 *>(qs + (c >> 3) * (PM * 128) + m * 128 + (((c & 7) ^ (m & 7)) << 4)) = q;
        }
        fence_proxy_async_smem();
        mbar_arrive(bb.qfull[x]);
        q_item = it;
    };
    for (int item = blockIdx.x; item < total && ok; item += gridDim.x) {
        const PfTile t = tile_of(item);
        if (t.nkv == 0) continue;                  // the pair has no tile 1
        const bool valid = tok < t.ntok;
        const long long qrow = ((long long)(t.q0 + t.row0 + tok) * a.Hq + t.kvh * a.G + hh) * PD;
        if (q_item != item) store_q(item, t);
        const int vis = valid ? t.C + t.row0 + tok : 1;   // positions this row sees
        float mrun = -INFINITY, l = 0.f;
        for (int n = 0; n < t.nkv && ok; ++n) {
            if (!wait(bb.sfull[x], sc & 1)) break;
            ++sc;
            tc_fence_after_sync();
            // ---- the row of S, whole, in registers
            float s[PN];
#pragma unroll
            for (int q = 0; q < PN / 32; ++q) {
                uint32_t r[32];
                tmem_ld32(trow + scol + 32 * q, r);
#pragma unroll
                for (int c = 0; c < 32; ++c) s[32 * q + c] = __uint_as_float(r[c]);
            }
            tmem_wait_ld();
            const int t0 = n * PN;
            if (t0 + PN > vis) {   // the tile reaches past this row's position
#pragma unroll
                for (int c = 0; c < PN; ++c) s[c] = t0 + c < vis ? s[c] : -INFINITY;
            }
            // row maximum of the raw scores (scale > 0), eight partial maxima
            float mp[8];
#pragma unroll
            for (int j = 0; j < 8; ++j) mp[j] = s[j];
#pragma unroll
            for (int c = 8; c < PN; ++c) mp[c & 7] = fmaxf(mp[c & 7], s[c]);
            const float mx = fmaxf(fmaxf(fmaxf(mp[0], mp[1]), fmaxf(mp[2], mp[3])),
                                   fmaxf(fmaxf(mp[4], mp[5]), fmaxf(mp[6], mp[7]))) * sl2;
            // rescale decided per row, run warp-wide (tensor-memory accesses are
            // warp-collective); rows that do not grow scale by exactly 1
            const bool grow = mx > mrun + RESCALE_THRESHOLD;
            if (__any_sync(0xffffffffu, grow)) {
                const float nm = grow ? fmaxf(mrun, mx) : mrun;
                const float alpha = grow ? fast_exp2(mrun - nm) : 1.f;
                if (n > 0) {   // PV_x(n - 1) is complete (S_x(n) was committed after it)
#pragma unroll 1
                    for (int c4 = 0; c4 < PD / 32; ++c4) {
                        uint32_t o[32];
                        tmem_ld32(trow + ocol + c4 * 32, o);
                        tmem_wait_ld();
#pragma unroll
                        for (int c = 0; c < 32; ++c) o[c] = __float_as_uint(__uint_as_float(o[c]) * alpha);
                        tmem_st32(trow + ocol + c4 * 32, o);
                    }
                    tmem_wait_st();
                }
                l *= alpha;
                mrun = nm;
            }
            // ---- the sequence's last KV tile: V rows past the context are zeroed
            // (P is 0 there, but the slots may hold anything); tile 0 runs every
            // KV tile of the pair, and PV1(n) is issued after PV0(n)
            bool zeroed = false;
            if (x == 0) {
                const int vs = vcount % P2_RV;
                const int vphase = (vcount / P2_RV) & 1;
                ++vcount;
                if (t0 + PN > t.L) {
                    if (!wait(bb.vfull[vs], vphase)) break;
                    const int first = t.L - t0;
                    uint8_t *vt = smem + P2_OFF_V + vs * KV_BYTES;
                    for (int k = tid; k < 2 * PN * 8; k += 128) {
                        const int h = k / (PN * 8), rr = (k / 8) % PN, cc = k % 8;
                        if (rr >= first)
                            *reinterpret_cast<uint4 *>(vt + h * (PN * 128) + rr * 128 + cc * 16) =
                                make_uint4(0, 0, 0, 0);
                    }
                    zeroed = true;
                }
            }
            // ---- p = 2^(s scale log2(e) - m), packed two per column over the
            // first 64 columns of S (already read), and the row sum
            float lp[8];
#pragma unroll
            for (int j = 0; j < 8; ++j) lp[j] = 0.f;
#pragma unroll
            for (int h = 0; h < 2; ++h) {
                uint32_t r[32];
#pragma unroll
                for (int c = 0; c < 8; ++c) {   // tokens 64 h + 8 c .. + 7
                    float pv[8];
#pragma unroll
                    for (int j = 0; j < 8; ++j) {
                        pv[j] = fast_exp2(fmaf(s[64 * h + 8 * c + j], sl2, -mrun));
                        lp[j] += pv[j];
                    }
                    r[4 * c] = pack_p<KV>(pv[0], pv[1]);
                    r[4 * c + 1] = pack_p<KV>(pv[2], pv[3]);
                    r[4 * c + 2] = pack_p<KV>(pv[4], pv[5]);
                    r[4 * c + 3] = pack_p<KV>(pv[6], pv[7]);
                }
                tmem_st32(trow + scol + 32 * h, r);
            }
            l += ((lp[0] + lp[1]) + (lp[2] + lp[3])) + ((lp[4] + lp[5]) + (lp[6] + lp[7]));
            tmem_wait_st();
            if (zeroed) fence_proxy_async_smem();   // the zeroed V rows, for the tensor cores
            tc_fence_before_sync();
            mbar_arrive(bb.pfull[x]);
            ++pvc;
        }
        if (!ok) break;
        // ---- epilogue: O / l once this tile's last PV is done; the next
        // item's Q_x first, if it has this tile
        if (!wait(bb.pvdone[x], (pvc - 1) & 1)) break;
        tc_fence_after_sync();
        if (item + (int)gridDim.x < total) {
            const PfTile tn = tile_of(item + gridDim.x);
            if (tn.nkv > 0) store_q(item + gridDim.x, tn);
        }
        const bool bad = *pf_bad_slot(smem, P2_OFF_CTRL, pf_local(item)) == pf_local(item) + 1;
        const float inv = bad ? __int_as_float(0x7fc00000) : a.v_scale / l;
        uint16_t *orow = a.out + qrow;
#pragma unroll 1
        for (int c4 = 0; c4 < PD / 32; ++c4) {
            uint32_t o[32];
            tmem_ld32(trow + ocol + c4 * 32, o);
            tmem_wait_ld();
            if (valid) {
#pragma unroll
                for (int c = 0; c < 32; c += 8) {
                    uint4 v;
                    v.x = (uint32_t)out_bits<KV>(__uint_as_float(o[c]) * inv) |
                          ((uint32_t)out_bits<KV>(__uint_as_float(o[c + 1]) * inv) << 16);
                    v.y = (uint32_t)out_bits<KV>(__uint_as_float(o[c + 2]) * inv) |
                          ((uint32_t)out_bits<KV>(__uint_as_float(o[c + 3]) * inv) << 16);
                    v.z = (uint32_t)out_bits<KV>(__uint_as_float(o[c + 4]) * inv) |
                          ((uint32_t)out_bits<KV>(__uint_as_float(o[c + 5]) * inv) << 16);
                    v.w = (uint32_t)out_bits<KV>(__uint_as_float(o[c + 6]) * inv) |
                          ((uint32_t)out_bits<KV>(__uint_as_float(o[c + 7]) * inv) << 16);
                    *reinterpret_cast<uint4 *>(orow + c4 * 32 + c) = v;
                }
            }
        }
        tc_fence_before_sync();
    }
}

template <int KV>
__global__ void __launch_bounds__(P2_THREADS, 1) prefill2_kernel(const __grid_constant__ CUtensorMap tmk,
                                                                  const __grid_constant__ CUtensorMap tmv,
                                                                  const PrefillArgs a) {
    extern __shared__ uint8_t smem_raw[];
    uint8_t *smem = reinterpret_cast<uint8_t *>((reinterpret_cast<uintptr_t>(smem_raw) + 1023) & ~uintptr_t(1023));
    const P2Bars bb = p2_bars(smem);
    volatile int *abort_flag = reinterpret_cast<volatile int *>(smem + P2_OFF_CTRL + CTRL_ABORT);
    const int warp = threadIdx.x >> 5;
    const int total = *reinterpret_cast<volatile int *>(&a.hdr->pf2_items);   // written by the prep kernel
    if ((int)blockIdx.x >= total) return;   // no work item for this CTA (the whole CTA leaves)
    if (threadIdx.x == 0) {
        for (int s = 0; s < P2_RK; ++s) {
            mbar_init(bb.kfull[s], 1);
            mbar_init(bb.kempty[s], 1);
        }
        for (int s = 0; s < P2_RV; ++s) {
            mbar_init(bb.vfull[s], 1);
            mbar_init(bb.vempty[s], 1);
        }
        for (int x = 0; x < 2; ++x) {
            mbar_init(bb.sfull[x], 1);
            mbar_init(bb.pfull[x], 128);
            mbar_init(bb.pvdone[x], 1);
            mbar_init(bb.qfull[x], 128);
        }
        mbar_init(bb.flags, 1);            // all MMAs completed (before tensor memory is freed)
        for (int k = 0; k < BAD_SLOTS; ++k) *pf_bad_slot(smem, P2_OFF_CTRL, k) = 0;
        *abort_flag = 0;
        fence_mbar_init();
    }
    if (warp == 2) {   // this warp owns the tensor memory
        tmem_alloc(bb.tmem_slot, TMEM_COLS);
        tmem_relinquish();
    }
    tc_fence_before_sync();
    __syncthreads();
    tc_fence_after_sync();
    const uint32_t tmem = *reinterpret_cast<volatile uint32_t *>(smem + (bb.tmem_slot - smem_u32(smem)));
    // register split: the producer / MMA warpgroup gives registers to the two
    // softmax warpgroups (128 x 104 + 256 x 200 = 384 x 168, the launch's pool)
    if (warp >= 4) {
        regs_increase<P2_REGS_HIGH>();
        p2_softmax<KV>(smem, a, bb, tmem, abort_flag, total, (warp - 4) >> 2);
    } else {
        regs_decrease<P2_REGS_LOW>();
        if (warp < 2) {
            // both producers stream the pair's whole range: tile 0's, the longer one
            auto range = [&](int item) {
                const P2Item p = p2_item(a, item);
                return PfRange{p.t[0].seq, p.t[0].kvh, p.t[0].nkv, p.t[0].L, 0};
            };
            if (warp == 0) {
                const int off[1] = {P2_OFF_K};
                const BarRing full[1] = {bb.kfull};
                const BarRing empty[1] = {bb.kempty};
                const CUtensorMap *maps[1] = {&tmk};
                pf_stream<P2_RK, false, 1>(smem, off, P2_OFF_CTRL, full, empty, maps, a, abort_flag, total, range);
            } else {
                const int off[1] = {P2_OFF_V};
                const BarRing full[1] = {bb.vfull};
                const BarRing empty[1] = {bb.vempty};
                const CUtensorMap *maps[1] = {&tmv};
                pf_stream<P2_RV, false, 1>(smem, off, P2_OFF_CTRL, full, empty, maps, a, abort_flag, total, range);
            }
        } else if (warp == 2) {
            if ((threadIdx.x & 31) == 0) {
                p2_mma<KV>(smem, a, bb, tmem, abort_flag, total);
                // every MMA issued has completed before tensor memory is released
                umma_commit(bb.flags);
                mbar_wait_bounded(bb.flags, 0, WAIT_LIMIT);
            }
            __syncwarp();
        }
    }
    tc_fence_before_sync();
    __syncthreads();
    if (warp == 2) {
        tc_fence_after_sync();
        tmem_dealloc(tmem, TMEM_COLS);
    }
}

// One-time set-up of the two-tile kernel for a cache type: shared memory,
// grid, and whether it may run at all.  The register split assumes the
// kernel launches with P2_REGS_LAUNCH registers per thread; were it built with
// another count, the warpgroups' shares would not match the pool and the
// softmax warpgroups' register increase could wait forever -- then the kernel
// is never launched and pairs go to the one-tile kernel instead.
struct P2Setup {
    int grid = 0;
    bool usable = false;
    cudaError_t err = cudaSuccess;
};

template <int KV>
const P2Setup &prefill2_setup() {
    static P2Setup su;
    static std::once_flag once;
    std::call_once(once, [] {   // one CTA per SM
        su.err = cudaFuncSetAttribute(prefill2_kernel<KV>, cudaFuncAttributeMaxDynamicSharedMemorySize, P2_SMEM);
        int dev = 0, sms = 0;
        cudaFuncAttributes fa;
        if (su.err == cudaSuccess) su.err = cudaGetDevice(&dev);
        if (su.err == cudaSuccess) su.err = cudaDeviceGetAttribute(&sms, cudaDevAttrMultiProcessorCount, dev);
        if (su.err == cudaSuccess) su.err = cudaFuncGetAttributes(&fa, prefill2_kernel<KV>);
        su.grid = sms;
        su.usable = su.err == cudaSuccess && sms > 0 && fa.numRegs == P2_REGS_LAUNCH;
    });
    return su;
}

template <int KV>
int launch_prefill2_kv(const CUtensorMap &tmk, const CUtensorMap &tmv, const PrefillArgs &args, long long max_items,
                       cudaStream_t st) {
    const P2Setup &su = prefill2_setup<KV>();
    if (su.err != cudaSuccess) return PA_ERR_CUDA;
    if (!su.usable) return PA_ERR_UNSUPPORTED;
    const int g = (int)(max_items < su.grid ? (max_items > 0 ? max_items : 1) : su.grid);
    prefill2_kernel<KV><<<g, P2_THREADS, P2_SMEM, st>>>(tmk, tmv, args);
    return cuda_status(cudaGetLastError());
}

// One-time set-up of the one-tile kernel: shared memory and grid; for an FP8
// cache also the check that the kernel launches with the register count its
// register split assumes (otherwise it is never launched, see prefill_usable).
template <int KV, int MODE>
const P2Setup &prefill_setup() {
    static P2Setup su;
    static std::once_flag once;
    std::call_once(once, [] {   // one CTA per SM
        su.err = cudaFuncSetAttribute(prefill_kernel<KV, MODE>, cudaFuncAttributeMaxDynamicSharedMemorySize,
                                      PfL<KV>::SMEM);
        int dev = 0, sms = 0;
        cudaFuncAttributes fa;
        if (su.err == cudaSuccess) su.err = cudaGetDevice(&dev);
        if (su.err == cudaSuccess) su.err = cudaDeviceGetAttribute(&sms, cudaDevAttrMultiProcessorCount, dev);
        if (su.err == cudaSuccess) su.err = cudaFuncGetAttributes(&fa, prefill_kernel<KV, MODE>);
        su.grid = sms;
        su.usable = su.err == cudaSuccess && sms > 0 && (!PfL<KV>::F8 || fa.numRegs == PfL<KV>::LAUNCH_REGS);
    });
    return su;
}

template <int KV, int MODE>
int launch_prefill_kv(const CUtensorMap &tmk, const CUtensorMap &tmv, const PrefillArgs &args, long long max_items,
                      cudaStream_t st) {
    const P2Setup &su = prefill_setup<KV, MODE>();
    if (su.err != cudaSuccess) return PA_ERR_CUDA;
    if (!su.usable) return PA_ERR_UNSUPPORTED;
    const int grid = su.grid;
    const int g = (int)(max_items < grid ? (max_items > 0 ? max_items : 1) : grid);
    prefill_kernel<KV, MODE><<<g, PfL<KV>::THREADS, PfL<KV>::SMEM, st>>>(tmk, tmv, args);
    return cuda_status(cudaGetLastError());
}

}  // namespace

int launch_prefill(int kv, const CUtensorMap &tmk, const CUtensorMap &tmv, const PrefillArgs &args,
                   long long max_items, cudaStream_t st) {
    if (kv == PA_KV_BF16) return launch_prefill_kv<PA_KV_BF16, PF_CAUSAL>(tmk, tmv, args, max_items, st);
    if (kv == PA_KV_F16) return launch_prefill_kv<PA_KV_F16, PF_CAUSAL>(tmk, tmv, args, max_items, st);
    if (kv == PA_KV_FP8_E4M3) return launch_prefill_kv<PA_KV_FP8_E4M3, PF_CAUSAL>(tmk, tmv, args, max_items, st);
    return PA_ERR_UNSUPPORTED;
}

int launch_shared_ranges(const CUtensorMap &tmk, const CUtensorMap &tmv, const PrefillArgs &args,
                         long long max_items, cudaStream_t st) {
    return launch_prefill_kv<PA_KV_F16, PF_SHARED>(tmk, tmv, args, max_items, st);
}

bool prefill_usable(int kv) {
    if (kv == PA_KV_BF16) return prefill_setup<PA_KV_BF16, PF_CAUSAL>().usable;
    if (kv == PA_KV_F16) return prefill_setup<PA_KV_F16, PF_CAUSAL>().usable;
    if (kv == PA_KV_FP8_E4M3) return prefill_setup<PA_KV_FP8_E4M3, PF_CAUSAL>().usable;
    return false;
}

bool prefill2_usable(int kv) {
    if (kv == PA_KV_BF16) return prefill2_setup<PA_KV_BF16>().usable;
    if (kv == PA_KV_F16) return prefill2_setup<PA_KV_F16>().usable;
    return false;
}

int launch_prefill2(int kv, const CUtensorMap &tmk, const CUtensorMap &tmv, const PrefillArgs &args,
                    long long max_items, cudaStream_t st) {
    if (kv == PA_KV_BF16) return launch_prefill2_kv<PA_KV_BF16>(tmk, tmv, args, max_items, st);
    if (kv == PA_KV_F16) return launch_prefill2_kv<PA_KV_F16>(tmk, tmv, args, max_items, st);
    return PA_ERR_UNSUPPORTED;
}

}  // namespace pa
