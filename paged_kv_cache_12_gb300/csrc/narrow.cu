// Paged attention for work items of few query rows -- the new tokens of a
// speculative step, a few per sequence, or the members of a shared-prefix
// group over a range of their shared blocks -- on the 5th-generation tensor
// cores.
//
// What is computed is the one-tile kernel's (prefill.cu): each query row
// attends to the positions it sees through the block table (deepsonar page,
// section 2.5 for new tokens; section 2.3 for parallel samples sharing a
// prompt's blocks).  There an item of at most 32 rows (4 speculative tokens x
// 8 heads) fills a quarter of the 128-row tile, and its softmax runs over 128
// positions per row while three quarters of the tile's rows are padding.
// Here the item's 32 rows are copied into all four 32-row quarters of the
// tile, and the softmax warp of quarter q takes only tokens 32 q .. 32 q + 31
// of every 128-token KV tile: its P row is zero elsewhere, so after
// O += P V lane (q, r) of O holds row r's attention over quarter q's tokens,
// with quarter q's own running maximum and row sum.  Each thread therefore
// owns one row in one quarter -- 32 scores per tile, its maximum and sum in
// registers, no exchange between warps -- and the four partial results of a
// row are merged once, at the end of the item, through a scratch area of the
// workspace (m = max of the four, O and l scaled by 2^(m_q - m) and summed).
//
// Products (M 128, N 128, K 16 per instruction):
//   S = Q' K^T   A = Q' (the four copies of Q, tensor memory), B = K tile;
//   O += P V     A = P (tensor memory, written by the softmax), B = V tile.
// Tensor memory: S in two buffers of 128 columns, P and Q' (two fp16/bf16
// per column) 64 each, O 128: all 512 columns, one CTA per SM; shared memory
// holds only the K/V rings (and an FP8 cache's staging rings).
//
// One CTA per SM, persistent over the item list; warps:
//   0, 1   producers: K and V tiles of 128 tokens by TMA through the block
//          table (16-bit caches: 4-stage K and 3-stage V rings; FP8: the
//          codes, 3-stage staging rings before 2-stage 16-bit rings);
//   2, 3   MMA issuers (one thread each): warp 2 the S products, warp 3 the
//          PV products -- one thread takes about 100 cycles per tcgen05.mma,
//          two streams halve the time the products hold the pipeline;
//   4-7    softmax, quarter q = warp - 4, one row per thread;
//   8-15   FP8 only: the staged codes to fp16 tiles, four warps per cache.
// Every wait is bounded; warp-collective instructions run in warp-uniform
// control flow; tensor memory is released on every path.

#include <cmath>
#include <mutex>

#include "prefill_common.cuh"

namespace pa {
namespace {

constexpr int NR = NARROW_ROWS;           // query rows of an item (padded): one per lane of a quarter
constexpr int NW_SOFT0 = 4;               // first softmax warp
// tensor memory: S 0, S 1 (PN fp32 columns each), P (PN / 2: two 16-bit
// values per column), Q' (PD / 2), O (PD)
constexpr int NW_S = 0, NW_P = 2 * PN, NW_Q = NW_P + PN / 2, NW_O = NW_Q + PD / 2;
constexpr int NW_TMEM_COLS = 512;
static_assert(NR == 32 && PM == 4 * NR, "four copies of the item's rows fill the tile");
static_assert(PN == 128, "a quarter of a KV tile per softmax warp: 32 tokens");
static_assert(NW_O + PD <= NW_TMEM_COLS, "tensor-memory columns");

constexpr int NW_MAXST = 4;   // barrier slots per ring

#ifndef PA_NW_RK16
#define PA_NW_RK16 4
#endif
#ifndef PA_NW_RV16
#define PA_NW_RV16 3
#endif
#ifndef PA_NW_R8
#define PA_NW_R8 2
#endif
#ifndef PA_NW_S8
#define PA_NW_S8 3
#endif

// Shared memory per cache type: K and V rings of R 16-bit stages (the TMA
// fills them, or for an FP8 cache the converting warps from staging rings of
// S8 stages of codes).
template <int KV>
struct NwL {
    static constexpr bool F8 = KV == PA_KV_FP8_E4M3;
    static constexpr int RK = F8 ? PA_NW_R8 : PA_NW_RK16;   // 16-bit K ring stages
    static constexpr int RV = F8 ? PA_NW_R8 : PA_NW_RV16;   // 16-bit V ring stages
    static constexpr int S8 = F8 ? PA_NW_S8 : 0;            // FP8 staging stages
    static constexpr int OFF_K = 0;
    static constexpr int OFF_V = RK * KV_BYTES;
    static constexpr int OFF_K8 = (RK + RV) * KV_BYTES;
    static constexpr int OFF_V8 = OFF_K8 + S8 * F8_BYTES;
    static constexpr int OFF_CTRL = OFF_V8 + S8 * F8_BYTES;
    static constexpr int SMEM = OFF_CTRL + CTRL_BYTES + 1024;   // + alignment slack
    // 16-bit caches: warps 0 / 1 produce K / V, 2 / 3 issue the MMAs, 4-7 run
    // the softmax.  FP8 caches: warps 0 / 1 stage the codes and 8-11 / 12-15
    // convert K / V, a quarter of the rows each (two per SM sub-partition).
    static constexpr int THREADS = (F8 ? 16 : 8) * 32;
    static_assert(SMEM <= 227 * 1024, "shared memory of one CTA");
    static_assert(OFF_K8 % 1024 == 0, "swizzled tiles 1024-byte aligned");
    static_assert(RK <= NW_MAXST && RV <= NW_MAXST && S8 <= NW_MAXST, "ring stages");
    static_assert(!F8 || RK == RV, "the converting warps fill K and V rings of one depth");
};

struct NwBars {
    // sfull / sfree: S buffers; pfull / pvdone: P buffers (by PV-number parity)
    BarRing kfull, kempty, vfull, vempty, k8full, v8full, k8empty, v8empty;   // NW_MAXST each
    BarRing sfull, sfree, pfull, pvdone;                                      // 2 each
    uint32_t qfull, merged, tmem_slot, flags;                                 // shared addresses
};
static_assert(8 * (8 * NW_MAXST + 8 + 4) <= CTRL_BAD, "control block layout");

__device__ __forceinline__ NwBars nw_bars(uint8_t *smem, int off_ctrl) {
    uint32_t a = smem_u32(smem + off_ctrl);
    NwBars b;
    BarRing *rings[8] = {&b.kfull, &b.kempty, &b.vfull, &b.vempty, &b.k8full, &b.v8full, &b.k8empty, &b.v8empty};
    for (int r = 0; r < 8; ++r) rings[r]->base = a, a += 8 * NW_MAXST;
    BarRing *pairs[4] = {&b.sfull, &b.sfree, &b.pfull, &b.pvdone};
    for (int r = 0; r < 4; ++r) pairs[r]->base = a, a += 16;
    b.qfull = a, a += 8;
    b.merged = a, a += 8;
    b.tmem_slot = a, a += 8;
    b.flags = a;
    return b;
}

// Work items: causal row tiles come from their own list, shared ranges from
// the decode call's list; the prep kernel writes their counts.
template <int MODE>
__device__ __forceinline__ int nw_total(const PrefillArgs &a) {
    if constexpr (MODE == PF_SHARED)
        return *reinterpret_cast<volatile int *>(&a.hdr->pf_items);
    else
        return *reinterpret_cast<volatile int *>(&a.hdr->pfn_items);
}

__device__ __forceinline__ void prefetch_l2(const void *p) { asm volatile("prefetch.global.L2 [%0];" ::"l"(p)); }

// The causal item list: items below `whole` are whole (sequence, kv head)
// items; each later one is one of k pieces of the KV range of one of the last
// items (the prep kernel splits the last, partial round of items so that it
// fills the grid).  Shared ranges are never split.
struct NwSplit {
    int whole, k;
};

template <int MODE>
__device__ __forceinline__ NwSplit nw_split(const PrefillArgs &a, int total) {
    if constexpr (MODE == PF_SHARED)
        return NwSplit{total, 1};
    else
        return NwSplit{*reinterpret_cast<volatile int *>(&a.hdr->pfn_whole),
                       *reinterpret_cast<volatile int *>(&a.hdr->pfn_split)};
}

template <int MODE>
__device__ __forceinline__ PfTile nw_item(const PrefillArgs &a, const NwSplit &sp, int item) {
    if constexpr (MODE == PF_SHARED) {
        return pf_shared_item(a, item);
    } else {
        if (item < sp.whole) return pf_tile(a, item);
        const int j = item - sp.whole, sid = j / sp.k, piece = j - sid * sp.k;
        PfTile t = pf_tile(a, sp.whole + sid);
        // KV tiles [n0, n1) of the item's range; positions relative to the piece
        const int n0 = piece * t.nkv / sp.k, n1 = (piece + 1) * t.nkv / sp.k;
        t.kv0 = n0 * PN;
        t.L = min(n1 * PN, t.L) - t.kv0;
        t.C -= t.kv0;
        t.nkv = n1 - n0;
        t.piece = piece;
        t.np = sp.k;
        t.sid = sid;
        return t;
    }
}

// ----------------------------------------------------------- MMA issuers

template <int KV, int MODE>
__device__ void nw_mma(uint8_t *smem, const PrefillArgs &a, const NwSplit &sp, const NwBars &bb, uint32_t tmem,
                       volatile int *abort_flag, int total, bool pv_role) {
    using L = NwL<KV>;
    constexpr int RK = L::RK, RV = L::RV;
    constexpr bool BF = KV == PA_KV_BF16;
    const uint32_t base = smem_u32(smem);
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
    int it = 0;
    if (!pv_role) {
        const uint32_t id_s = idesc_f16(PM, PN, BF, false);
        // Q' (A) in tensor memory, two dims per column; K (B) K-major: 128-byte
        // rows of 64 dims, one per token, the next 64 dims PN rows further.
        // K-step k (16 dims): columns 8 k .. 8 k + 7 of Q', byte 32 (k % 4)
        // of K's 64-dim block k / 4.
        const uint64_t dk0 = sw128_desc(base + L::OFF_K, 16, 1024);
        int kc = 0, sc = 0;
        for (int item = blockIdx.x; item < total && ok; item += gridDim.x, ++it) {
            const PfTile t = nw_item<MODE>(a, sp, item);
            if (!wait(bb.qfull, it & 1)) break;   // this item's Q' is in tensor memory
            for (int n = 0; n < t.nkv && ok; ++n) {   // S(n) into tensor-memory buffer sc & 1
                const int ks = kc % RK, b = sc & 1;
                if (!wait(bb.kfull[ks], (kc / RK) & 1)) break;
                if (sc >= 2 && !wait(bb.sfree[b], ((sc >> 1) - 1) & 1)) break;
                tc_fence_after_sync();
                const uint64_t dk = dk0 + (uint64_t)(ks * (KV_BYTES >> 4));
#pragma unroll
                for (int k = 0; k < PD / 16; ++k)
                    umma_f16_ts(tmem + NW_S + b * PN, tmem + NW_Q + 8 * k,
                                dk + (uint64_t)((((k >> 2) * (PN * 128)) + (k & 3) * 32) >> 4), id_s, k > 0 ? 1u : 0u);
                umma_commit(bb.sfull[b]);
                umma_commit(bb.kempty[ks]);
                ++kc;
                ++sc;
            }
        }
    } else {
        const uint32_t id_o = idesc_f16(PM, PD, BF, true);
        // V (B) with N (dims) contiguous: 128-byte rows of 64 dims, one per
        // token (K); the next 64 dims PN rows further.  K-step k (16 tokens):
        // P columns 8 k .. 8 k + 7, V rows 16 k ..
        const uint64_t dv0 = sw128_desc(base + L::OFF_V, PN * 128, 1024);
        int vc = 0, pc = 0;
        for (int item = blockIdx.x; item < total && ok; item += gridDim.x, ++it) {
            const PfTile t = nw_item<MODE>(a, sp, item);
            for (int n = 0; n < t.nkv && ok; ++n) {
                const int pb = pc & 1;   // barrier parity of PV number pc (one P buffer)
                if (!wait(bb.pfull[pb], (pc >> 1) & 1)) break;
                ++pc;
                const int vs = vc % RV;
                if (!wait(bb.vfull[vs], (vc / RV) & 1)) break;
                tc_fence_after_sync();
                const uint64_t dv = dv0 + (uint64_t)(vs * (KV_BYTES >> 4));
#pragma unroll
                for (int k = 0; k < PN / 16; ++k)
                    umma_f16_ts(tmem + NW_O, tmem + NW_P + 8 * k,
                                dv + (uint64_t)((k * 16 * 128) >> 4), id_o, (n > 0 || k > 0) ? 1u : 0u);
                umma_commit(bb.pvdone[pb]);
                umma_commit(bb.vempty[vs]);
                ++vc;
            }
        }
    }
}

// ------------------------------------------------------------- softmax

template <int KV, int MODE>
__device__ void nw_softmax(uint8_t *smem, const PrefillArgs &a, const NwSplit &sp, const NwBars &bb, uint32_t tmem,
                           volatile int *abort_flag, int total) {
    using L = NwL<KV>;
    constexpr int RV = L::RV;
    const int lane = threadIdx.x & 31;            // the row r of the item
    const int quarter = (threadIdx.x >> 5) & 3;   // tensor-memory lanes 32 quarter .. + 31; tokens 32 quarter ..
    const int tl = quarter * 32 + lane;           // this thread's tensor-memory lane
    const uint32_t trow = tmem + ((uint32_t)(quarter * 32) << 16);
    const float sl2 = a.scale_log2;
    // this CTA's merge scratch: per item parity, O as [quarter][dim][row] and
    // (m, l) as [quarter][row]
    float *scr = reinterpret_cast<float *>(a.scratch + (size_t)blockIdx.x * NW_SCRATCH_PER_CTA);
    int sc = 0, g = 0, vcount = 0, it = 0, mph = 0;   // mph: phases of `merged` used
    bool ok = true;
    // every thread of a warp takes the same decision, so warp-collective
    // instructions are never reached by part of a warp
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
    // Q': this thread's lane holds row `lane` of the item (every quarter a
    // copy), 128 dims two per column; zeros past the item's rows
    auto q_src = [&](const PfTile &tq) -> const uint4 * {
        const int tok = lane / a.G, hh = lane - tok * a.G;
        if (tok >= tq.ntok) return nullptr;
        return reinterpret_cast<const uint4 *>(a.query +
                                               ((long long)(tq.q0 + tq.row0 + tok) * a.Hq + tq.kvh * a.G + hh) * PD);
    };
    auto store_q = [&](const PfTile &tq) {
        const uint4 *src = q_src(tq);
#pragma unroll
        for (int h = 0; h < 2; ++h) {
            uint32_t r[32];
#pragma unroll
            for (int c = 0; c < 8; ++c) {
                const uint4 x = src ? __ldg(src + 8 * h + c) : make_uint4(0, 0, 0, 0);
                r[4 * c] = x.x;
                r[4 * c + 1] = x.y;
                r[4 * c + 2] = x.z;
                r[4 * c + 3] = x.w;
            }
            tmem_st32(trow + NW_Q + 32 * h, r);
        }
        tmem_wait_st();
        tc_fence_before_sync();
        mbar_arrive(bb.qfull);
    };
    // P columns of the other quarters' tokens stay zero: each thread writes
    // only its quarter's 16 columns
    {
        uint32_t z[32];
#pragma unroll
        for (int c = 0; c < 32; ++c) z[c] = 0;
        tmem_st32(trow + NW_P, z);
        tmem_st32(trow + NW_P + 32, z);
        tmem_wait_st();
    }
    if ((int)blockIdx.x < total) store_q(nw_item<MODE>(a, sp, blockIdx.x));
    for (int item = blockIdx.x; item < total && ok; item += gridDim.x, ++it) {
        const PfTile t = nw_item<MODE>(a, sp, item);
        const bool has_next = item + (int)gridDim.x < total;
        const PfTile tn = nw_item<MODE>(a, sp, has_next ? item + (int)gridDim.x : item);
        if (has_next) {
            if (const uint4 *src = q_src(tn)) {
                prefetch_l2(src);
                prefetch_l2(src + 8);
            }
        }
        // positions this row sees: up to its own new token (causal), or the
        // whole range (shared); the first row's bound decides whether a tile
        // needs the mask at all
        const int tok = lane / a.G;
        const int vis0 = MODE == PF_SHARED ? t.L : t.C + t.row0;
        const int vis = MODE == PF_SHARED ? t.L : min(t.C + t.row0 + tok, t.L);
        float mrun = -INFINITY, l = 0.f;
        for (int n = 0; n < t.nkv && ok; ++n) {
            // ---- this row's scores for this quarter's 32 tokens of the tile
            const int b = sc & 1;
            if (!wait(bb.sfull[b], (sc >> 1) & 1)) break;
            ++sc;
            tc_fence_after_sync();
            float s[32];
            {
                uint32_t r[32];
                tmem_ld32(trow + NW_S + b * PN + 32 * quarter, r);
                tmem_wait_ld();
#pragma unroll
                for (int c = 0; c < 32; ++c) s[c] = __uint_as_float(r[c]);
            }
            tc_fence_before_sync();
            mbar_arrive(bb.sfree[b]);
            // the item's last S is done, and with it every product that read
            // Q': the next item's rows go in now
            if (n + 1 == t.nkv && has_next) store_q(tn);
            const int t0 = n * PN;
            if (t0 + PN > vis0) {
                const int first = vis - (t0 + 32 * quarter);   // tokens c >= first are not seen
#pragma unroll
                for (int c = 0; c < 32; ++c) s[c] = c < first ? s[c] : -INFINITY;
            }
            // ---- the running maximum of this row over this quarter's tokens,
            // rescaled only when it grows by more than 2^8 (O's row then in
            // tensor memory); the branch is warp-collective, so when any row of
            // the warp grows every lane takes it, the others scaling by 1.
            float mx;
            {
                float m4[4];
#pragma unroll
                for (int j = 0; j < 4; ++j)
                    m4[j] = fmaxf(fmaxf(s[8 * j], s[8 * j + 1]), fmaxf(s[8 * j + 2], s[8 * j + 3]));
#pragma unroll
                for (int j = 0; j < 4; ++j)
                    m4[j] = fmaxf(m4[j], fmaxf(fmaxf(s[8 * j + 4], s[8 * j + 5]), fmaxf(s[8 * j + 6], s[8 * j + 7])));
                mx = fmaxf(fmaxf(m4[0], m4[1]), fmaxf(m4[2], m4[3])) * sl2;
            }
            const bool grow = mx > mrun + RESCALE_THRESHOLD;
            if (__any_sync(0xffffffffu, grow)) {
                const float nm = grow ? mx : mrun;
                const float alpha = grow ? fast_exp2(mrun - nm) : 1.f;   // 0 from a maximum of -inf
                if (n > 0) {   // O holds PV up to number g - 1: rescale its row
                    if (!wait(bb.pvdone[(g - 1) & 1], ((g - 1) >> 1) & 1)) break;
                    tc_fence_after_sync();
#pragma unroll 1
                    for (int c4 = 0; c4 < PD / 32; ++c4) {
                        uint32_t o[32];
                        tmem_ld32(trow + NW_O + 32 * c4, o);
                        tmem_wait_ld();
#pragma unroll
                        for (int c = 0; c < 32; ++c) o[c] = __float_as_uint(__uint_as_float(o[c]) * alpha);
                        tmem_st32(trow + NW_O + 32 * c4, o);
                    }
                    tmem_wait_st();
                }
                l *= alpha;
                mrun = nm;
            }
            // ---- the last KV tile: V rows past the range are zeroed (P is 0
            // there, but the rows hold stale bits)
            const int vs = vcount % RV;
            const int vphase = (vcount / RV) & 1;
            ++vcount;
            const bool zero_v = t0 + PN > t.L;
            if (zero_v) {
                if (!wait(bb.vfull[vs], vphase)) break;
                const int first = t.L - t0;
                uint8_t *vt = smem + L::OFF_V + vs * KV_BYTES;
                for (int k = tl; k < 2 * PN * 8; k += 128) {
                    const int h = k / (PN * 8), rr = (k / 8) % PN, cc = k % 8;
                    if (rr >= first)
                        *reinterpret_cast<uint4 *>(vt + h * (PN * 128) + rr * 128 + cc * 16) = make_uint4(0, 0, 0, 0);
                }
            }
            // ---- p = 2^(s scale log2(e) - m) for this quarter's tokens, into
            // this thread's 16 columns of P (PV number g - 1 read it before);
            // while no token of the quarter has been seen (maximum -inf) p is 0
            const float msub = mrun == -INFINITY ? 0.f : mrun;
            uint32_t pw[16];
            float lp[4] = {0.f, 0.f, 0.f, 0.f};
#pragma unroll
            for (int c = 0; c < 16; ++c) {
                const float p0 = fast_exp2(fmaf(s[2 * c], sl2, -msub));
                const float p1 = fast_exp2(fmaf(s[2 * c + 1], sl2, -msub));
                lp[c & 3] += p0 + p1;
                pw[c] = pack_p<KV>(p0, p1);
            }
            l += (lp[0] + lp[1]) + (lp[2] + lp[3]);
            if (g >= 1 && !wait(bb.pvdone[(g - 1) & 1], ((g - 1) >> 1) & 1)) break;
            tmem_st16(trow + NW_P + 16 * quarter, pw);
            tmem_wait_st();
            if (zero_v) fence_proxy_async_smem();   // the zeroed V rows, for the tensor cores
            tc_fence_before_sync();
            mbar_arrive(bb.pfull[g & 1]);
            ++g;
        }
        if (!ok) break;
        // ---- epilogue once the item's last PV (number g - 1) is done: the four
        // quarters' partial rows, through the scratch area, into one
        if (!wait(bb.pvdone[(g - 1) & 1], ((g - 1) >> 1) & 1)) break;
        tc_fence_after_sync();
        float *so = scr + (it & 1) * (NW_SCRATCH_PER_CTA / 8);      // [quarter][dim][row]
        float2 *sml = reinterpret_cast<float2 *>(so + 4 * PD * 32);  // [quarter][row]
#pragma unroll 1
        for (int c4 = 0; c4 < PD / 32; ++c4) {
            uint32_t o[32];
            tmem_ld32(trow + NW_O + 32 * c4, o);
            tmem_wait_ld();
#pragma unroll
            for (int c = 0; c < 32; ++c) so[(quarter * PD + 32 * c4 + c) * 32 + lane] = __uint_as_float(o[c]);
        }
        sml[quarter * 32 + lane] = make_float2(mrun, l);
        tc_fence_before_sync();
        __threadfence_block();
        mbar_arrive(bb.merged);
        if (!wait(bb.merged, mph & 1)) break;
        ++mph;
        // row `lane`: its maximum over all positions, each quarter's weight,
        // its sum; this thread then writes dims 32 quarter .. 32 quarter + 31
        float2 mlq[4];
#pragma unroll
        for (int q = 0; q < 4; ++q) mlq[q] = __ldcg(sml + q * 32 + lane);
        const float mall = fmaxf(fmaxf(mlq[0].x, mlq[1].x), fmaxf(mlq[2].x, mlq[3].x));
        float wq[4], lall = 0.f;
#pragma unroll
        for (int q = 0; q < 4; ++q) {
            wq[q] = mlq[q].x == -INFINITY ? 0.f : fast_exp2(mlq[q].x - mall);
            lall += wq[q] * mlq[q].y;
        }
        const bool bad = *pf_bad_slot(smem, L::OFF_CTRL, pf_local(item)) == pf_local(item) + 1;
        const float qnan = __int_as_float(0x7fc00000);
        const int hh = lane - tok * a.G;
        const bool valid = tok < t.ntok;
        float ov[32];
#pragma unroll
        for (int c = 0; c < 32; ++c) {
            const int d = 32 * quarter + c;
            float x = 0.f;
#pragma unroll
            for (int q = 0; q < 4; ++q) x = fmaf(wq[q], __ldcg(so + (q * PD + d) * 32 + lane), x);
            ov[c] = x;
        }
        if constexpr (MODE == PF_CAUSAL) {
            if (t.np > 1) {
                // A piece of a split item: its partial rows (unnormalised O and
                // (m, l)) into the split area; the CTA that completes the item's
                // last piece (its ticket) merges the pieces into the output.
                const NwSplitArea sa = nw_split_area(a.scratch);
                const int slot = t.sid * t.np + t.piece;
                float *po = sa.o + ((size_t)slot * 32 + lane) * PD + 32 * quarter;
#pragma unroll
                for (int c = 0; c < 32; c += 4)
                    *reinterpret_cast<float4 *>(po + c) =
                        bad ? make_float4(qnan, qnan, qnan, qnan) : make_float4(ov[c], ov[c + 1], ov[c + 2], ov[c + 3]);
                if (quarter == 0) sa.ml[slot * 32 + lane] = bad ? make_float2(qnan, qnan) : make_float2(mall, lall);
                __threadfence();
                mbar_arrive(bb.merged);
                if (!wait(bb.merged, mph & 1)) break;
                ++mph;
                volatile int *last = reinterpret_cast<volatile int *>(smem + L::OFF_CTRL + CTRL_ABORT + 4);
                if (tl == 0) *last = atomicAdd(sa.tickets + t.sid, 1) == t.np - 1;
                mbar_arrive(bb.merged);
                if (!wait(bb.merged, mph & 1)) break;
                ++mph;
                if (!*last) continue;
                __threadfence();
                const int s0 = t.sid * t.np;
                float mp = -INFINITY;
                for (int p = 0; p < t.np; ++p) mp = fmaxf(mp, __ldcg(sa.ml + (s0 + p) * 32 + lane).x);
                float lp = 0.f, acc[32];
#pragma unroll
                for (int c = 0; c < 32; ++c) acc[c] = 0.f;
                for (int p = 0; p < t.np; ++p) {
                    const float2 ml = __ldcg(sa.ml + (s0 + p) * 32 + lane);
                    const float w = fast_exp2(ml.x - mp);   // NaN from a piece that met a bad block id
                    lp += w * ml.y;
                    const float *pp = sa.o + ((size_t)(s0 + p) * 32 + lane) * PD + 32 * quarter;
#pragma unroll
                    for (int c = 0; c < 32; c += 4) {
                        const float4 x = __ldcg(reinterpret_cast<const float4 *>(pp + c));
                        acc[c] = fmaf(w, x.x, acc[c]);
                        acc[c + 1] = fmaf(w, x.y, acc[c + 1]);
                        acc[c + 2] = fmaf(w, x.z, acc[c + 2]);
                        acc[c + 3] = fmaf(w, x.w, acc[c + 3]);
                    }
                }
                if (valid) {
                    const float inv = a.v_scale / lp;
                    uint16_t *orow =
                        a.out + ((long long)(t.q0 + t.row0 + tok) * a.Hq + t.kvh * a.G + hh) * PD + 32 * quarter;
#pragma unroll
                    for (int c = 0; c < 32; c += 8) {
                        uint4 v;
                        v.x = (uint32_t)out_bits<KV>(acc[c] * inv) | ((uint32_t)out_bits<KV>(acc[c + 1] * inv) << 16);
                        v.y = (uint32_t)out_bits<KV>(acc[c + 2] * inv) | ((uint32_t)out_bits<KV>(acc[c + 3] * inv) << 16);
                        v.z = (uint32_t)out_bits<KV>(acc[c + 4] * inv) | ((uint32_t)out_bits<KV>(acc[c + 5] * inv) << 16);
                        v.w = (uint32_t)out_bits<KV>(acc[c + 6] * inv) | ((uint32_t)out_bits<KV>(acc[c + 7] * inv) << 16);
                        *reinterpret_cast<uint4 *>(orow + c) = v;
                    }
                }
                continue;
            }
        }
        if constexpr (MODE == PF_SHARED) {
            // the member's partial row of this shared range: unnormalised O
            // (times the V scale) and (m, l) -- the decode kernel's partial
            // format -- at row part_off[member] + the range's partition index
            if (valid) {
                const long long wrow = ((long long)a.part_off[t.q0 + tok] + t.kv0 / a.pt) * a.Hq + t.kvh * a.G + hh;
                float *prow = a.ws_o + wrow * PD + 32 * quarter;
#pragma unroll
                for (int c = 0; c < 32; c += 4)
                    *reinterpret_cast<float4 *>(prow + c) =
                        bad ? make_float4(qnan, qnan, qnan, qnan)
                            : make_float4(ov[c] * a.v_scale, ov[c + 1] * a.v_scale, ov[c + 2] * a.v_scale,
                                          ov[c + 3] * a.v_scale);
                if (quarter == 0) a.ws_ml[wrow] = bad ? make_float2(qnan, qnan) : make_float2(mall, lall);
            }
        } else if (valid) {
            const float inv = bad ? qnan : a.v_scale / lall;
            uint16_t *orow = a.out + ((long long)(t.q0 + t.row0 + tok) * a.Hq + t.kvh * a.G + hh) * PD + 32 * quarter;
#pragma unroll
            for (int c = 0; c < 32; c += 8) {
                uint4 v;
                v.x = (uint32_t)out_bits<KV>(ov[c] * inv) | ((uint32_t)out_bits<KV>(ov[c + 1] * inv) << 16);
                v.y = (uint32_t)out_bits<KV>(ov[c + 2] * inv) | ((uint32_t)out_bits<KV>(ov[c + 3] * inv) << 16);
                v.z = (uint32_t)out_bits<KV>(ov[c + 4] * inv) | ((uint32_t)out_bits<KV>(ov[c + 5] * inv) << 16);
                v.w = (uint32_t)out_bits<KV>(ov[c + 6] * inv) | ((uint32_t)out_bits<KV>(ov[c + 7] * inv) << 16);
                *reinterpret_cast<uint4 *>(orow + c) = v;
            }
        }
    }
}

template <int KV, int MODE>
__global__ void __launch_bounds__(NwL<KV>::THREADS, 1) narrow_kernel(const __grid_constant__ CUtensorMap tmk,
                                                                   const __grid_constant__ CUtensorMap tmv,
                                                                   const PrefillArgs a) {
    extern __shared__ uint8_t smem_raw[];
    uint8_t *smem = reinterpret_cast<uint8_t *>((reinterpret_cast<uintptr_t>(smem_raw) + 1023) & ~uintptr_t(1023));
    using L = NwL<KV>;
    const NwBars bb = nw_bars(smem, L::OFF_CTRL);
    volatile int *abort_flag = reinterpret_cast<volatile int *>(smem + L::OFF_CTRL + CTRL_ABORT);
    const int warp = threadIdx.x >> 5;
    const int total = nw_total<MODE>(a);   // written by the prep kernel
    if ((int)blockIdx.x >= total) return;  // no work item for this CTA (the whole CTA leaves)
    const NwSplit sp = nw_split<MODE>(a, total);
    if (threadIdx.x == 0) {
        constexpr uint32_t fill = L::F8 ? 4 : 1;   // FP8: four converting warps per ring
        for (int s = 0; s < L::RK; ++s) {
            mbar_init(bb.kfull[s], fill);
            mbar_init(bb.kempty[s], 1);
        }
        for (int s = 0; s < L::RV; ++s) {
            mbar_init(bb.vfull[s], fill);
            mbar_init(bb.vempty[s], 1);
        }
        for (int s = 0; s < L::S8; ++s) {
            mbar_init(bb.k8full[s], 1);
            mbar_init(bb.v8full[s], 1);
            mbar_init(bb.k8empty[s], 4);
            mbar_init(bb.v8empty[s], 4);
        }
        for (int x = 0; x < 2; ++x) {
            mbar_init(bb.sfull[x], 1);
            mbar_init(bb.sfree[x], 128);
            mbar_init(bb.pfull[x], 128);
            mbar_init(bb.pvdone[x], 1);
        }
        mbar_init(bb.qfull, 128);
        mbar_init(bb.merged, 128);
        mbar_init(bb.flags, 2);   // all MMAs of both issuing threads completed (before tensor memory is freed)
        for (int k = 0; k < BAD_SLOTS; ++k) *pf_bad_slot(smem, L::OFF_CTRL, k) = 0;
        *abort_flag = 0;
        fence_mbar_init();
    }
    if (warp == 2) {   // this warp owns the tensor memory
        tmem_alloc(bb.tmem_slot, NW_TMEM_COLS);
        tmem_relinquish();
    }
    tc_fence_before_sync();
    __syncthreads();
    tc_fence_after_sync();
    const uint32_t tmem = *reinterpret_cast<volatile uint32_t *>(smem + (bb.tmem_slot - smem_u32(smem)));
    auto range = [&](int item) {
        const PfTile t = nw_item<MODE>(a, sp, item);
        return PfRange{t.seq, t.kvh, t.nkv, t.L, t.kv0};
    };
    if (warp == 2 || warp == 3) {
        if ((threadIdx.x & 31) == 0) {
            nw_mma<KV, MODE>(smem, a, sp, bb, tmem, abort_flag, total, warp == 3);
            // every MMA issued (by both threads) has completed before tensor
            // memory is released
            umma_commit(bb.flags);
            mbar_wait_bounded(bb.flags, 0, WAIT_LIMIT);
        }
        __syncwarp();
    } else if (warp >= NW_SOFT0 && warp < NW_SOFT0 + 4) {
        nw_softmax<KV, MODE>(smem, a, sp, bb, tmem, abort_flag, total);
    } else if (warp < 2) {
        if constexpr (L::F8) {   // the codes of K (warp 0) and V (warp 1) into their staging rings
            const int off[1] = {warp ? L::OFF_V8 : L::OFF_K8};
            const BarRing full[1] = {warp ? bb.v8full : bb.k8full};
            const BarRing empty[1] = {warp ? bb.v8empty : bb.k8empty};
            const CUtensorMap *maps[1] = {warp ? &tmv : &tmk};
            pf_stream<L::S8, true, 1>(smem, off, L::OFF_CTRL, full, empty, maps, a, abort_flag, total, range);
        } else {
            const int off[1] = {warp ? L::OFF_V : L::OFF_K};
            const BarRing full[1] = {warp ? bb.vfull : bb.kfull};
            const BarRing empty[1] = {warp ? bb.vempty : bb.kempty};
            const CUtensorMap *maps[1] = {warp ? &tmv : &tmk};
            if (warp)
                pf_stream<L::RV, false, 1>(smem, off, L::OFF_CTRL, full, empty, maps, a, abort_flag, total, range);
            else
                pf_stream<L::RK, false, 1>(smem, off, L::OFF_CTRL, full, empty, maps, a, abort_flag, total, range);
        }
    } else if constexpr (L::F8) {
        if (warp >= 8) {   // 8-11: K; 12-15: V; a quarter of the rows each
            const int kv = (warp - 8) >> 2;
            pf_convert_ring<L::RK, L::S8, 4>(smem + (kv ? L::OFF_V8 : L::OFF_K8), smem + (kv ? L::OFF_V : L::OFF_K),
                                            kv ? bb.v8full : bb.k8full, kv ? bb.v8empty : bb.k8empty,
                                            kv ? bb.vfull : bb.kfull, kv ? bb.vempty : bb.kempty, a, abort_flag,
                                            total, warp & 3, [&](int item) { return nw_item<MODE>(a, sp, item).nkv; });
        }
    }
    tc_fence_before_sync();
    __syncthreads();
    if (warp == 2) {
        tc_fence_after_sync();
        tmem_dealloc(tmem, NW_TMEM_COLS);
    }
}

// One-time set-up per cache type and mode: shared memory and grid (one CTA
// per SM, at most NW_MAX_CTAS: the merge scratch has that many slots).
struct NwSetup {
    int grid = 0;
    cudaError_t err = cudaSuccess;
};

template <int KV, int MODE>
const NwSetup &narrow_setup() {
    static NwSetup su;
    static std::once_flag once;
    std::call_once(once, [] {
        su.err = cudaFuncSetAttribute(narrow_kernel<KV, MODE>, cudaFuncAttributeMaxDynamicSharedMemorySize,
                                      NwL<KV>::SMEM);
        int dev = 0, sms = 0;
        if (su.err == cudaSuccess) su.err = cudaGetDevice(&dev);
        if (su.err == cudaSuccess) su.err = cudaDeviceGetAttribute(&sms, cudaDevAttrMultiProcessorCount, dev);
        su.grid = sms < NW_MAX_CTAS ? sms : NW_MAX_CTAS;
    });
    return su;
}

template <int KV, int MODE>
int launch_narrow_kv(const CUtensorMap &tmk, const CUtensorMap &tmv, const PrefillArgs &args, long long max_items,
                     cudaStream_t st) {
    const NwSetup &su = narrow_setup<KV, MODE>();
    if (su.err != cudaSuccess || su.grid <= 0) return PA_ERR_CUDA;
    if (!args.scratch) return PA_ERR_INVALID_ARG;
    const int g = (int)(max_items < su.grid ? (max_items > 0 ? max_items : 1) : su.grid);
    narrow_kernel<KV, MODE><<<g, NwL<KV>::THREADS, NwL<KV>::SMEM, st>>>(tmk, tmv, args);
    return cuda_status(cudaGetLastError());
}

}  // namespace

int launch_narrow(int kv, const CUtensorMap &tmk, const CUtensorMap &tmv, const PrefillArgs &args,
                  long long max_items, cudaStream_t st) {
    if (kv == PA_KV_BF16) return launch_narrow_kv<PA_KV_BF16, PF_CAUSAL>(tmk, tmv, args, max_items, st);
    if (kv == PA_KV_F16) return launch_narrow_kv<PA_KV_F16, PF_CAUSAL>(tmk, tmv, args, max_items, st);
    if (kv == PA_KV_FP8_E4M3) return launch_narrow_kv<PA_KV_FP8_E4M3, PF_CAUSAL>(tmk, tmv, args, max_items, st);
    return PA_ERR_UNSUPPORTED;
}

int launch_narrow_shared(const CUtensorMap &tmk, const CUtensorMap &tmv, const PrefillArgs &args,
                         long long max_items, cudaStream_t st) {
    return launch_narrow_kv<PA_KV_F16, PF_SHARED>(tmk, tmv, args, max_items, st);
}

int narrow_grid() { return narrow_setup<PA_KV_F16, PF_CAUSAL>().grid; }

bool narrow_usable(int kv) {
    if (kv == PA_KV_BF16) return narrow_setup<PA_KV_BF16, PF_CAUSAL>().err == cudaSuccess;
    if (kv == PA_KV_F16) return narrow_setup<PA_KV_F16, PF_CAUSAL>().err == cudaSuccess;
    if (kv == PA_KV_FP8_E4M3) return narrow_setup<PA_KV_FP8_E4M3, PF_CAUSAL>().err == cudaSuccess;
    return false;
}

}  // namespace pa
