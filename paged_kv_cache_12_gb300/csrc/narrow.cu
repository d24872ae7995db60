// Paged attention for work items of few query rows -- the new tokens of a
// speculative step, a few per sequence, or the members of a shared-prefix
// group over a range of their shared blocks -- on the 5th-generation tensor
// cores, with the KV tokens rather than the query rows on the MMAs' M side.
//
// What is computed is the one-tile kernel's (prefill.cu): each query row
// attends to the positions it sees through the block table (deepsonar page,
// section 2.5 for new tokens; section 2.3 for parallel samples sharing a
// prompt's blocks).  There an item of at most 32 rows (4 speculative tokens x
// 8 heads) fills a quarter of the 128-row tile, and the tensor work, the
// softmax and the tensor-memory traffic per KV tile are four times what its
// rows need.  Here both products are transposed:
//   S^T = K Q^T      M 128 tokens, N 32 rows, K 128 dims: A = the K tile as
//                    the TMA wrote it, B = Q^T (the rows, K-major);
//   O^T += V^T P^T   M 128 dims, N 32 rows, K 128 tokens: A = the V tile read
//                    MN-major, B = P^T (K-major, written by the softmax);
// S^T and O^T take 32 tensor-memory columns each, and one softmax thread holds
// one token's 32 scores.  A row's maximum then spans the 128 softmax threads:
// each warp reduces its 32 tokens with a transposed butterfly (lane i ends
// with row i), the four warps exchange their maxima through shared memory,
// and since every warp takes the maximum of the same four values, the running
// maximum and the decision to rescale (only when it grows by more than 2^8;
// O^T is then rescaled in tensor memory) are the same in all of them.  Row
// sums stay per thread until the item's end.
//
// One CTA per SM, persistent over the item list; warps:
//   0, 1   producers: K and V tiles of 128 tokens by TMA through the block
//          table (16-bit caches: one warp per cache, 3-stage rings); for an
//          FP8 cache the same warps stage the caches' codes (4 stages), so
//          that K's codes run ahead of V's conversion;
//   2, 3   MMA issuers (one thread each): warp 2 the S^T products, warp 3
//          the O^T += V^T P^T products, so neither waits for the other;
//   4-7    softmax: one token (S^T lane) per thread; in the epilogue one dim
//          (O^T lane) per thread;
//   8-15   FP8 only: the staged codes to fp16, K (8-11) into tensor memory
//          as the A operand of S^T, V (12-15) into a 2-stage shared-memory
//          ring (a register split gives the softmax warpgroup the most).
// P^T has two buffers in shared memory; S^T two buffers and O^T two
// accumulators (by item parity, so that an item's epilogue overlaps the next
// item's first products) in tensor memory.
// Every wait is bounded; warp-collective instructions (tensor-memory loads
// and stores, shuffles, votes) run in warp-uniform control flow, and the four
// softmax warps take every branch around them together; tensor memory is
// released on every path.

#include <cmath>
#include <mutex>

#include "prefill_common.cuh"

namespace pa {
namespace {

constexpr int NR = 32;                    // query rows of an item, padded: the MMAs' N
constexpr int NQ_BYTES = NR * PD * 2;     // Q^T: NR rows x 128 dims, 16-bit, 128-byte swizzled K-major
constexpr int NP_BYTES = NR * PN * 2;     // P^T: NR rows x PN tokens, the same layout
constexpr int NW_SOFT0 = 4;               // first softmax warp
// tensor memory: S^T 0, S^T 1, O^T 0, O^T 1 (NR columns each), and for an
// FP8 cache the two K tiles (128 tokens x 128 dims, two per column)
constexpr int NW_S = 0, NW_O = 2 * NR, NW_K = 4 * NR, NW_KT = PD / 2;
static_assert(PN == 128, "one softmax thread per token of a KV tile");
static_assert(NR == 32, "one row per lane in the transposed reductions");

#ifndef PA_NW_R16
#define PA_NW_R16 3
#endif
#ifndef PA_NW_R8
#define PA_NW_R8 2
#endif
#ifndef PA_NW_S8
#define PA_NW_S8 4
#endif
constexpr int NW_MAXST = 4;               // barrier slots per ring

// Shared memory per cache type.  16-bit caches: K and V rings of R stages
// that the TMA fills.  FP8 caches: staging rings of S8 stages for the codes
// of K and V, the V ring of R 16-bit tiles the converting warps fill, and no
// K ring: the K tiles are converted into tensor memory (two buffers), the A
// operand of S^T.
template <int KV>
struct NwL {
    static constexpr bool F8 = KV == PA_KV_FP8_E4M3;
    static constexpr int R = F8 ? PA_NW_R8 : PA_NW_R16;   // 16-bit ring stages
    static constexpr int S8 = F8 ? PA_NW_S8 : 0;          // FP8 staging stages
    static constexpr int KR = F8 ? 2 : R;                 // K tiles in flight (tensor-memory buffers for FP8)
    static constexpr int OFF_K = 0;
    static constexpr int OFF_V = F8 ? 0 : R * KV_BYTES;
    static constexpr int OFF_K8 = OFF_V + R * KV_BYTES;
    static constexpr int OFF_V8 = OFF_K8 + S8 * F8_BYTES;
    static constexpr int OFF_Q = OFF_V8 + S8 * F8_BYTES;
    static constexpr int OFF_P = OFF_Q + NQ_BYTES;              // two P^T buffers
    static constexpr int OFF_MAX = OFF_P + 2 * NP_BYTES;        // float [2][4][NR]: the warps' row maxima
    static constexpr int OFF_SUM = OFF_MAX + 2 * 4 * NR * 4;    // float [4][NR]: the warps' row sums
    static constexpr int OFF_VOTE = OFF_SUM + 4 * NR * 4;      // int [2][4]: the warps' votes
    static constexpr int OFF_CTRL = OFF_VOTE + 2 * 4 * 4;
    static constexpr int SMEM = OFF_CTRL + CTRL_BYTES + 1024;   // + alignment slack
    // 16-bit caches: warps 0 / 1 produce K / V, 2 / 3 issue the MMAs, 4-7 run
    // the softmax.  FP8 caches: warps 0 / 1 stage the codes, 2 / 3 issue the
    // MMAs, 4-7 run the softmax and 8-15 convert (four warps per cache, two
    // on every SM sub-partition), with a register split (SOFT_REGS for the
    // softmax warpgroup, OTHER_REGS for the others).
    static constexpr int THREADS = (F8 ? 16 : 8) * 32;
    static constexpr int SOFT_REGS = 200, OTHER_REGS = 104, LAUNCH_REGS = 128;   // FP8: 65536 / 512 at launch
    static_assert(!F8 || 128 * SOFT_REGS + (THREADS - 128) * OTHER_REGS <= THREADS * LAUNCH_REGS, "register split");
    static_assert(SMEM <= 227 * 1024, "shared memory of one CTA");
    static_assert(OFF_Q % 1024 == 0 && OFF_P % 1024 == 0 && NP_BYTES % 1024 == 0, "swizzled tiles 1024-byte aligned");
    static_assert(R <= NW_MAXST && S8 <= NW_MAXST && KR <= NW_MAXST, "ring stages");
    static constexpr int TMEM_COLS = F8 ? 256 : 128;
    static_assert(NW_O + 2 * NR <= NW_K && NW_K + (F8 ? 2 * NW_KT : 0) <= TMEM_COLS, "tensor-memory columns");
};

struct NwBars {
    // sfull / sfree: S^T buffers; pfull / pvdone: P^T buffers (by PV-number
    // parity); maxfull: the warps' row maxima of a KV tile (by tile parity)
    BarRing kfull, kempty, vfull, vempty, k8full, v8full, k8empty, v8empty;   // NW_MAXST each
    BarRing sfull, sfree, pfull, pvdone, maxfull;                             // 2 each
    uint32_t qfull, sumfull, tmem_slot, flags;                                // shared addresses
};
static_assert(8 * (8 * NW_MAXST + 10 + 4) <= CTRL_BAD, "control block layout");

__device__ __forceinline__ NwBars nw_bars(uint8_t *smem, int off_ctrl) {
    uint32_t a = smem_u32(smem + off_ctrl);
    NwBars b;
    BarRing *rings[8] = {&b.kfull, &b.kempty, &b.vfull, &b.vempty, &b.k8full, &b.v8full, &b.k8empty, &b.v8empty};
    for (int r = 0; r < 8; ++r) rings[r]->base = a, a += 8 * NW_MAXST;
    BarRing *pairs[5] = {&b.sfull, &b.sfree, &b.pfull, &b.pvdone, &b.maxfull};
    for (int r = 0; r < 5; ++r) pairs[r]->base = a, a += 16;
    b.qfull = a, a += 8;
    b.sumfull = a, a += 8;
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

// Transposed butterfly over a warp: v[r] is this lane's value of row r; lane
// i returns op over the warp's 32 lanes of row i.  v is overwritten.  At the
// step of distance k a lane keeps the half of its rows on its own side of bit
// k and sends the other half to the lane across it.
template <class Op>
__device__ __forceinline__ float warp_rows(float (&v)[NR], Op op) {
    const int lane = threadIdx.x & 31;
#pragma unroll
    for (int k = NR / 2; k >= 1; k >>= 1) {
        const bool up = (lane & k) != 0;
#pragma unroll
        for (int j = 0; j < k; ++j) {
            const float send = up ? v[j] : v[j + k];
            const float keep = up ? v[j + k] : v[j];
            v[j] = op(keep, __shfl_xor_sync(0xffffffffu, send, k));
        }
    }
    return v[0];
}

// ----------------------------------------------------------- MMA issuers
//
// One thread takes about 100 cycles to issue a tcgen05.mma whatever its N,
// while the tensor cores accept several such streams at once: the S^T products
// (warp 2) and the PV products (warp 3) are issued by two threads.  They share
// nothing but the barriers the softmax sits between: S^T reads K and Q^T and
// writes an S^T buffer, PV reads V and P^T and accumulates into O^T.

template <int KV, int MODE>
__device__ void nw_mma(uint8_t *smem, const PrefillArgs &a, const NwBars &bb, uint32_t tmem,
                       volatile int *abort_flag, int total, bool pv_role) {
    using L = NwL<KV>;
    constexpr int R = L::R;
    constexpr bool BF = KV == PA_KV_BF16;
    const uint32_t base = smem_u32(smem);
    // K-step k (16 elements) of a K-major tile with `rows` rows: byte 32 (k % 4)
    // of the 64-element block k / 4
    auto kstep = [](int k, int rows) { return (uint64_t)((((k >> 2) * (rows * 128)) + (k & 3) * 32) >> 4); };
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
        const uint32_t id_s = idesc_f16(128, NR, BF, false);   // A = K, B = Q^T, both K-major
        // K as A: 128-byte rows of 64 dims, one per token (M); the next 64 dims
        // PN rows further (FP8: one token per tensor-memory lane, two dims per
        // column).  Q^T as B: 128-byte rows of 64 dims, one per query row (N);
        // the next 64 NR rows further.
        const uint64_t dk0 = sw128_desc(base + L::OFF_K, 16, 1024);
        const uint64_t dq = sw128_desc(base + L::OFF_Q, 16, 1024);
        constexpr int KR = L::KR;
        int kc = 0, sc = 0;
        for (int item = blockIdx.x; item < total && ok; item += gridDim.x, ++it) {
            const PfTile t = pf_item<MODE>(a, item);
            if (!wait(bb.qfull, it & 1)) break;   // this item's Q^T is in shared memory
            for (int n = 0; n < t.nkv && ok; ++n) {   // S^T(n) into tensor-memory buffer sc & 1
                const int ks = kc % KR, b = sc & 1;
                if (!wait(bb.kfull[ks], (kc / KR) & 1)) break;
                if (sc >= 2 && !wait(bb.sfree[b], ((sc >> 1) - 1) & 1)) break;
                tc_fence_after_sync();
                if constexpr (L::F8) {
                    // K-step k: columns 8 k .. 8 k + 7 of the K tile in tensor memory
#pragma unroll
                    for (int k = 0; k < PD / 16; ++k)
                        umma_f16_ts(tmem + NW_S + b * NR, tmem + NW_K + ks * NW_KT + 8 * k, dq + kstep(k, NR), id_s,
                                    k > 0 ? 1u : 0u);
                } else {
                    const uint64_t dk = dk0 + (uint64_t)(ks * (KV_BYTES >> 4));
#pragma unroll
                    for (int k = 0; k < PD / 16; ++k)
                        umma_f16(tmem + NW_S + b * NR, dk + kstep(k, PN), dq + kstep(k, NR), id_s, k > 0 ? 1u : 0u);
                }
                umma_commit(bb.sfull[b]);
                umma_commit(bb.kempty[ks]);
                ++kc;
                ++sc;
            }
        }
    } else {
        const uint32_t id_o = idesc_f16_at(128, NR, BF, false);   // A = V^T (MN-major), B = P^T (K-major)
        // V^T as A with M (dims) contiguous: 128-byte rows of 64 dims, one per
        // token (K); the next 64 dims PN rows further.  P^T as B: 128-byte rows
        // of 64 tokens, one per query row (N); the next 64 NR rows further.
        const uint64_t dv0 = sw128_desc(base + L::OFF_V, PN * 128, 1024);
        const uint64_t dp0 = sw128_desc(base + L::OFF_P, 16, 1024);
        int vc = 0, pc = 0;
        for (int item = blockIdx.x; item < total && ok; item += gridDim.x, ++it) {
            const PfTile t = pf_item<MODE>(a, item);
            const uint32_t d_o = tmem + NW_O + (it & 1) * NR;
            for (int n = 0; n < t.nkv && ok; ++n) {
                const int pb = pc & 1;
                if (!wait(bb.pfull[pb], (pc >> 1) & 1)) break;
                ++pc;
                const int vs = vc % R;
                if (!wait(bb.vfull[vs], (vc / R) & 1)) break;
                tc_fence_after_sync();
                const uint64_t dv = dv0 + (uint64_t)(vs * (KV_BYTES >> 4));
                const uint64_t dp = dp0 + (uint64_t)(pb * (NP_BYTES >> 4));
#pragma unroll
                for (int k = 0; k < PN / 16; ++k)   // tokens 16 k .. 16 k + 15: V rows, P^T columns
                    umma_f16(d_o, dv + (uint64_t)((k * 16 * 128) >> 4), dp + kstep(k, NR), id_o,
                             (n > 0 || k > 0) ? 1u : 0u);
                umma_commit(bb.pvdone[pb]);
                umma_commit(bb.vempty[vs]);
                ++vc;
            }
        }
    }
}

// --------------------------------------------- FP8: K codes to tensor memory

// The K tile of an FP8 cache, converted into tensor memory by warps 8-11: the
// thread of lane l of warp 8 + q takes token 32 q + l (its tensor-memory
// lane), reads the token's 128 codes from the staging ring and stores them as
// 64 fp16 pairs, dims 2 c and 2 c + 1 in column c of K buffer `conv % 2` --
// the A operand layout of S^T.  Every E4M3 value is an fp16 value; the K scale
// is folded into the softmax scale.
template <int MODE>
__device__ void nw_convert_k(uint8_t *smem, const PrefillArgs &a, const NwBars &bb, uint32_t tmem,
                             volatile int *abort_flag, int total) {
    using L = NwL<PA_KV_FP8_E4M3>;
    constexpr int S8 = L::S8, KR = L::KR;
    const int lane = threadIdx.x & 31;
    const int quarter = (threadIdx.x >> 5) & 3;
    const int tok = quarter * 32 + lane;
    const uint32_t trow = tmem + ((uint32_t)(quarter * 32) << 16) + NW_K;
    int conv = 0;
    for (int item = blockIdx.x; item < total; item += gridDim.x) {
        const int nkv = pf_item<MODE>(a, item).nkv;
        for (int n = 0; n < nkv; ++n, ++conv) {
            const int s8 = conv % S8, c = conv % KR;
            const bool got = !*abort_flag &&
                             mbar_wait_bounded(bb.k8full[s8], (uint32_t)((conv / S8) & 1), a.wait_limit) &&
                             mbar_wait_bounded(bb.kempty[c], (uint32_t)(((conv / KR) & 1) ^ 1), a.wait_limit);
            if (!__all_sync(0xffffffffu, got)) {
                if (lane == 0) pf_error(a);
                *abort_flag = 1;
                return;   // the staging warp drains its own copies
            }
            tc_fence_after_sync();
            // the token's row of codes: 16-byte chunk j (dims 16 j ..) at chunk j ^ (tok % 8)
            const uint8_t *row = smem + L::OFF_K8 + s8 * F8_BYTES + tok * 128;
#pragma unroll
            for (int h = 0; h < 2; ++h) {   // dims 64 h .. 64 h + 63: columns 32 h .. 32 h + 31
                uint32_t w[32];
#pragma unroll
                for (int j = 0; j < 4; ++j) {
                    const uint4 x = *reinterpret_cast<const uint4 *>(row + (((4 * h + j) ^ (tok & 7)) << 4));
                    w[8 * j + 0] = e4m3x2_lo_to_f16x2(x.x);
                    w[8 * j + 1] = e4m3x2_hi_to_f16x2(x.x);
                    w[8 * j + 2] = e4m3x2_lo_to_f16x2(x.y);
                    w[8 * j + 3] = e4m3x2_hi_to_f16x2(x.y);
                    w[8 * j + 4] = e4m3x2_lo_to_f16x2(x.z);
                    w[8 * j + 5] = e4m3x2_hi_to_f16x2(x.z);
                    w[8 * j + 6] = e4m3x2_lo_to_f16x2(x.w);
                    w[8 * j + 7] = e4m3x2_hi_to_f16x2(x.w);
                }
                tmem_st32(trow + c * NW_KT + 32 * h, w);
            }
            tmem_wait_st();
            tc_fence_before_sync();
            mbar_arrive(bb.kfull[c]);
            mbar_arrive(bb.k8empty[s8]);
        }
    }
}

// ------------------------------------------------------------- softmax

template <int KV, int MODE>
__device__ void nw_softmax(uint8_t *smem, const PrefillArgs &a, const NwBars &bb, uint32_t tmem,
                           volatile int *abort_flag, int total) {
    using L = NwL<KV>;
    constexpr int R = L::R;
    const int lane = threadIdx.x & 31;
    const int quarter = (threadIdx.x >> 5) & 3;   // tensor-memory lanes 32 quarter .. + 31
    const int tl = quarter * 32 + lane;           // token of a KV tile (S^T lane); dim (O^T lane)
    const uint32_t trow = tmem + ((uint32_t)(quarter * 32) << 16);
    const float sl2 = a.scale_log2;
    float *wmax = reinterpret_cast<float *>(smem + L::OFF_MAX);
    float *wsum = reinterpret_cast<float *>(smem + L::OFF_SUM);
    int *votes = reinterpret_cast<int *>(smem + L::OFF_VOTE);
    uint8_t *qt = smem + L::OFF_Q;
    // this thread's column of P^T: its token's 64-token block, 16-byte chunk
    // (before the swizzle) and place in the chunk
    const int ptok = (quarter & 1) * 32 + lane;
    uint8_t *pcol = smem + L::OFF_P + (quarter >> 1) * (NR * 128) + (ptok & 7) * 2;
    const int pchunk = ptok >> 3;
    int sc = 0, g = 0, vcount = 0, xp = 0, xr = 0, it = 0;
    bool ok = true;
    // every thread of a warp takes the same decision, and the four warps see
    // the same barriers, so warp-collective instructions are never reached by
    // part of a warp
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
    // rows r = tl / 16 + 8 j (j < 4) of an item, 16-byte chunk tl % 16 each:
    // global address (zeros past the item's rows) and swizzled place in Q^T
    const int qc = tl & 15;
    auto q_src = [&](const PfTile &tq, int r) -> const uint4 * {
        const int tok = r / a.G, hh = r - tok * a.G;
        if (tok >= tq.ntok) return nullptr;
        return reinterpret_cast<const uint4 *>(a.query +
                                               ((long long)(tq.q0 + tq.row0 + tok) * a.Hq + tq.kvh * a.G + hh) * PD) +
               qc;
    };
    auto store_q = [&](const PfTile &tq) {
#pragma unroll
        for (int j = 0; j < 4; ++j) {
            const int r = (tl >> 4) + 8 * j;
            const uint4 *src = q_src(tq, r);
            const uint4 x = src ? __ldg(src) : make_uint4(0, 0, 0, 0);
            *reinterpret_cast<uint4 *>(qt + (qc >> 3) * (NR * 128) + r * 128 + (((qc & 7) ^ (r & 7)) << 4)) = x;
        }
        fence_proxy_async_smem();   // for the tensor cores
        mbar_arrive(bb.qfull);
    };
    if ((int)blockIdx.x < total) store_q(pf_item<MODE>(a, blockIdx.x));
    for (int item = blockIdx.x; item < total && ok; item += gridDim.x, ++it) {
        const PfTile t = pf_item<MODE>(a, item);
        const bool has_next = item + (int)gridDim.x < total;
        const PfTile tn = pf_item<MODE>(a, has_next ? item + (int)gridDim.x : item);
        if (has_next) {
#pragma unroll
            for (int j = 0; j < 4; ++j)
                if (const uint4 *src = q_src(tn, (tl >> 4) + 8 * j)) prefetch_l2(src);
        }
        // positions the item's first row sees: a tile past them needs the mask
        const int vis0 = MODE == PF_SHARED ? t.L : t.C + t.row0;
        const uint32_t t_o = trow + NW_O + (it & 1) * NR;
        float mr[NR], lp[NR];   // running maximum of every row (log2 units; the same in every thread), row sums
#pragma unroll
        for (int r = 0; r < NR; ++r) mr[r] = -INFINITY, lp[r] = 0.f;
        float mrow = -INFINITY;   // the running maximum of row `lane`
        // ---- the exchanges of the four softmax warps (maxfull, by parity):
        // xp of them published so far, xr resolved (waited for and read)
        auto publish_vote = [&](bool up) {
            int *vslot = votes + (xp & 1) * 4;
            const bool wup = __any_sync(0xffffffffu, up);
            if (lane == 0) vslot[quarter] = wup ? 1 : 0;
            mbar_arrive(bb.maxfull[xp & 1]);
            ++xp;
        };
        auto resolve_vote = [&](bool &up) {
            if (!wait(bb.maxfull[xr & 1], (xr >> 1) & 1)) return false;
            const int *vslot = votes + (xr & 1) * 4;
            up = (vslot[0] | vslot[1] | vslot[2] | vslot[3]) != 0;
            ++xr;
            return true;
        };
        // ---- S^T(n): this thread's token's score for every row, masked
        // where the row does not see the token; then the thread's vote:
        // does any of them stand more than 2^8 above its row's running
        // maximum?  (A row's maximum grows by more than 2^8 exactly when one
        // of its scores does: the scale is positive.)
        auto load_tile = [&](int n, float (&x)[NR]) {
            const int b = sc & 1;
            if (!wait(bb.sfull[b], (sc >> 1) & 1)) return false;
            ++sc;
            tc_fence_after_sync();
            {
                uint32_t r[32];
                tmem_ld32(trow + NW_S + b * NR, r);
                tmem_wait_ld();
#pragma unroll
                for (int c = 0; c < NR; ++c) x[c] = __uint_as_float(r[c]);
            }
            tc_fence_before_sync();
            mbar_arrive(bb.sfree[b]);
            // the item's last S^T is done, and with it every product that read
            // Q^T: the next item's rows go in now
            if (n + 1 == t.nkv && has_next) store_q(tn);
            const int t0 = n * PN;
            if (t0 + PN > vis0) {
                // row r = G tok + h sees positions < vis0 + tok (causal), or the
                // whole range (shared); rows below rmin do not see this token
                const int pos = t0 + tl;
                int rmin = 0;
                if (pos >= t.L)
                    rmin = NR;
                else if (MODE == PF_CAUSAL && pos >= vis0)
                    rmin = (pos - vis0 + 1) * a.G;
#pragma unroll
                for (int r = 0; r < NR; ++r) x[r] = r >= rmin ? x[r] : -INFINITY;
            }
            bool up = false;
#pragma unroll
            for (int r = 0; r < NR; ++r) up |= x[r] * sl2 > mr[r] + RESCALE_THRESHOLD;
            publish_vote(up);
            return true;
        };
        // The vote on tile n + 1 is published before tile n's P is computed,
        // so that the exchange's round trip overlaps that work; it compares
        // with the running maxima after tile n's rescale, if there was one.
        float s[NR];
        if (!load_tile(0, s)) break;
        for (int n = 0; n < t.nkv && ok; ++n) {
            // ---- Rescale only when some row's maximum grows by more than 2^8:
            // when the vote says so (an item's first tile, and rarely later)
            // the rows' maxima are reduced -- over this warp's tokens, then
            // over the four warps' -- and the growing rows rescaled.  Every
            // warp sees the same votes and compares the same numbers, so the
            // branches are the same in all four; rows that do not grow scale by
            // exactly 1.
            bool up;
            if (!resolve_vote(up)) break;
            if (up) {
                float m;
                {
                    float v[NR];
#pragma unroll
                    for (int r = 0; r < NR; ++r) v[r] = s[r];
                    m = warp_rows(v, [](float x, float y) { return fmaxf(x, y); });
                }
                float *slot = wmax + (xp & 1) * (4 * NR);
                slot[quarter * NR + lane] = m;
                mbar_arrive(bb.maxfull[xp & 1]);
                ++xp;
                if (!wait(bb.maxfull[xr & 1], (xr >> 1) & 1)) break;
                ++xr;
                const float mt =
                    fmaxf(fmaxf(slot[lane], slot[NR + lane]), fmaxf(slot[2 * NR + lane], slot[3 * NR + lane])) * sl2;
                const bool grow = mt > mrow + RESCALE_THRESHOLD;
                const float nm = grow ? mt : mrow;
                const float al = grow ? fast_exp2(mrow - nm) : 1.f;
                mrow = nm;
                if (n > 0) {   // O^T holds the products up to PV number g - 1: scale its row columns
                    if (!wait(bb.pvdone[(g - 1) & 1], ((g - 1) >> 1) & 1)) break;
                    tc_fence_after_sync();
                    uint32_t o[32];
                    tmem_ld32(t_o, o);
                    tmem_wait_ld();
#pragma unroll
                    for (int r = 0; r < NR; ++r) {
                        const float ar = __shfl_sync(0xffffffffu, al, r);
                        mr[r] = __shfl_sync(0xffffffffu, mrow, r);
                        lp[r] *= ar;
                        o[r] = __float_as_uint(__uint_as_float(o[r]) * ar);
                    }
                    tmem_st32(t_o, o);
                    tmem_wait_st();
                } else {
#pragma unroll
                    for (int r = 0; r < NR; ++r) mr[r] = __shfl_sync(0xffffffffu, mrow, r);
                }
            }
            // ---- the next tile's scores and vote
            float sn[NR];
            if (n + 1 < t.nkv && !load_tile(n + 1, sn)) break;
            // ---- the last KV tile: V rows past the range are zeroed (P is 0
            // there, but the rows hold stale bits)
            const int t0 = n * PN;
            const int vs = vcount % R;
            const int vphase = (vcount / R) & 1;
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
            // ---- p = 2^(s scale log2(e) - m) into this thread's column of
            // P^T buffer g & 1 (PV number g - 2 read it before): two bytes per
            // row; a warp's 32 tokens fill 64 bytes of a row, no bank conflict
            if (g >= 2 && !wait(bb.pvdone[g & 1], ((g - 2) >> 1) & 1)) break;
            uint8_t *pbuf = pcol + (g & 1) * NP_BYTES;
#pragma unroll
            for (int r = 0; r < NR; ++r) {
                const float p = fast_exp2(fmaf(s[r], sl2, -mr[r]));
                lp[r] += p;
                *reinterpret_cast<uint16_t *>(pbuf + r * 128 + ((pchunk ^ (r & 7)) << 4)) = out_bits<KV>(p);
            }
            fence_proxy_async_smem();   // P^T and the zeroed V rows, for the tensor cores
            tc_fence_before_sync();
            mbar_arrive(bb.pfull[g & 1]);
            ++g;
#pragma unroll
            for (int r = 0; r < NR; ++r) s[r] = sn[r];
        }
        if (!ok) break;
        // ---- epilogue once the item's last PV (number g - 1) is done
        if (!wait(bb.pvdone[(g - 1) & 1], ((g - 1) >> 1) & 1)) break;
        tc_fence_after_sync();
        float l = warp_rows(lp, [](float x, float y) { return x + y; });   // row `lane`, this warp's tokens
        wsum[quarter * NR + lane] = l;
        mbar_arrive(bb.sumfull);
        if (!wait(bb.sumfull, it & 1)) break;
        l = (wsum[lane] + wsum[NR + lane]) + (wsum[2 * NR + lane] + wsum[3 * NR + lane]);
        const bool bad = *pf_bad_slot(smem, L::OFF_CTRL, pf_local(item)) == pf_local(item) + 1;
        const float qnan = __int_as_float(0x7fc00000);
        uint32_t o[32];
        tmem_ld32(t_o, o);
        tmem_wait_ld();
        tc_fence_before_sync();
        if constexpr (MODE == PF_SHARED) {
            // each member's partial row of this shared range: unnormalised O
            // (times the V scale) and (m, l) -- the decode kernel's partial
            // format -- at row part_off[member] + the range's partition index
            int tok = 0, hh = 0;
#pragma unroll
            for (int r = 0; r < NR; ++r) {
                if (tok < t.ntok) {
                    const long long wrow =
                        ((long long)a.part_off[t.q0 + tok] + t.kv0 / a.pt) * a.Hq + t.kvh * a.G + hh;
                    a.ws_o[wrow * PD + tl] = bad ? qnan : __uint_as_float(o[r]) * a.v_scale;
                    if (quarter == 0 && lane == r) a.ws_ml[wrow] = bad ? make_float2(qnan, qnan) : make_float2(mrow, l);
                }
                if (++hh == a.G) hh = 0, ++tok;
            }
        } else {
            const float inv = bad ? qnan : a.v_scale / l;   // of row `lane`
            int tok = 0, hh = 0;
#pragma unroll
            for (int r = 0; r < NR; ++r) {
                const float iv = __shfl_sync(0xffffffffu, inv, r);
                if (tok < t.ntok)
                    a.out[((long long)(t.q0 + t.row0 + tok) * a.Hq + t.kvh * a.G + hh) * PD + tl] =
                        out_bits<KV>(__uint_as_float(o[r]) * iv);
                if (++hh == a.G) hh = 0, ++tok;
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
    if (threadIdx.x == 0) {
        // FP8: the 128 threads converting K arrive on kfull and k8empty, the
        // four warps converting V (one lane each) on vfull and v8empty
        for (int s = 0; s < L::KR; ++s) {
            mbar_init(bb.kfull[s], L::F8 ? 128 : 1);
            mbar_init(bb.kempty[s], 1);
        }
        for (int s = 0; s < L::R; ++s) {
            mbar_init(bb.vfull[s], L::F8 ? 4 : 1);
            mbar_init(bb.vempty[s], 1);
        }
        for (int s = 0; s < L::S8; ++s) {
            mbar_init(bb.k8full[s], 1);
            mbar_init(bb.v8full[s], 1);
            mbar_init(bb.k8empty[s], 128);
            mbar_init(bb.v8empty[s], 4);
        }
        for (int x = 0; x < 2; ++x) {
            mbar_init(bb.sfull[x], 1);
            mbar_init(bb.sfree[x], 128);
            mbar_init(bb.pfull[x], 128);
            mbar_init(bb.pvdone[x], 1);
            mbar_init(bb.maxfull[x], 128);
        }
        mbar_init(bb.qfull, 128);
        mbar_init(bb.sumfull, 128);
        mbar_init(bb.flags, 2);   // all MMAs of both issuing threads completed (before tensor memory is freed)
        for (int k = 0; k < BAD_SLOTS; ++k) *pf_bad_slot(smem, L::OFF_CTRL, k) = 0;
        *abort_flag = 0;
        fence_mbar_init();
    }
    if (warp == 2) {   // this warp owns the tensor memory
        tmem_alloc(bb.tmem_slot, L::TMEM_COLS);
        tmem_relinquish();
    }
    tc_fence_before_sync();
    __syncthreads();
    tc_fence_after_sync();
    const uint32_t tmem = *reinterpret_cast<volatile uint32_t *>(smem + (bb.tmem_slot - smem_u32(smem)));
    auto range = [&](int item) {
        const PfTile t = pf_item<MODE>(a, item);
        return PfRange{t.seq, t.kvh, t.nkv, t.L, t.kv0};
    };
    auto mma = [&]() {
        if ((threadIdx.x & 31) == 0) {
            nw_mma<KV, MODE>(smem, a, bb, tmem, abort_flag, total, warp == 3);
            // every MMA issued (by both threads) has completed before tensor
            // memory is released
            umma_commit(bb.flags);
            mbar_wait_bounded(bb.flags, 0, WAIT_LIMIT);
        }
        __syncwarp();
    };
    if constexpr (L::F8) {
        // register split: the softmax warpgroup (warps 4-7) gets SOFT_REGS
        // registers, the others OTHER_REGS (the host checks the launch count)
        if (warp >= NW_SOFT0 && warp < NW_SOFT0 + 4) {
            regs_increase<L::SOFT_REGS>();
            nw_softmax<KV, MODE>(smem, a, bb, tmem, abort_flag, total);
        } else {
            regs_decrease<L::OTHER_REGS>();
            if (warp == 2 || warp == 3) {
                mma();
            } else if (warp < 2) {   // the codes of K (warp 0) and V (warp 1) into their staging rings
                const int off[1] = {warp ? L::OFF_V8 : L::OFF_K8};
                const BarRing full[1] = {warp ? bb.v8full : bb.k8full};
                const BarRing empty[1] = {warp ? bb.v8empty : bb.k8empty};
                const CUtensorMap *maps[1] = {warp ? &tmv : &tmk};
                pf_stream<L::S8, true, 1>(smem, off, L::OFF_CTRL, full, empty, maps, a, abort_flag, total, range);
            } else if (warp >= 12) {   // V: a quarter of the rows each, into the 16-bit ring
                pf_convert_ring<L::R, L::S8, 4>(smem + L::OFF_V8, smem + L::OFF_V, bb.v8full, bb.v8empty, bb.vfull,
                                                bb.vempty, a, abort_flag, total, warp & 3,
                                                [&](int item) { return pf_item<MODE>(a, item).nkv; });
            } else if (warp >= 8) {    // K: a token per thread, into tensor memory
                nw_convert_k<MODE>(smem, a, bb, tmem, abort_flag, total);
            }
        }
    } else {
        if (warp == 2 || warp == 3) {
            mma();
        } else if (warp >= NW_SOFT0 && warp < NW_SOFT0 + 4) {
            nw_softmax<KV, MODE>(smem, a, bb, tmem, abort_flag, total);
        } else if (warp < 2) {
            const int off[1] = {warp ? L::OFF_V : L::OFF_K};
            const BarRing full[1] = {warp ? bb.vfull : bb.kfull};
            const BarRing empty[1] = {warp ? bb.vempty : bb.kempty};
            const CUtensorMap *maps[1] = {warp ? &tmv : &tmk};
            pf_stream<L::R, false, 1>(smem, off, L::OFF_CTRL, full, empty, maps, a, abort_flag, total, range);
        }
    }
    tc_fence_before_sync();
    __syncthreads();
    if (warp == 2) {
        tc_fence_after_sync();
        tmem_dealloc(tmem, L::TMEM_COLS);
    }
}

// One-time set-up per cache type and mode: shared memory and grid (one CTA
// per SM).
struct NwSetup {
    int grid = 0;
    bool usable = false;
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
        cudaFuncAttributes fa;
        if (su.err == cudaSuccess) su.err = cudaGetDevice(&dev);
        if (su.err == cudaSuccess) su.err = cudaDeviceGetAttribute(&sms, cudaDevAttrMultiProcessorCount, dev);
        if (su.err == cudaSuccess) su.err = cudaFuncGetAttributes(&fa, narrow_kernel<KV, MODE>);
        su.grid = sms;
        // the FP8 kernel's register split assumes LAUNCH_REGS registers per
        // thread at launch; with another count a warpgroup's increase could
        // wait forever, so the kernel is then never launched
        su.usable = su.err == cudaSuccess && sms > 0 && (!NwL<KV>::F8 || fa.numRegs == NwL<KV>::LAUNCH_REGS);
    });
    return su;
}

template <int KV, int MODE>
int launch_narrow_kv(const CUtensorMap &tmk, const CUtensorMap &tmv, const PrefillArgs &args, long long max_items,
                     cudaStream_t st) {
    const NwSetup &su = narrow_setup<KV, MODE>();
    if (su.err != cudaSuccess) return PA_ERR_CUDA;
    if (!su.usable) return PA_ERR_UNSUPPORTED;
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

bool narrow_usable(int kv) {
    if (kv == PA_KV_BF16) return narrow_setup<PA_KV_BF16, PF_CAUSAL>().usable;
    if (kv == PA_KV_F16) return narrow_setup<PA_KV_F16, PF_CAUSAL>().usable;
    if (kv == PA_KV_FP8_E4M3) return narrow_setup<PA_KV_FP8_E4M3, PF_CAUSAL>().usable;
    return false;
}

}  // namespace pa
