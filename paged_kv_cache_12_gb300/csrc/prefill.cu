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

#include "decode_common.cuh"
#include "prefill.h"
#include "umma.cuh"

namespace pa {
namespace {

constexpr int PM = 128;                    // query rows per work tile
#ifndef PA_PF_PN
#define PA_PF_PN 128
#endif
#ifndef PA_PF_STAGES
#define PA_PF_STAGES 3
#endif
constexpr int PN = PA_PF_PN;               // KV tokens per tile (64 or 128)
constexpr int PD = 128;                    // head dim
constexpr int PST = PA_PF_STAGES;          // K and V ring stages of a 16-bit cache
constexpr int KV_BYTES = PN * PD * 2;      // a 16-bit K or V tile: 2 blocks (64 dims) x PN tokens x 128 B
constexpr int F8_BYTES = PN * PD;          // an FP8 tile: PN tokens x 128 B
constexpr int MAXST = 3;                   // barrier slots per ring
constexpr int CTRL_BYTES = 512;
constexpr int BAD_SLOTS = 16;              // out-of-range marks, one per work item of this CTA modulo 16
constexpr int CTRL_BAD = 416;              // int[BAD_SLOTS]: 1 + the CTA-local index of an item that met an
                                           // out-of-range block id (producers run at most a few KV tiles,
                                           // hence items, ahead of the softmax that reads the mark)
constexpr int CTRL_ABORT = CTRL_BAD + 4 * BAD_SLOTS;   // int: a role gave up waiting
constexpr int PF_THREADS = 7 * 32;         // K producer, V producer, MMA, 4 softmax warps

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
static_assert(8 * (6 * MAXST + 11) + 8 <= CTRL_BAD && CTRL_ABORT + 4 <= CTRL_BYTES, "control block layout");

struct PfBars {
    // pfull / pvdone: one per PV-number parity, so that a softmax warp a step
    // ahead of another never adds its arrival to the other step's phase
    // k8full / v8full: FP8 codes staged (TMA bytes landed)
    uint32_t kfull[MAXST], kempty[MAXST], vfull[MAXST], vempty[MAXST], k8full[MAXST], v8full[MAXST];
    uint32_t sfull[2], sfree[2], pfull[2], pvdone[2], qfull;
    uint32_t tmem_slot, flags;   // shared addresses
};

__device__ __forceinline__ PfBars pf_bars(uint8_t *smem, int off_ctrl) {
    const uint32_t c = smem_u32(smem + off_ctrl);
    PfBars b;
    uint32_t a = c;
    for (int s = 0; s < MAXST; ++s) b.kfull[s] = a, a += 8;
    for (int s = 0; s < MAXST; ++s) b.kempty[s] = a, a += 8;
    for (int s = 0; s < MAXST; ++s) b.vfull[s] = a, a += 8;
    for (int s = 0; s < MAXST; ++s) b.vempty[s] = a, a += 8;
    for (int s = 0; s < MAXST; ++s) b.k8full[s] = a, a += 8;
    for (int s = 0; s < MAXST; ++s) b.v8full[s] = a, a += 8;
    b.sfull[0] = a, a += 8;
    b.sfull[1] = a, a += 8;
    b.sfree[0] = a, a += 8;
    b.sfree[1] = a, a += 8;
    b.pfull[0] = a, a += 8;
    b.pfull[1] = a, a += 8;
    b.pvdone[0] = a, a += 8;
    b.pvdone[1] = a, a += 8;
    b.qfull = a, a += 8;
    b.tmem_slot = a, a += 8;
    b.flags = a;   // barriers and slots end at byte 8 (6 MAXST + 11) + 8 = 240 <= CTRL_BAD
    return b;
}

// Geometry of one work tile, the same in every warp.
struct PfTile {
    int seq, kvh, row0, ntok, C, nkv, L, q0;
};

__device__ __forceinline__ PfTile pf_tile(const PrefillArgs &a, int item) {
    const int4 rec = a.tiles[item / a.Hkv];
    PfTile t;
    t.seq = rec.x;
    t.kvh = item % a.Hkv;
    const int tpt = PM / a.G;               // new tokens per tile
    t.L = a.context_lens[t.seq];
    t.q0 = a.query_start[t.seq];
    const int T = a.query_start[t.seq + 1] - t.q0;
    t.row0 = rec.y * tpt;                   // first new token of the tile
    t.ntok = min(tpt, T - t.row0);
    t.C = t.L - T + 1;                      // positions the first new token sees
    t.nkv = (t.C + t.row0 + t.ntok - 1 + PN - 1) / PN;
    return t;
}

__device__ __forceinline__ void pf_error(const PrefillArgs &a) { atomicExch(&a.hdr->error, PA_ERR_TIMEOUT); }

// The CTA-local index of a work item (items are dealt round-robin) and its
// out-of-range mark in the control block.
__device__ __forceinline__ int pf_local(int item) { return (item - (int)blockIdx.x) / (int)gridDim.x; }
__device__ __forceinline__ volatile int *pf_bad_slot(uint8_t *smem, int off_ctrl, int local) {
    return reinterpret_cast<volatile int *>(smem + off_ctrl + CTRL_BAD) + (local % BAD_SLOTS);
}

// ----------------------------------------------------------- producer

template <int KV>
__device__ void pf_producer(uint8_t *smem, const CUtensorMap *map, const PrefillArgs &a, const PfBars &bb,
                            volatile int *abort_flag, int total, int kv) {
    using L = PfL<KV>;
    constexpr int PST = L::R;
    const int lane = threadIdx.x & 31;
    const uint64_t pol = policy_evict_normal();
    const int box_rows = a.bs < 16 ? a.bs : 16;    // rows per TMA box: one box per block or 16-row group
    const uint32_t base = smem_u32(smem) + (kv ? L::OFF_V : L::OFF_K);
    const uint32_t *full = kv ? bb.vfull : bb.kfull;
    const uint32_t *empty = kv ? bb.vempty : bb.kempty;
    int cnt = 0;
    // Before leaving, the last copy into every stage has landed (bounded).
    auto drain = [&]() {
        for (int s = 0; s < PST; ++s)
            if (cnt > s) mbar_wait_bounded(full[s], (uint32_t)(((s + (cnt - 1 - s) / PST * PST) / PST) & 1), WAIT_LIMIT);
    };
    for (int item = blockIdx.x; item < total; item += gridDim.x) {
        const PfTile t = pf_tile(a, item);
        const int32_t *row = a.block_tables + (long long)t.seq * a.mbps;
        for (int n = 0; n < t.nkv; ++n) {
            // lane j owns box j of the tile (tokens t0 + j box_rows ..): its block id,
            // loaded before the wait so that the load's latency overlaps it
            const int t0 = n * PN;
            const int tok = t0 + lane * box_rows;
            const bool mine = lane < PN / box_rows && tok < t.L;
            const int32_t blk = mine ? __ldg(row + tok / a.bs) : 0;
            const int s = cnt % PST;
            // the warp decides together (no lane may leave alone)
            const bool got = !*abort_flag && mbar_wait_bounded(empty[s], ((cnt / PST) & 1) ^ 1, a.wait_limit);
            if (!__all_sync(0xffffffffu, got)) {
                if (lane == 0) pf_error(a);
                *abort_flag = 1;
                drain();
                return;
            }
            const unsigned boxes = __ballot_sync(0xffffffffu, mine);
            const bool bad = __any_sync(0xffffffffu, mine && (blk < 0 || blk >= a.num_blocks));
            if (lane == 0) {
                if (bad) *pf_bad_slot(smem, L::OFF_CTRL, pf_local(item)) = pf_local(item) + 1;
                mbar_arrive_expect_tx(full[s], bad ? 0u : (uint32_t)(__popc(boxes) * 2 * box_rows * 128));
            }
            __syncwarp();
            if (!bad && mine) {
                const uint32_t dst = base + s * KV_BYTES + lane * box_rows * 128;
                const int y = (int)(((long long)blk * a.Hkv + t.kvh) * a.bs) + tok % a.bs;
                tma_load_2d(dst, map, 0, y, full[s], pol);
                tma_load_2d(dst + PN * 128, map, 64, y, full[s], pol);
            }
            __syncwarp();
            ++cnt;
        }
    }
    drain();
}

// FP8 cache: the same work, through a staging ring.  The warp issues the TMA
// copies of the codes of up to S8 KV tiles ahead (one 128-byte box column per
// block); behind them it turns each staged tile into the 16-bit tile the MMAs
// read, in the same swizzled layout a 16-bit TMA copy would have written:
// code chunk j (dims 16 j .. 16 j + 15) of row r becomes fp16 chunks 2 (j % 4)
// and 2 (j % 4) + 1 of the 64-dim block j / 4.  Every E4M3 value is an fp16
// value, so the tile is exact; the scales are applied to the scores and the
// output.  A staging slot is refilled only after this warp converted it.
__device__ void pf_producer_fp8(uint8_t *smem, const CUtensorMap *map, const PrefillArgs &a, const PfBars &bb,
                                volatile int *abort_flag, int total, int kv) {
    using L = PfL<PA_KV_FP8_E4M3>;
    constexpr int R = L::R, S8 = L::S8;
    const int lane = threadIdx.x & 31;
    const uint64_t pol = policy_evict_normal();
    const int box_rows = a.bs < 16 ? a.bs : 16;
    const uint32_t stage = smem_u32(smem) + (kv ? L::OFF_V8 : L::OFF_K8);
    const uint8_t *stage_p = smem + (kv ? L::OFF_V8 : L::OFF_K8);
    uint8_t *ring = smem + (kv ? L::OFF_V : L::OFF_K);
    const uint32_t *full8 = kv ? bb.v8full : bb.k8full;
    const uint32_t *full = kv ? bb.vfull : bb.kfull;
    const uint32_t *empty = kv ? bb.vempty : bb.kempty;
    // issue and conversion walk the same sequence of (work item, KV tile)
    struct Walk {
        int item, n;
        PfTile t;
    };
    auto start = [&](Walk &w) {
        w.item = blockIdx.x;
        w.n = 0;
        if (w.item < total) w.t = pf_tile(a, w.item);
    };
    auto step = [&](Walk &w) {
        if (++w.n < w.t.nkv) return;
        w.n = 0;
        w.item += gridDim.x;
        if (w.item < total) w.t = pf_tile(a, w.item);
    };
    Walk wi, wc;
    start(wi);
    start(wc);
    int issued = 0, conv = 0;
    bool ok = true;
    auto fail = [&]() {
        if (lane == 0) pf_error(a);
        *abort_flag = 1;
        ok = false;
    };
    auto issue = [&]() {
        const int s8 = issued % S8;
        const int t0 = wi.n * PN;
        const int tok = t0 + lane * box_rows;
        const bool mine = lane < PN / box_rows && tok < wi.t.L;
        const int32_t blk = mine ? __ldg(a.block_tables + (long long)wi.t.seq * a.mbps + tok / a.bs) : 0;
        const unsigned boxes = __ballot_sync(0xffffffffu, mine);
        const bool bad = __any_sync(0xffffffffu, mine && (blk < 0 || blk >= a.num_blocks));
        if (lane == 0) {
            if (bad) *pf_bad_slot(smem, L::OFF_CTRL, pf_local(wi.item)) = pf_local(wi.item) + 1;
            mbar_arrive_expect_tx(full8[s8], bad ? 0u : (uint32_t)(__popc(boxes) * box_rows * 128));
        }
        __syncwarp();
        if (!bad && mine) {
            const int y = (int)(((long long)blk * a.Hkv + wi.t.kvh) * a.bs) + tok % a.bs;
            tma_load_2d(stage + s8 * F8_BYTES + lane * box_rows * 128, map, 0, y, full8[s8], pol);
        }
        __syncwarp();
        ++issued;
        step(wi);
    };
    auto convert = [&]() {
        const int s8 = conv % S8, c = conv % R;
        const bool got = !*abort_flag && mbar_wait_bounded(full8[s8], (uint32_t)((conv / S8) & 1), a.wait_limit) &&
                         mbar_wait_bounded(empty[c], (uint32_t)(((conv / R) & 1) ^ 1), a.wait_limit);
        if (!__all_sync(0xffffffffu, got)) return fail();
        const uint8_t *src = stage_p + s8 * F8_BYTES;
        uint8_t *dst = ring + c * KV_BYTES;
#pragma unroll 4
        for (int i = 0; i < PN / 4; ++i) {   // 4 rows x 8 code chunks per pass
            const int r = 4 * i + (lane >> 3), j = lane & 7;
            const uint4 x = *reinterpret_cast<const uint4 *>(src + r * 128 + ((j ^ (r & 7)) << 4));
            const uint4 lo = make_uint4(e4m3x2_lo_to_f16x2(x.x), e4m3x2_hi_to_f16x2(x.x), e4m3x2_lo_to_f16x2(x.y),
                                        e4m3x2_hi_to_f16x2(x.y));
            const uint4 hi = make_uint4(e4m3x2_lo_to_f16x2(x.z), e4m3x2_hi_to_f16x2(x.z), e4m3x2_lo_to_f16x2(x.w),
                                        e4m3x2_hi_to_f16x2(x.w));
            uint8_t *row = dst + (j >> 2) * (PN * 128) + r * 128;
            const int c0 = 2 * (j & 3);
            *reinterpret_cast<uint4 *>(row + ((c0 ^ (r & 7)) << 4)) = lo;
            *reinterpret_cast<uint4 *>(row + (((c0 + 1) ^ (r & 7)) << 4)) = hi;
        }
        // the tile, written through the generic proxy, is for the tensor cores;
        // the staged codes have been read before their slot is refilled
        fence_proxy_async_smem();
        __syncwarp();
        if (lane == 0) mbar_arrive(full[c]);
        ++conv;
        step(wc);
    };
    while (ok && wc.item < total) {
        while (wi.item < total && issued < conv + S8) issue();
        convert();
    }
    // staged copies not converted (only after a failure) land before the warp leaves
    for (int k = conv; k < issued; ++k) mbar_wait_bounded(full8[k % S8], (uint32_t)((k / S8) & 1), WAIT_LIMIT);
}

// ----------------------------------------------------------- MMA issuer

template <int KV>
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
        const PfTile t = pf_tile(a, item);
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

template <int KV>
__device__ void pf_softmax(uint8_t *smem, const PrefillArgs &a, const PfBars &bb, uint32_t tmem,
                           volatile int *abort_flag, int total) {
    using L = PfL<KV>;
    constexpr int PST = L::R;
    constexpr int OFF_V = L::OFF_V, OFF_CTRL = L::OFF_CTRL;
    const int tid = threadIdx.x - 96;             // 0 .. 127
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
    for (int item = blockIdx.x; item < total && ok; item += gridDim.x) {
        const PfTile t = pf_tile(a, item);
        const int tok = m / a.G, hh = m - tok * a.G;
        const bool valid = tok < t.ntok;
        const long long qrow = ((long long)(t.q0 + t.row0 + tok) * a.Hq + t.kvh * a.G + hh) * PD;
        // ---- Q row into this thread's lane of the tensor-memory A tile, two
        // dims per column (zeros past the new tokens); the previous tile's
        // products, which read Q, are done (its last PV was waited for)
        {
            const uint4 *src = reinterpret_cast<const uint4 *>(a.query + qrow);
#pragma unroll
            for (int h = 0; h < 2; ++h) {
                uint32_t r[32];
#pragma unroll
                for (int c = 0; c < 8; ++c) {
                    const uint4 v = valid ? __ldg(src + 8 * h + c) : make_uint4(0, 0, 0, 0);
                    r[4 * c] = v.x;
                    r[4 * c + 1] = v.y;
                    r[4 * c + 2] = v.z;
                    r[4 * c + 3] = v.w;
                }
                tmem_st32(trow + TM_Q + 32 * h, r);
            }
            tmem_wait_st();
            tc_fence_before_sync();
            mbar_arrive(bb.qfull);
        }
        const int vis = valid ? t.C + t.row0 + tok : 1;   // positions this row sees
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
        // ---- epilogue: O / l once the tile's last PV (number g - 1) is done
        if (!wait(bb.pvdone[(g - 1) & 1], ((g - 1) >> 1) & 1)) break;
        tc_fence_after_sync();
        const bool bad = *pf_bad_slot(smem, OFF_CTRL, pf_local(item)) == pf_local(item) + 1;
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

template <int KV>
__global__ void __launch_bounds__(PF_THREADS, 1) prefill_kernel(const __grid_constant__ CUtensorMap tmk,
                                                                 const __grid_constant__ CUtensorMap tmv,
                                                                 const PrefillArgs a) {
    extern __shared__ uint8_t smem_raw[];
    uint8_t *smem = reinterpret_cast<uint8_t *>((reinterpret_cast<uintptr_t>(smem_raw) + 1023) & ~uintptr_t(1023));
    using L = PfL<KV>;
    const PfBars bb = pf_bars(smem, L::OFF_CTRL);
    volatile int *abort_flag = reinterpret_cast<volatile int *>(smem + L::OFF_CTRL + CTRL_ABORT);
    const int warp = threadIdx.x >> 5;
    const int total = *reinterpret_cast<volatile int *>(&a.hdr->pf_items);   // written by the prep kernel
    if (threadIdx.x == 0) {
        for (int s = 0; s < L::R; ++s) {
            mbar_init(bb.kfull[s], 1);
            mbar_init(bb.kempty[s], 1);
            mbar_init(bb.vfull[s], 1);
            mbar_init(bb.vempty[s], 1);
        }
        for (int s = 0; s < L::S8; ++s) {
            mbar_init(bb.k8full[s], 1);
            mbar_init(bb.v8full[s], 1);
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
    if (warp < 2) {
        if constexpr (L::F8)
            pf_producer_fp8(smem, warp ? &tmv : &tmk, a, bb, abort_flag, total, warp);
        else
            pf_producer<KV>(smem, warp ? &tmv : &tmk, a, bb, abort_flag, total, warp);
    } else if (warp == 2) {
        if ((threadIdx.x & 31) == 0) {
            pf_mma<KV>(smem, a, bb, tmem, KV == PA_KV_BF16, abort_flag, total);
            // every MMA issued has completed before tensor memory is released
            umma_commit(bb.flags);
            mbar_wait_bounded(bb.flags, 0, WAIT_LIMIT);
        }
        __syncwarp();
    } else {
        pf_softmax<KV>(smem, a, bb, tmem, abort_flag, total);
    }
    tc_fence_before_sync();
    __syncthreads();
    if (warp == 2) {
        tc_fence_after_sync();
        tmem_dealloc(tmem, TMEM_COLS);
    }
}

template <int KV>
int launch_prefill_kv(const CUtensorMap &tmk, const CUtensorMap &tmv, const PrefillArgs &args, long long max_items,
                      cudaStream_t st) {
    static int grid = 0;
    static cudaError_t init_err = cudaSuccess;
    static std::once_flag once;
    std::call_once(once, [] {   // one CTA per SM
        init_err =
            cudaFuncSetAttribute(prefill_kernel<KV>, cudaFuncAttributeMaxDynamicSharedMemorySize, PfL<KV>::SMEM);
        int dev = 0, sms = 0;
        if (init_err == cudaSuccess) init_err = cudaGetDevice(&dev);
        if (init_err == cudaSuccess) init_err = cudaDeviceGetAttribute(&sms, cudaDevAttrMultiProcessorCount, dev);
        grid = sms;
    });
    if (init_err != cudaSuccess || grid <= 0) return PA_ERR_CUDA;
    const int g = (int)(max_items < grid ? (max_items > 0 ? max_items : 1) : grid);
    prefill_kernel<KV><<<g, PF_THREADS, PfL<KV>::SMEM, st>>>(tmk, tmv, args);
    return cuda_status(cudaGetLastError());
}

}  // namespace

int launch_prefill(int kv, const CUtensorMap &tmk, const CUtensorMap &tmv, const PrefillArgs &args,
                   long long max_items, cudaStream_t st) {
    if (kv == PA_KV_BF16) return launch_prefill_kv<PA_KV_BF16>(tmk, tmv, args, max_items, st);
    if (kv == PA_KV_F16) return launch_prefill_kv<PA_KV_F16>(tmk, tmv, args, max_items, st);
    if (kv == PA_KV_FP8_E4M3) return launch_prefill_kv<PA_KV_FP8_E4M3>(tmk, tmv, args, max_items, st);
    return PA_ERR_UNSUPPORTED;
}

}  // namespace pa
