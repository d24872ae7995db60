// Pieces shared by the tensor-core kernels for runs of new tokens
// (prefill.cu, narrow.cu): tile sizes, the geometry of a work item, the
// producer warp that streams K/V tiles through the block table by TMA, and the
// warps that turn staged FP8 E4M3 codes into 16-bit tiles.
#pragma once

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

// Geometry of one work tile, the same in every warp.
// Modes of the one-tile kernel: new tokens of a sequence attending causally
// (their output rows), or the members of a shared-prefix group over a range
// of their shared blocks (their partial rows, merged by the decode kernel).
constexpr int PF_CAUSAL = 0, PF_SHARED = 1;

// seq: the block-table row; tokens kv0 .. kv0 + L - 1 of it are the KV range,
// nkv tiles of PN tokens; rows: ntok query tokens (or members) from query row
// q0 + row0, G heads each; C: positions the first new token sees (causal).
// piece / np / sid: a work item may be one of np pieces of a sequence's KV
// range (the narrow kernel's split of its last round of items); sid indexes
// the split items (-1: a whole item).
struct PfTile {
    int seq, kvh, row0, ntok, C, nkv, L, q0, kv0;
    int piece, np, sid;
};

// Row tile `rt` (128 / G consecutive new tokens) of sequence `seq`, kv head kvh.
__device__ __forceinline__ PfTile pf_row_tile(const PrefillArgs &a, int seq, int kvh, int rt) {
    PfTile t;
    t.seq = seq;
    t.kvh = kvh;
    const int tpt = PM / a.G;               // new tokens per tile
    t.L = a.context_lens[t.seq];
    t.q0 = a.query_start[t.seq];
    const int T = a.query_start[t.seq + 1] - t.q0;
    t.row0 = rt * tpt;                      // first new token of the tile
    t.ntok = min(tpt, T - t.row0);
    t.C = t.L - T + 1;                      // positions the first new token sees
    t.nkv = (t.C + t.row0 + t.ntok - 1 + PN - 1) / PN;
    t.kv0 = 0;
    t.piece = 0;
    t.np = 1;
    t.sid = -1;
    return t;
}

// Work item of the one-tile kernel: (row tile, kv head).
__device__ __forceinline__ PfTile pf_tile(const PrefillArgs &a, int item) {
    const int4 rec = a.tiles[item / a.Hkv];
    return pf_row_tile(a, rec.x, item % a.Hkv, rec.y);
}

// Work item of the shared-prefix mode: (first member, members, shared range
// [t0, t1)) x kv head.  The members' query rows (G heads each, member-major)
// all see the whole range, read through the first member's table (the
// members' first shared / block_size entries are the same blocks).
__device__ __forceinline__ PfTile pf_shared_item(const PrefillArgs &a, int item) {
    const int4 rec = a.tiles[item / a.Hkv];
    PfTile t;
    t.seq = rec.x;
    t.kvh = item % a.Hkv;
    t.q0 = rec.x;        // the members' query rows are rows rec.x ... of the decode query
    t.row0 = 0;
    t.ntok = rec.y;      // members
    t.kv0 = rec.z;
    t.L = rec.w - rec.z; // tokens of the range
    t.C = t.L;
    t.nkv = (t.L + PN - 1) / PN;
    t.piece = 0;
    t.np = 1;
    t.sid = -1;
    return t;
}

template <int MODE>
__device__ __forceinline__ PfTile pf_item(const PrefillArgs &a, int item) {
    if constexpr (MODE == PF_SHARED)
        return pf_shared_item(a, item);
    else
        return pf_tile(a, item);
}

// What a producer warp needs of a work item: the KV range it streams, tokens
// kv0 .. kv0 + L - 1 of table row seq.
struct PfRange {
    int seq, kvh, nkv, L, kv0;
};

__device__ __forceinline__ void pf_error(const PrefillArgs &a) { atomicExch(&a.hdr->error, PA_ERR_TIMEOUT); }

// The CTA-local index of a work item (items are dealt round-robin) and its
// out-of-range mark in the control block.
__device__ __forceinline__ int pf_local(int item) { return (item - (int)blockIdx.x) / (int)gridDim.x; }
__device__ __forceinline__ volatile int *pf_bad_slot(uint8_t *smem, int off_ctrl, int local) {
    return reinterpret_cast<volatile int *>(smem + off_ctrl + CTRL_BAD) + (local % BAD_SLOTS);
}

// ----------------------------------------------------------- producer

// A producer warp: streams the K or V tiles (NMAP = 1: map[0]) or both (NMAP
// = 2: map[0] into ring 0, map[1] into ring 1, the same block ids) of every
// work item of this CTA -- range(item) gives the item's KV range -- into rings
// of PST stages at byte offsets off_ring[] of shared memory, paced by full[]
// and empty[].  A 16-bit tile is two 64-column boxes per row group; an FP8
// tile (F8: codes for a staging ring) one 128-byte box per row group.
// The copies carry the L2 evict-first policy: a tile read by one CTA once
// (narrow and single-tile items) should not displace anything, and even where
// neighbouring pairs of row tiles re-read a range (long chunks) evict-first
// measured no slower than evict-normal (speculative steps of 8 and 16 tokens
// on the one-tile kernel 5 % faster, of 4 tokens on the narrow kernel 7 %).
template <int PST, bool F8, int NMAP, class RangeOf>
__device__ void pf_stream(uint8_t *smem, const int *off_ring, int off_ctrl, const BarRing *full, const BarRing *empty,
                          const CUtensorMap *const *map, const PrefillArgs &a, volatile int *abort_flag, int total,
                          RangeOf range) {
    constexpr int TILE = F8 ? F8_BYTES : KV_BYTES;
    constexpr int NBOX = F8 ? 1 : 2;
    const int lane = threadIdx.x & 31;
    const uint64_t pol = policy_evict_first();
    const int box_rows = a.bs < 16 ? a.bs : 16;    // rows per TMA box: one box per block or 16-row group
    int cnt = 0;
    // Before leaving, the last copy into every stage has landed (bounded).
    auto drain = [&]() {
        for (int r = 0; r < NMAP; ++r)
            for (int s = 0; s < PST; ++s)
                if (cnt > s)
                    mbar_wait_bounded(full[r][s], (uint32_t)(((s + (cnt - 1 - s) / PST * PST) / PST) & 1), WAIT_LIMIT);
    };
    // Lane j owns box j of a tile (tokens t0 + j box_rows ..).  Its block id
    // is loaded before the wait for the ring slot, so that the load's round
    // trip overlaps the wait.  (Loading it two tiles ahead instead, through a
    // cursor carried across iterations, made every kernel slower: the
    // speculative fp8 step 0.381 -> 0.437 ms, chunked fp8 0.727 -> 0.773.)
    for (int item = blockIdx.x; item < total; item += gridDim.x) {
        const PfRange t = range(item);
        const int32_t *row = a.block_tables + (long long)t.seq * a.mbps;
        for (int n = 0; n < t.nkv; ++n) {
            const int tok = n * PN + lane * box_rows;   // within the range
            const bool mine = lane < PN / box_rows && tok < t.L;
            const int32_t blk = mine ? __ldg(row + (t.kv0 + tok) / a.bs) : 0;
            const int s = cnt % PST;
            // the warp decides together (no lane may leave alone)
            bool got = !*abort_flag;
#pragma unroll
            for (int r = 0; r < NMAP; ++r)
                got = got && mbar_wait_bounded(empty[r][s], ((cnt / PST) & 1) ^ 1, a.wait_limit);
            if (!__all_sync(0xffffffffu, got)) {
                if (lane == 0) pf_error(a);
                *abort_flag = 1;
                drain();
                return;
            }
            const unsigned boxes = __ballot_sync(0xffffffffu, mine);
            const bool bad = __any_sync(0xffffffffu, mine && (blk < 0 || blk >= a.num_blocks));
            if (lane == 0) {
                if (bad) *pf_bad_slot(smem, off_ctrl, pf_local(item)) = pf_local(item) + 1;
#pragma unroll
                for (int r = 0; r < NMAP; ++r)
                    mbar_arrive_expect_tx(full[r][s], bad ? 0u : (uint32_t)(__popc(boxes) * NBOX * box_rows * 128));
            }
            __syncwarp();
            if (!bad && mine) {
                const int y = (int)(((long long)blk * a.Hkv + t.kvh) * a.bs) + (t.kv0 + tok) % a.bs;
#pragma unroll
                for (int r = 0; r < NMAP; ++r) {
                    const uint32_t dst = smem_u32(smem) + off_ring[r] + s * TILE + lane * box_rows * 128;
                    tma_load_2d(dst, map[r], 0, y, full[r][s], pol);
                    if (!F8) tma_load_2d(dst + PN * 128, map[r], 64, y, full[r][s], pol);
                }
            }
            __syncwarp();
            ++cnt;
        }
    }
    drain();
}

// FP8 cache: a staging warp streams the codes of the K and V tiles into
// staging rings (pf_stream, one 128-byte box column per block), and NPART
// warps per cache (part `part` of the rows each) turn each staged tile into
// the 16-bit tile the MMAs read, in the same swizzled layout a 16-bit TMA copy
// would have written: code chunk j (dims 16 j .. 16 j + 15) of row r becomes
// fp16 chunks 2 (j % 4) and 2 (j % 4) + 1 of the 64-dim block j / 4.  Every
// E4M3 value is an fp16 value, so the tile is exact; the scales are applied to
// the scores and the output.  The converting warp loads no block id and issues
// no copy, so it never waits on memory latency except for the staged tile
// itself.  stage_p / ring: the staging ring (S8 stages) and the 16-bit ring (R
// stages) of one cache; full8 / empty8 pace the first, full / empty the
// second; nkv_of(item): the KV tiles of a work item.
template <int R, int S8, int NPART, class NkvOf>
__device__ void pf_convert_ring(const uint8_t *stage_p, uint8_t *ring, BarRing full8, BarRing empty8, BarRing full,
                                BarRing empty, const PrefillArgs &a, volatile int *abort_flag, int total, int part,
                                NkvOf nkv_of) {
    static_assert(NPART == 2 || NPART == 4, "rows of a tile per converting warp");
    const int lane = threadIdx.x & 31;
    int conv = 0;
    for (int item = blockIdx.x; item < total; item += gridDim.x) {
        const int nkv = nkv_of(item);
        for (int n = 0; n < nkv; ++n, ++conv) {
            const int s8 = conv % S8, c = conv % R;
            const bool got = !*abort_flag &&
                             mbar_wait_bounded(full8[s8], (uint32_t)((conv / S8) & 1), a.wait_limit) &&
                             mbar_wait_bounded(empty[c], (uint32_t)(((conv / R) & 1) ^ 1), a.wait_limit);
            if (!__all_sync(0xffffffffu, got)) {
                if (lane == 0) pf_error(a);
                *abort_flag = 1;
                return;   // the staging warp drains its own copies
            }
            const uint8_t *src = stage_p + s8 * F8_BYTES;
            uint8_t *dst = ring + c * KV_BYTES;
            // lane: row r, code chunk j; its fp16 chunks 2 (j % 4) (dims 0-7 of
            // the chunk) and 2 (j % 4) + 1 (dims 8-15) go to the 64-dim half
            // j / 4.  Lanes of the second half store the odd chunk first, so
            // each group of 8 lanes (one row) stores to 8 distinct 16-byte bank
            // groups in either store (the halves are 16 KB apart: same banks).
            const int j = lane & 7, h = j >> 2, c0 = 2 * (j & 3);
#pragma unroll 4
            for (int i = part * (PN / 4 / NPART); i < (part + 1) * (PN / 4 / NPART); ++i) {   // this warp's rows
                const int r = 4 * i + (lane >> 3);
                const uint4 x = *reinterpret_cast<const uint4 *>(src + r * 128 + ((j ^ (r & 7)) << 4));
                const uint32_t a0 = h ? x.z : x.x, a1 = h ? x.w : x.y, b0 = h ? x.x : x.z, b1 = h ? x.y : x.w;
                const uint4 first = make_uint4(e4m3x2_lo_to_f16x2(a0), e4m3x2_hi_to_f16x2(a0),
                                               e4m3x2_lo_to_f16x2(a1), e4m3x2_hi_to_f16x2(a1));
                const uint4 second = make_uint4(e4m3x2_lo_to_f16x2(b0), e4m3x2_hi_to_f16x2(b0),
                                                e4m3x2_lo_to_f16x2(b1), e4m3x2_hi_to_f16x2(b1));
                uint8_t *row = dst + h * (PN * 128) + r * 128;
                *reinterpret_cast<uint4 *>(row + (((c0 + h) ^ (r & 7)) << 4)) = first;
                *reinterpret_cast<uint4 *>(row + (((c0 + 1 - h) ^ (r & 7)) << 4)) = second;
            }
            // the tile, written through the generic proxy, is for the tensor
            // cores, and the staged codes were read before the slot is refilled
            fence_proxy_async_smem();
            __syncwarp();
            if (lane == 0) {
                mbar_arrive(full[c]);
                mbar_arrive(empty8[s8]);
            }
        }
    }
}

}  // namespace
}  // namespace pa
