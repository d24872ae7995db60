// Shared by the decode translation units: workspace layout, work-item
// records, the persistent decode kernel and its launch.  See decode.cu for
// what is computed and how.
#pragma once

#include <cudaTypedefs.h>

#include <cmath>
#include <cstdlib>
#include <mutex>
#include <vector>

#include "common.cuh"

#ifndef PA_DECODE_CONSUMERS
#define PA_DECODE_CONSUMERS 1
#endif
#ifndef PA_DECODE_DEPTH
#define PA_DECODE_DEPTH 2
#endif
#ifndef PA_DECODE_MINB_FP8
#define PA_DECODE_MINB_FP8 6
#endif
#ifndef PA_DECODE_DEPTH_FP8
#define PA_DECODE_DEPTH_FP8 (2 * PA_DECODE_DEPTH)
#endif
#ifndef PA_FP8_LATE_V
#define PA_FP8_LATE_V 0
#endif
#ifndef PA_DECODE_MINB_WIDE
#define PA_DECODE_MINB_WIDE 4
#endif
#ifndef PA_DECODE_DEPTH_WIDE
#define PA_DECODE_DEPTH_WIDE 5
#endif
#ifndef PA_DECODE_MINB
#define PA_DECODE_MINB 8
#endif
#ifndef PA_DECODE_SPLIT
#define PA_DECODE_SPLIT 1
#endif
#ifndef PA_CAUSAL_L2
#define PA_CAUSAL_L2 0
#endif
#ifndef PA_CAUSAL_NT
#define PA_CAUSAL_NT 2
#endif

namespace pa {


constexpr int MAX_PART_TOKENS = 1024;           // largest partition (one work item)
#ifndef PA_DECODE_TARGET_ITEMS
#define PA_DECODE_TARGET_ITEMS 4096
#endif
constexpr long long TARGET_ITEMS = PA_DECODE_TARGET_ITEMS;   // work items wanted for load balance
constexpr int CHUNK = 16;                       // tokens per pipeline stage (one MMA K step of P V)
constexpr int NC = PA_DECODE_CONSUMERS;         // consumer warps per CTA
constexpr int NWARPS = NC + 1;                  // + the producer warp
constexpr long long WAIT_LIMIT = 1LL << 31;     // clock cycles (about a second): default wait bound, drain bound
constexpr int PREP_THREADS = 1024;
constexpr float RESCALE_THRESHOLD = 8.f;        // log2 units: rescale when the max grows by more than 2^8
constexpr int ENTRIES = MAX_PART_TOKENS / 8 / 32;   // block-table entries per lane for one item (block size >= 8)

// Partition size: the largest of 1024, 512, 256 tokens whose estimated item
// count (sequences x kv heads x partitions of the longest context) reaches
// the target, so that long batches get long, cheap items and short ones
// still spread over every SM.  An item's fixed costs (its query rows, the
// partials it writes and merges) grow with the GQA group G, so groups
// smaller than 8 aim at 8 / G times as many items: at G = 1 (64 sequences of
// 512 .. 2048 tokens) that is 0.244 -> 0.228 ms, while G = 8 keeps its
// 1024-token items.  It depends on the shapes only, so a given call always
// partitions the same way.
inline int part_tokens(int B, int Hkv, int G, int max_ctx) {
    const long long target = TARGET_ITEMS * (G < 8 && G > 0 ? 8 / G : 1);
    for (int pt = MAX_PART_TOKENS; pt > 256; pt /= 2)
        if ((long long)B * Hkv * ((max_ctx + pt - 1) / pt) >= target) return pt;
    return 256;
}

struct WsHeader {
    int error;
    int total_items;
    int counter;
    int pf_items;    // multi-token form: work items of the one-tile tensor-core kernel
    int pf2_items;   // multi-token form: work items of the two-tile tensor-core kernel
    int pfn_items;   // multi-token form: work items of the narrow tensor-core kernel
    int pfn_whole;   // ... of which the first pfn_whole are whole (sequence, kv head) items,
    int pfn_split;   // the others pfn_split pieces each of the last items' KV ranges
    int pad[56];
};
static_assert(sizeof(WsHeader) == 256, "header is one 256-byte line");

// The narrow tensor-core kernel merges the four partial results of a work
// item's rows through a scratch area of the workspace: per CTA (at most
// NW_MAX_CTAS of them) and item parity, 4 x 128 dims x 32 rows of fp32 O and
// 4 x 32 (m, l) pairs.
constexpr int NW_MAX_CTAS = 160;
constexpr size_t NW_SCRATCH_PER_CTA = 2 * (4 * 128 * 32 * 4 + 4 * 32 * 8);
// ... and, after the CTAs' areas, the pieces of split items (at most
// NW_MAX_CTAS of them): 32 rows of fp32 O (128 dims) and (m, l) each, and a
// ticket per split item.
constexpr size_t NW_SPLIT_BYTES = (size_t)NW_MAX_CTAS * 32 * (128 * 4 + 8) + NW_MAX_CTAS * 4;

struct NwSplitArea {
    float *o;       // [piece][row][128]
    float2 *ml;     // [piece][row]
    int *tickets;   // [split item]
};

__host__ __device__ inline NwSplitArea nw_split_area(uint8_t *nscr) {
    uint8_t *p = nscr + (size_t)NW_MAX_CTAS * NW_SCRATCH_PER_CTA;
    NwSplitArea s;
    s.o = reinterpret_cast<float *>(p);
    p += (size_t)NW_MAX_CTAS * 32 * 128 * 4;
    s.ml = reinterpret_cast<float2 *>(p);
    p += (size_t)NW_MAX_CTAS * 32 * 8;
    s.tickets = reinterpret_cast<int *>(p);
    return s;
}

struct WsLayout {
    size_t part_off, gsize, gshared, items, grp, ml, o, ptiles, ppairs, ntiles, nscr, total;
    int pmax, pt;
    long long item_cap, ptile_cap;
};

inline size_t up256(size_t x) { return (x + 255) & ~size_t(255); }

// Workspace of one call.  grouped: sequences may share a prefix, which adds
// at most one partition per sequence and as many shared items again.
inline WsLayout ws_layout(int B, int Hq, int Hkv, int D, int max_ctx, bool grouped) {
    WsLayout w;
    w.pt = part_tokens(B, Hkv, Hq / Hkv, max_ctx);
    w.pmax = max_ctx > 0 ? (max_ctx + w.pt - 1) / w.pt : 1;
    const long long parts = (long long)B * (w.pmax + (grouped ? 1 : 0));   // partial-result rows per head
    w.item_cap = (long long)B * w.pmax * (grouped ? 2 : 1);
    size_t off = sizeof(WsHeader);
    w.part_off = off;
    off += up256(sizeof(int) * ((size_t)B + 1));
    w.gsize = off;
    if (grouped) off += up256(sizeof(int) * (size_t)B);
    w.gshared = off;
    if (grouped) off += up256(sizeof(int) * (size_t)B);
    w.items = off;
    off += up256(2 * sizeof(int4) * (size_t)w.item_cap);
    const bool multi = w.pmax > 1 || grouped;
    w.grp = off;
    if (multi) off += up256(sizeof(int) * (size_t)B * Hq);
    w.ml = off;
    if (multi) off += up256(sizeof(float2) * (size_t)parts * Hq);
    w.o = off;
    if (multi) off += up256(sizeof(float) * (size_t)parts * Hq * D);
    // grouped calls: the list of shared ranges for the tensor-core kernel (at
    // most one per leader, partition and member group: B x pmax)
    w.ptile_cap = grouped ? (long long)B * w.pmax : 0;
    w.ptiles = off;
    off += up256(sizeof(int4) * (size_t)w.ptile_cap);
    w.ppairs = off;
    w.ntiles = off;
    // the narrow kernel's merge scratch (shared ranges of up to 32 rows)
    w.nscr = off;
    if (grouped && D == 128 && 32 % (Hq / Hkv) == 0 && 32 / (Hq / Hkv) >= 4) off += NW_MAX_CTAS * NW_SCRATCH_PER_CTA;
    w.total = off;
    return w;
}

// Workspace of one call of the multi-token (causal) form: NQ query rows of B
// sequences; per row its visible length and partial-row offset, per sequence
// the first of its member groups (ms consecutive rows read together), and a
// partial row per (query row, partition).
inline WsLayout ws_layout_causal(int B, int NQ, int Hq, int Hkv, int D, int max_ctx) {
    WsLayout w;
    const int G = Hq / Hkv;
    const int ms = 8 * PA_CAUSAL_NT / G > 1 ? 8 * PA_CAUSAL_NT / G : 1;
    w.pt = part_tokens(B, Hkv, Hq / Hkv, max_ctx);
    w.pmax = max_ctx > 0 ? (max_ctx + w.pt - 1) / w.pt : 1;
    w.item_cap = (long long)w.pmax * ((NQ + ms - 1) / ms + B);
    const long long parts = (long long)NQ * w.pmax;
    size_t off = sizeof(WsHeader);
    w.part_off = off;
    off += up256(sizeof(int) * ((size_t)NQ + 1));
    w.gsize = off;   // visible length of every query row
    off += up256(sizeof(int) * ((size_t)NQ + 1));
    w.gshared = off;   // first member group of every sequence
    off += up256(sizeof(int) * ((size_t)B + 1));
    w.items = off;
    off += up256(2 * sizeof(int4) * (size_t)w.item_cap);
    w.grp = off;
    off += up256(sizeof(int) * ((size_t)NQ + 1) * Hkv);
    w.ml = off;
    off += up256(sizeof(float2) * (size_t)parts * Hq);
    w.o = off;
    off += up256(sizeof(float) * (size_t)parts * Hq * D);
    // prefill tiles: 128 query rows (new tokens x G) of one sequence each,
    // listed alone or in pairs of neighbouring tiles
    w.ptile_cap = ((long long)NQ * G + 127) / 128 + B;
    w.ptiles = off;
    off += up256(sizeof(int4) * (size_t)w.ptile_cap);
    w.ppairs = off;
    off += up256(sizeof(int4) * (size_t)w.ptile_cap);
    // narrow tensor-core kernel: sequences whose new tokens fill at most 32
    // rows, and its merge scratch
    w.ntiles = off;
    off += up256(sizeof(int4) * (size_t)B);
    w.nscr = off;
    if (D == 128 && 128 % G == 0) off += NW_MAX_CTAS * NW_SCRATCH_PER_CTA + up256(NW_SPLIT_BYTES);
    w.total = off;
    return w;
}

// A work item record (two int4): a token range [t0, t1) of the caches read
// for nmem consecutive sequences seq0 .. seq0 + nmem - 1 that share those
// blocks, the range's partition index in each member's partition list, the
// group's shared length, the context length of seq0 and the partial's
// canonical row index -- or -1 for a shared-prefix item, whose members each
// have their own (part_off[member] + partition).
struct ItemRec {
    int4 a;   // seq0, nmem, t0, t1
    int4 b;   // pidx, shared, L0, canon
};

struct DecodeArgs {
    uint16_t *out;           // fp16 or bf16 bit patterns
    const uint16_t *query;
    const int32_t *block_tables;
    const int32_t *context_lens;
    int Hq, Hkv, G, bs, mbps, pt, ms;
    int pts;                 // partition length of shared ranges (pt, or longer when the tensor cores take them)
    long long num_blocks;
    long long wait_limit;   // bound of every pipeline wait, clock cycles
    float scale_log2;        // softmax scale (times the K scale of an fp8 cache) * log2(e)
    float v_scale;           // V scale of an fp8 cache (1 otherwise)
    int tc_shared;           // shared ranges were reduced by the tensor-core kernel before this one
    WsHeader *hdr;
    const int *part_off;
    const ItemRec *items;
    int *grp;
    float2 *ws_ml;
    float *ws_o;
};

// What the producer tells a consumer about its next item (64 bytes).
struct ItemDesc {
    int seq0, kvh, nmem, pidx, shared, P0, canon0, nchunks;
    int ntok_last, bad, end, t0, pad[4];
};

// KV: cache element type (PA_KV_F16, PA_KV_BF16, PA_KV_FP8_E4M3).
template <int D, int NT, int KV>
struct Cfg {
    static constexpr bool FP8 = KV == PA_KV_FP8_E4M3;
    static constexpr int ESZ = FP8 ? 1 : 2;               // bytes per cache element
    // pipeline stages per consumer: a two-tile consumer keeps fewer warps on
    // an SM (registers), so each keeps more stages in flight; one-byte
    // elements make a stage half as large, so there are twice as many
    static constexpr int DEPTH = NT == 1 ? (FP8 ? PA_DECODE_DEPTH_FP8 : PA_DECODE_DEPTH)
                                         : PA_DECODE_DEPTH_WIDE * (FP8 ? 2 : 1);
    static constexpr int BOXES = D * ESZ / 128;            // 128-byte boxes per tile row
    static constexpr int BOX_ELEMS = 128 / ESZ;            // elements per box row
    static constexpr int TILE = BOXES * CHUNK * 128;       // one 16-token K or V tile
    static constexpr int STAGE = 2 * TILE;                 // K tile then V tile
    static constexpr int QSLOT = NT * 8 * D * 2;           // the group's query rows (16-bit)
    static constexpr int DATA = DEPTH * STAGE + 2 * QSLOT; // per consumer, a multiple of 1024
    static constexpr int CTRL_USED = (2 * DEPTH + 2) * 8 + 16 + 2 * 64;
    static constexpr int CTRL = (CTRL_USED + 255) / 256 * 256;   // per consumer: barriers and descriptors
    // CTA shape.  In general one producer warp feeds NC consumer warps and
    // the CTA's warps all hold what the consumer needs (the register count
    // bounds the CTAs per SM).  Single-token decode at head_dim 128 (SPLIT)
    // is bound by its consumers' latency, so it gives them the registers the
    // producers do not need: four producer warps (one warpgroup, each feeding
    // one consumer) lower their registers to PROD_REGS and hand them to the
    // four consumer warps (the other warpgroup, CONS_REGS), two CTAs per SM.
    // FP8 (167 registers a consumer) gets 8 consumer warps per SM instead of
    // 6; fp16/bf16 keep 8 but without the spills of a 128-register bound.  The
    // split must fit the pool the CTA is launched with (threads x
    // LAUNCH_REGS); the host checks the compiled count before the first launch.
    static constexpr bool SPLIT = NT == 1 && D == 128 && PA_DECODE_SPLIT != 0;
    static constexpr int NCON = SPLIT ? 4 : NC;             // consumer warps per CTA
    static constexpr int PER = SPLIT ? 1 : NC;              // consumers per producer warp
    static constexpr int WARPS = SPLIT ? 8 : NWARPS;
    static constexpr int MINB = SPLIT ? 2 : NT == 1 ? (FP8 ? PA_DECODE_MINB_FP8 : PA_DECODE_MINB) : PA_DECODE_MINB_WIDE;
    static constexpr int LAUNCH_REGS = 65536 / (WARPS * 32 * MINB);
    static constexpr int PROD_REGS = 80, CONS_REGS = 176;
    static_assert(!SPLIT || (WARPS == 8 && 128 * PROD_REGS + 128 * CONS_REGS <= WARPS * 32 * LAUNCH_REGS),
                  "register split");
    static constexpr int SMEM = NCON * (DATA + CTRL) + 1024;
    static_assert(BOXES >= 1, "a tile row is at least one 128-byte box");
    static_assert(DATA % 1024 == 0, "stages must stay 1024-byte aligned for the 128-byte swizzle");
};

// 16-bit output element of a cache type: bf16 for a bf16 cache, else fp16.
template <int KV>
__device__ __forceinline__ uint16_t out_bits(float x) {
    if constexpr (KV == PA_KV_BF16)
        return __bfloat16_as_ushort(__float2bfloat16_rn(x));
    else
        return __half_as_ushort(__float2half_rn(x));
}

template <int KV>
__device__ __forceinline__ uint32_t pack_p(float lo, float hi) {
    if constexpr (KV == PA_KV_BF16)
        return pack_bf162(lo, hi);
    else
        return pack_half2(lo, hi);
}

template <int KV>
__device__ __forceinline__ void mma_kv(float &d0, float &d1, float &d2, float &d3, uint32_t a0, uint32_t a1,
                                       uint32_t a2, uint32_t a3, uint32_t b0, uint32_t b1) {
    if constexpr (KV == PA_KV_BF16)
        mma_16816_bf16(d0, d1, d2, d3, a0, a1, a2, a3, b0, b1, d0, d1, d2, d3);
    else
        mma_16816(d0, d1, d2, d3, a0, a1, a2, a3, b0, b1, d0, d1, d2, d3);
}

// Byte offset, inside a swizzled tile, of 16-byte column `col` (0 .. D/8-1)
// of row `row`: 64-column boxes of CHUNK rows x 128 bytes; chunk j of row r
// sits at position j ^ (r & 7) (the TMA 128-byte swizzle).
__host__ __device__ constexpr int swz(int row, int col) {
    return (col >> 3) * (CHUNK * 128) + row * 128 + (((col & 7) ^ (row & 7)) << 4);
}

// Partitions of one sequence: its shared prefix [0, S) and its own range
// [S, L), each cut into pieces of pt tokens (S = 0 for a sequence that
// shares nothing).
// Partitions of a sequence of L positions whose first S are shared: the shared
// range in pieces of pts, the rest in pieces of pt.
__device__ __forceinline__ int partitions_of(int L, int S, int pt, int pts) {
    return (S + pts - 1) / pts + (L - S + pt - 1) / pt;
}

namespace {

// ------------------------------------------------------------ decode

struct ConsumerSmem {
    uint32_t data;        // shared address of the consumer's stages and query slots
    uint64_t *full;       // [DEPTH]: stage loaded (producer arrive + TMA bytes)
    uint64_t *empty;      // [DEPTH]: stage consumed (consumer arrive)
    uint64_t *qfree;      // [2]: query slot / descriptor free again
    ItemDesc *desc;       // [2]
};

template <int D, int NT, int KV>
__device__ __forceinline__ ConsumerSmem consumer_smem(uint8_t *smem, int c) {
    using C = Cfg<D, NT, KV>;
    constexpr int DEPTH = C::DEPTH;
    uint8_t *ctrl = smem + C::NCON * C::DATA + c * C::CTRL;
    ConsumerSmem s;
    s.data = smem_u32(smem + c * C::DATA);
    s.full = reinterpret_cast<uint64_t *>(ctrl);
    s.empty = s.full + DEPTH;
    s.qfree = s.empty + DEPTH;
    s.desc = reinterpret_cast<ItemDesc *>(ctrl + (2 * DEPTH + 2) * 8 + 16);
    return s;
}

// Producer warp: hands items to its consumers (C::PER of them from consumer
// c0 on) round-robin and keeps their rings full.  All lanes run the loop;
// lane 0 issues the copies.
template <int D, int NT, bool CAUSAL, int KV>
__device__ void producer(uint8_t *smem, const CUtensorMap *tmk, const CUtensorMap *tmv, const DecodeArgs &a, int c0) {
    using C = Cfg<D, NT, KV>;
    constexpr int NC = C::PER;   // this warp's consumers
    constexpr int DEPTH = C::DEPTH;
    const int lane = threadIdx.x & 31;
    const int total = a.hdr->total_items;
    const uint64_t pol = !CAUSAL || PA_CAUSAL_L2 == 0 ? policy_evict_first()
                         : PA_CAUSAL_L2 == 1               ? policy_evict_normal()
                                                           : policy_evict_last();
    const int box_rows = a.bs < CHUNK ? a.bs : CHUNK;

    // Items are prefetched in three depths so that no latency is waited on
    // when a consumer needs its next item: the work-counter ticket three items
    // ahead (lane 0), the item record two ahead, and one ahead the item's
    // fields plus, per lane, its block-table entries lane and lane + 32.
    int raw = 0;
    int nn_item = -1;
    ItemRec nn_rec;
    nn_rec.a = nn_rec.b = make_int4(0, 0, 0, 0);
    int n_item = -1, n_fb = 0;
    ItemRec n_rec = nn_rec;
    int n_e[ENTRIES];
#pragma unroll
    for (int e = 0; e < ENTRIES; ++e) n_e[e] = 0;
    auto advance = [&]() {
        n_item = nn_item;
        if (n_item >= 0) {
            n_rec = nn_rec;
            n_fb = n_rec.a.z / a.bs;
            const int nb = (n_rec.a.w + a.bs - 1) / a.bs - n_fb;
            const int trow = CAUSAL ? n_rec.b.z : n_rec.a.x;   // block-table row of the item
            const int32_t *row = a.block_tables + (long long)trow * a.mbps + n_fb;
#pragma unroll
            for (int e = 0; e < ENTRIES; ++e) n_e[e] = lane + 32 * e < nb ? row[lane + 32 * e] : 0;
        }
        const int j = __shfl_sync(0xffffffffu, raw, 0);
        nn_item = j < total ? j : -1;
        if (nn_item >= 0) nn_rec = a.items[nn_item / a.Hkv];
        if (lane == 0) raw = atomicAdd(&a.hdr->counter, 1);
    };

    // per-consumer state (NC is small and the loops over it are unrolled)
    int sc[NC], ic[NC], chunk[NC], nch[NC], t0[NC], t1[NC], fb[NC], y[NC][ENTRIES], qrow[NC], nmem[NC];
    bool done[NC], bad[NC];
#pragma unroll
    for (int c = 0; c < NC; ++c) {
        sc[c] = ic[c] = chunk[c] = nch[c] = t0[c] = t1[c] = fb[c] = qrow[c] = nmem[c] = 0;
#pragma unroll
        for (int e = 0; e < ENTRIES; ++e) y[c][e] = 0;
        done[c] = bad[c] = false;
    }
    // Before the producer leaves, every copy it issued has landed: only the
    // last issue into each ring slot can still be in flight (an earlier one
    // was consumed before its slot was reused), so wait for those, bounded
    // independently of the pipeline's own wait bound.
    auto drain = [&]() {
#pragma unroll
        for (int c = 0; c < NC; ++c) {
            const ConsumerSmem cs = consumer_smem<D, NT, KV>(smem, c0 + c);
            for (int slot = 0; slot < DEPTH; ++slot)
                if (sc[c] > slot) {
                    const int k = slot + (sc[c] - 1 - slot) / DEPTH * DEPTH;
                    mbar_wait_bounded(smem_u32(&cs.full[slot]), (uint32_t)((k / DEPTH) & 1), WAIT_LIMIT);
                }
        }
    };
    if (lane == 0) raw = atomicAdd(&a.hdr->counter, 1);
    advance();
    advance();
    int live = NC;
    while (live > 0) {
#pragma unroll
        for (int c = 0; c < NC; ++c) {
            if (done[c]) continue;
            const ConsumerSmem cs = consumer_smem<D, NT, KV>(smem, c0 + c);
            const int s = sc[c] % DEPTH;
            const uint32_t full = smem_u32(&cs.full[s]);
            // every lane waits; the warp goes on only if all of them saw the
            // phase (a lane alone past a timeout would meet the shuffles and
            // votes below without the others)
            bool ok = __all_sync(0xffffffffu,
                                 mbar_wait_bounded(smem_u32(&cs.empty[s]), ((sc[c] / DEPTH) & 1) ^ 1, a.wait_limit));
            bool first = false;
            if (ok && chunk[c] == nch[c]) {          // the consumer needs its next item
                const int q = ic[c] & 1;
                ok = __all_sync(0xffffffffu,
                                mbar_wait_bounded(smem_u32(&cs.qfree[q]), ((ic[c] >> 1) & 1) ^ 1, a.wait_limit));
                if (ok && n_item < 0) {              // nothing left: tell the consumer to stop
                    if (lane == 0) {
                        ItemDesc e;
                        e.seq0 = e.kvh = e.nmem = e.pidx = e.shared = e.P0 = e.canon0 = e.nchunks = 0;
                        e.ntok_last = e.bad = e.t0 = 0;
                        e.end = 1;
                        e.pad[0] = e.pad[1] = e.pad[2] = e.pad[3] = 0;
                        cs.desc[q] = e;
                        mbar_arrive(full);
                    }
                    ++sc[c];   // the end marker is this slot's last phase (no copies)
                    done[c] = true;
                    --live;
                    continue;
                }
                if (ok) {
                    const int kvh = n_item % a.Hkv;
                    t0[c] = n_rec.a.z;
                    t1[c] = n_rec.a.w;
                    fb[c] = n_fb;
                    nch[c] = (t1[c] - t0[c] + CHUNK - 1) / CHUNK;
                    nmem[c] = n_rec.a.y;
                    const int nb = (t1[c] + a.bs - 1) / a.bs - n_fb;
                    bool bad_any = false;
#pragma unroll
                    for (int e = 0; e < ENTRIES; ++e) {
                        bad_any |= lane + 32 * e < nb && (n_e[e] < 0 || n_e[e] >= a.num_blocks);
                        y[c][e] = (int)(((long long)n_e[e] * a.Hkv + kvh) * a.bs);
                    }
                    bad[c] = __any_sync(0xffffffffu, bad_any);
                    qrow[c] = n_rec.a.x * a.Hq + kvh * a.G;
                    chunk[c] = 0;
                    if (lane == 0) {
                        ItemDesc d;
                        d.seq0 = n_rec.a.x;
                        d.kvh = kvh;
                        d.nmem = n_rec.a.y;
                        d.pidx = n_rec.b.x;
                        d.shared = n_rec.b.y;
                        d.P0 = CAUSAL ? 0 : partitions_of(n_rec.b.z, n_rec.b.y, a.pt, a.pts);
                        d.canon0 = n_rec.b.w;
                        d.nchunks = nch[c];
                        d.ntok_last = t1[c] - (t0[c] + (nch[c] - 1) * CHUNK);
                        d.bad = bad[c] ? 1 : 0;
                        d.end = 0;
                        d.t0 = t0[c];
                        d.pad[0] = d.pad[1] = d.pad[2] = d.pad[3] = 0;
                        cs.desc[q] = d;
                    }
                    ++ic[c];
                    first = true;
                    advance();
                }
            }
            if (!ok) {   // a consumer stopped answering: record it and stop feeding everyone
                if (lane == 0) atomicExch(&a.hdr->error, PA_ERR_TIMEOUT);
                drain();
                return;
            }
            // issue chunk `chunk[c]` of the consumer's item into stage s
            const int tok0 = t0[c] + chunk[c] * CHUNK;
            const int ntok = min(CHUNK, t1[c] - tok0);
            const int lb0 = tok0 / a.bs - fb[c];
            const int lb1 = lb0 + 1;
            int va = y[c][0], vb = y[c][0];
#pragma unroll
            for (int e = 1; e < ENTRIES; ++e) {
                va = (lb0 >> 5) == e ? y[c][e] : va;
                vb = (lb1 >> 5) == e ? y[c][e] : vb;
            }
            const int ya = __shfl_sync(0xffffffffu, va, lb0 & 31);
            const int yb = __shfl_sync(0xffffffffu, vb, lb1 & 31);
            if (lane == 0) {
                const bool two = a.bs < CHUNK && ntok > a.bs;
                uint32_t bytes = bad[c] ? 0u : 2u * C::BOXES * box_rows * 128u * (two ? 2u : 1u);
                if (first && !bad[c]) bytes += (uint32_t)(nmem[c] * a.G * D * 2);
                mbar_arrive_expect_tx(full, bytes);
                if (!bad[c]) {
                    const uint32_t kdst = cs.data + s * C::STAGE;
                    const uint32_t vdst = kdst + C::TILE;
                    const int y = ya + tok0 % a.bs;
#pragma unroll
                    for (int b = 0; b < C::BOXES; ++b) {
                        tma_load_2d(kdst + b * CHUNK * 128, tmk, C::BOX_ELEMS * b, y, full, pol);
                        tma_load_2d(vdst + b * CHUNK * 128, tmv, C::BOX_ELEMS * b, y, full, pol);
                    }
                    if (two) {
#pragma unroll
                        for (int b = 0; b < C::BOXES; ++b) {
                            tma_load_2d(kdst + b * CHUNK * 128 + a.bs * 128, tmk, C::BOX_ELEMS * b, yb, full, pol);
                            tma_load_2d(vdst + b * CHUNK * 128 + a.bs * 128, tmv, C::BOX_ELEMS * b, yb, full, pol);
                        }
                    }
                    if (first)   // the query rows of every member, one run of G rows each
                        for (int m = 0; m < nmem[c]; ++m)
                            bulk_load(cs.data + DEPTH * C::STAGE + ((ic[c] - 1) & 1) * C::QSLOT + m * a.G * D * 2,
                                      a.query + ((long long)qrow[c] + (long long)m * a.Hq) * D,
                                      (uint32_t)(a.G * D * 2), full);
                }
            }
            ++chunk[c];
            ++sc[c];
        }
    }
    drain();
}

// Log-sum-exp merge of the P partitions of one (sequence, kv head) group,
// run by the consumer warp that completed the group.  Partials are read
// through L2 (other warps wrote them) with many independent loads in flight.
//  1. lane g < G walks the partitions of head g once, keeping the running
//     maximum M_g and the rescaled normaliser L_g = sum_p 2^(m_p - M_g) l_p;
//  2. all lanes sum the partial outputs: the G x D outputs, as float4s, are
//     spread over the lanes; w = 2^(m_p - M_head) / L_head.
template <int D, int KV>
__device__ void merge_group(const DecodeArgs &a, int seq, int kvh, int P) {
    const int lane = threadIdx.x & 31;
    const long long p0 = a.part_off[seq];
    const int h0 = kvh * a.G;
    float M = -INFINITY, Ls = 0.f;
    if (lane < a.G) {
        const float2 *ml = a.ws_ml + p0 * a.Hq + h0 + lane;
        int p = 0;
        for (; p + 4 <= P; p += 4) {
            float2 v[4];
#pragma unroll
            for (int u = 0; u < 4; ++u) v[u] = __ldcg(ml + (long long)(p + u) * a.Hq);
#pragma unroll
            for (int u = 0; u < 4; ++u) {
                const float nm = fmaxf(M, v[u].x);
                Ls = Ls * fast_exp2(M - nm) + v[u].y * fast_exp2(v[u].x - nm);
                M = nm;
            }
        }
        for (; p < P; ++p) {
            const float2 v = __ldcg(ml + (long long)p * a.Hq);
            const float nm = fmaxf(M, v.x);
            Ls = Ls * fast_exp2(M - nm) + v.y * fast_exp2(v.x - nm);
            M = nm;
        }
    }
    constexpr int PER_HEAD = D / 4;                 // float4s per output row
    const int nvec = a.G * PER_HEAD;                // float4s of the group's outputs
    const float *ob = a.ws_o + (p0 * a.Hq + h0) * D;
    const float2 *mlb = a.ws_ml + p0 * a.Hq + h0;
    const long long pstride = (long long)a.Hq * D / 4;   // float4s between partitions
    uint16_t *orow = a.out + ((long long)seq * a.Hq + h0) * D;
    // 64 outputs (float4s) per pass, two per lane; partitions four at a time
    for (int base = 0; base < nvec; base += 64) {
        int k[2], hd[2];
        bool on[2];
        float Mh[2], inv[2];
        float4 acc[2];
#pragma unroll
        for (int i = 0; i < 2; ++i) {
            k[i] = base + 32 * i + lane;
            on[i] = k[i] < nvec;
            hd[i] = min(k[i] / PER_HEAD, a.G - 1);
            Mh[i] = __shfl_sync(0xffffffffu, M, hd[i]);
            inv[i] = 1.f / __shfl_sync(0xffffffffu, Ls, hd[i]);
            acc[i] = make_float4(0.f, 0.f, 0.f, 0.f);
        }
        const float4 *o4 = reinterpret_cast<const float4 *>(ob);
        int p = 0;
        for (; p + 4 <= P; p += 4) {
            float4 v[4][2];
            float mp[4][2];
#pragma unroll
            for (int u = 0; u < 4; ++u)
#pragma unroll
                for (int i = 0; i < 2; ++i)
                    if (on[i]) {
                        v[u][i] = __ldcg(o4 + (p + u) * pstride + k[i]);
                        mp[u][i] = __ldcg(&mlb[(long long)(p + u) * a.Hq + hd[i]].x);
                    }
#pragma unroll
            for (int u = 0; u < 4; ++u)
#pragma unroll
                for (int i = 0; i < 2; ++i)
                    if (on[i]) {
                        const float w = fast_exp2(mp[u][i] - Mh[i]) * inv[i];
                        acc[i].x += w * v[u][i].x;
                        acc[i].y += w * v[u][i].y;
                        acc[i].z += w * v[u][i].z;
                        acc[i].w += w * v[u][i].w;
                    }
        }
        for (; p < P; ++p)
#pragma unroll
            for (int i = 0; i < 2; ++i)
                if (on[i]) {
                    const float4 v = __ldcg(o4 + p * pstride + k[i]);
                    const float w = fast_exp2(__ldcg(&mlb[(long long)p * a.Hq + hd[i]].x) - Mh[i]) * inv[i];
                    acc[i].x += w * v.x;
                    acc[i].y += w * v.y;
                    acc[i].z += w * v.z;
                    acc[i].w += w * v.w;
                }
#pragma unroll
        for (int i = 0; i < 2; ++i)
            if (on[i]) {
                uint2 h;
                h.x = (uint32_t)out_bits<KV>(acc[i].x) | ((uint32_t)out_bits<KV>(acc[i].y) << 16);
                h.y = (uint32_t)out_bits<KV>(acc[i].z) | ((uint32_t)out_bits<KV>(acc[i].w) << 16);
                *reinterpret_cast<uint2 *>(orow + 4 * k[i]) = h;
            }
    }
}

// Consumer warp c: reduces the items its producer hands it.  CAUSAL: the
// item's query rows may see different lengths of its token range (several
// new tokens of one sequence); scores past a row's own position are masked.
template <int D, int NT, bool CAUSAL, int KV>
__device__ void consumer(uint8_t *smem, int c, const DecodeArgs &a) {
    using C = Cfg<D, NT, KV>;
    constexpr int DEPTH = C::DEPTH;
    constexpr int KS = D / 16;     // MMA k-steps of S^T = K Q^T
    constexpr int MT = D / 16;     // MMA m-tiles of O^T = V^T P^T
    const int lane = threadIdx.x & 31;
    const int r = lane >> 2, cq = lane & 3;
    const ConsumerSmem cs = consumer_smem<D, NT, KV>(smem, c);

    // per-lane swizzled ldmatrix offsets; the rest of each address is a constant
    const int mi = lane >> 3, li = lane & 7;
    int koff[4], voff[4];
#pragma unroll
    for (int u = 0; u < 4; ++u) {
        koff[u] = swz((mi & 1) * 8 + li, 2 * u + (mi >> 1));       // A = K rows (tokens), d-chunk 2u + ..
        voff[u] = swz((mi >> 1) * 8 + li, 2 * u + (mi & 1));       // A = V^T via transposed loads
    }
    const float sl2 = a.scale_log2;

    // Merge tickets.  After an item has stored partials for members of
    // multi-partition sequences, it owes one ticket per such member for the
    // (member, kv head) group; lane m holds member m's.  The tickets are taken
    // after the next item's first chunk (by then the partials' stores have
    // drained, so the fence is cheap) and inspected at that item's end (so the
    // atomics' latency is hidden); a lane holding a group's last ticket has
    // the warp merge that group.
    // owe_T: tickets of the group (its partitions this kernel reduces: all P,
    // or, when the tensor-core kernel already reduced the shared ranges, the
    // member's own ones); the merge runs over all P partitions
    bool owe = false;
    int owe_seq = 0, owe_kvh = 0, owe_P = 0, owe_T = 0;   // per lane: member lane
    int pend_ticket = 0, pend_seq = 0, pend_kvh = 0, pend_P = 0, pend_T = 0;
    auto take_ticket = [&]() {
        __syncwarp();
        __threadfence();
        pend_ticket = 0;
        if (owe_P > 1) pend_ticket = atomicAdd(&a.grp[owe_seq * a.Hkv + owe_kvh], 1);
        pend_seq = owe_seq;
        pend_kvh = owe_kvh;
        pend_P = owe_P;
        pend_T = owe_T;
        owe = false;
        owe_P = 0;
    };
    auto settle = [&]() {
        unsigned last = __ballot_sync(0xffffffffu, pend_P > 1 && pend_ticket == pend_T - 1);
        if (last) __threadfence();
        while (last) {
            const int l0 = __ffs(last) - 1;
            last &= last - 1;
            merge_group<D, KV>(a, __shfl_sync(0xffffffffu, pend_seq, l0), __shfl_sync(0xffffffffu, pend_kvh, l0),
                           __shfl_sync(0xffffffffu, pend_P, l0));
        }
        pend_P = 0;
    };

    int stage = 0;
    for (int item = 0;; ++item) {
        const int q = item & 1;
        int s = stage % DEPTH;
        // warp-uniform outcome: the MMAs and shuffles below need every lane
        if (!__all_sync(0xffffffffu, mbar_wait_bounded(smem_u32(&cs.full[s]), (stage / DEPTH) & 1, a.wait_limit))) {
            if (lane == 0) atomicExch(&a.hdr->error, PA_ERR_TIMEOUT);
            return;   // the producer drains the copies in flight before the CTA ends
        }
        // the descriptor stays in shared memory for the whole item (its slot is
        // released at the item's end); only the chunk count lives in registers
        const volatile ItemDesc *dp = &cs.desc[q];
        if (dp->end) {
            if (owe) take_ticket();
            settle();
            return;
        }

        // the group's query rows as MMA B fragments: B = Q^T (k = dim, n = head)
        // Columns past the item's query rows get zeros, not what an earlier
        // item left in the slot: a thread's two columns share one rescale
        // decision, so stale values there could move a real column's
        // running maximum and with it the rounding of the result.
        uint32_t qb[NT][KS][2];
        {
            const __half *qs = reinterpret_cast<const __half *>(smem + c * C::DATA + DEPTH * C::STAGE + q * C::QSLOT);
            const int rows = dp->nmem * a.G;
#pragma unroll
            for (int t = 0; t < NT; ++t) {
                const bool live = t * 8 + r < rows;
#pragma unroll
                for (int k = 0; k < KS; ++k) {
                    if constexpr (C::FP8) {
                        // the K fragments of an fp8 tile come in the order
                        // ldmatrix gives bytes (see below): k-step k of the
                        // pair u = k / 2 uses dims 32u + 16 (k % 2) + 4 cq .. + 3
                        const __half *row = qs + (t * 8 + r) * D + 16 * k + 4 * cq;
                        const uint2 v = *reinterpret_cast<const uint2 *>(row);
                        qb[t][k][0] = live ? v.x : 0u;
                        qb[t][k][1] = live ? v.y : 0u;
                    } else {
                        const __half *row = qs + (t * 8 + r) * D + 16 * k + 2 * cq;
                        qb[t][k][0] = live ? *reinterpret_cast<const uint32_t *>(row) : 0u;
                        qb[t][k][1] = live ? *reinterpret_cast<const uint32_t *>(row + 8) : 0u;
                    }
                }
            }
        }
        const int nchunks = dp->nchunks;
        // the second head tile holds query rows 8 .. 15; an item with at most
        // 8 rows (a private range at G <= 8, one decode row of a multi-token
        // call) skips its MMAs and softmax (warp-uniform; no bit changes)
        const bool tile1 = NT == 2 && dp->nmem * a.G > 8;
        // CAUSAL: tokens of the item (from its start) that each column's query
        // row sees -- at least one, as every member sees the item's first token
        int lim[NT][2];
        if constexpr (CAUSAL) {
            const int len = (nchunks - 1) * CHUNK + dp->ntok_last;
            const int v0 = dp->seq0, rows = dp->nmem * a.G, it0 = dp->t0;
#pragma unroll
            for (int t = 0; t < NT; ++t)
#pragma unroll
                for (int e = 0; e < 2; ++e) {
                    const int row = t * 8 + 2 * cq + e;
                    lim[t][e] = row < rows ? min(len, __ldg(&a.context_lens[v0 + row / a.G]) - it0) : len;
                }
        }

        // running state per head column (2 * cq, 2 * cq + 1) of each head tile
        float m[NT][2], l[NT][2];
        float acc[MT][NT][4];
#pragma unroll
        for (int t = 0; t < NT; ++t) {
            m[t][0] = m[t][1] = -INFINITY;
            l[t][0] = l[t][1] = 0.f;
#pragma unroll
            for (int i = 0; i < MT; ++i) acc[i][t][0] = acc[i][t][1] = acc[i][t][2] = acc[i][t][3] = 0.f;
        }

        for (int ch = 0; ch < nchunks; ++ch) {
            if (ch > 0) {
                s = stage % DEPTH;
                if (!__all_sync(0xffffffffu,
                                mbar_wait_bounded(smem_u32(&cs.full[s]), (stage / DEPTH) & 1, a.wait_limit))) {
                    if (lane == 0) atomicExch(&a.hdr->error, PA_ERR_TIMEOUT);
                    return;   // the producer drains the copies in flight before the CTA ends
                }
            }
            const uint32_t kt = cs.data + s * C::STAGE;
            const uint32_t vt = kt + C::TILE;
            const int ntok = ch == nchunks - 1 ? dp->ntok_last : CHUNK;

            // S^T (16 tokens x 8 heads per head tile): two accumulation chains
            float sa[NT][4], sb[NT][4];
#pragma unroll
            for (int t = 0; t < NT; ++t)
#pragma unroll
                for (int e = 0; e < 4; ++e) sa[t][e] = sb[t][e] = 0.f;
            if constexpr (C::FP8) {
                // one ldmatrix gives 16 tokens x 32 codes: per thread, row r and
                // r + 8, bytes 4 cq .. 4 cq + 3 of two 16-byte chunks; each pair
                // of codes becomes one fp16x2 A entry (k-steps 2u and 2u + 1)
#pragma unroll
                for (int u = 0; u < KS / 2; ++u) {
                    uint32_t r0, r1, r2, r3;
                    ldmatrix_x4(kt + koff[u], r0, r1, r2, r3);
                    uint32_t af[2][4];
                    af[0][0] = e4m3x2_lo_to_f16x2(r0);
                    af[0][2] = e4m3x2_hi_to_f16x2(r0);
                    af[0][1] = e4m3x2_lo_to_f16x2(r1);
                    af[0][3] = e4m3x2_hi_to_f16x2(r1);
                    af[1][0] = e4m3x2_lo_to_f16x2(r2);
                    af[1][2] = e4m3x2_hi_to_f16x2(r2);
                    af[1][1] = e4m3x2_lo_to_f16x2(r3);
                    af[1][3] = e4m3x2_hi_to_f16x2(r3);
#pragma unroll
                    for (int h = 0; h < 2; ++h)
#pragma unroll
                        for (int t = 0; t < NT; ++t) {
                            if (t == 1 && !tile1) continue;
                            float *acc_s = h ? sb[t] : sa[t];
                            mma_16816(acc_s[0], acc_s[1], acc_s[2], acc_s[3], af[h][0], af[h][1], af[h][2], af[h][3],
                                      qb[t][2 * u + h][0], qb[t][2 * u + h][1], acc_s[0], acc_s[1], acc_s[2], acc_s[3]);
                        }
                }
            } else {
#pragma unroll
                for (int k = 0; k < KS; ++k) {
                    uint32_t a0, a1, a2, a3;
                    ldmatrix_x4(kt + (k >> 2) * (C::BOXES > 1 ? CHUNK * 128 : 0) + koff[k & 3], a0, a1, a2, a3);
#pragma unroll
                    for (int t = 0; t < NT; ++t) {
                        if (t == 1 && !tile1) continue;
                        float *acc_s = (k & 1) ? sb[t] : sa[t];
                        mma_kv<KV>(acc_s[0], acc_s[1], acc_s[2], acc_s[3], a0, a1, a2, a3, qb[t][k][0], qb[t][k][1]);
                    }
                }
            }
            // V^T fragments, loaded ahead of the softmax
            uint32_t va[MT][4];
            if constexpr (C::FP8 && PA_FP8_LATE_V) {
                // converted just before their MMAs (below)
            } else if constexpr (C::FP8) {
                // transposed 8 x 8 loads of 16-bit pairs: per thread, tokens
                // 2 cq and 2 cq + 1, dims 2 r and 2 r + 1 of a 16-byte chunk; the
                // byte permutation regroups them by dim, so m-tile i holds
                // dims 16 i + 2 r (rows r) and 16 i + 2 r + 1 (rows r + 8)
#pragma unroll
                for (int u = 0; u < MT / 2; ++u) {
                    uint32_t r4[4];
                    ldmatrix_x4_trans(vt + koff[u], r4[0], r4[1], r4[2], r4[3]);
#pragma unroll
                    for (int h = 0; h < 2; ++h) {
                        const uint32_t lo = __byte_perm(r4[2 * h], 0, 0x3120);       // tokens 2cq, 2cq+1
                        const uint32_t hi = __byte_perm(r4[2 * h + 1], 0, 0x3120);   // tokens 2cq+8, 2cq+9
                        va[2 * u + h][0] = e4m3x2_lo_to_f16x2(lo);
                        va[2 * u + h][1] = e4m3x2_hi_to_f16x2(lo);
                        va[2 * u + h][2] = e4m3x2_lo_to_f16x2(hi);
                        va[2 * u + h][3] = e4m3x2_hi_to_f16x2(hi);
                    }
                }
            } else {
#pragma unroll
                for (int i = 0; i < MT; ++i)
                    ldmatrix_x4_trans(vt + (i >> 2) * (C::BOXES > 1 ? CHUNK * 128 : 0) + voff[i & 3], va[i][0],
                                      va[i][1], va[i][2], va[i][3]);
            }

            // softmax per head column; thread holds tokens r, r + 8
            const bool tail = ntok < CHUNK;
            const bool tok_lo = r < ntok, tok_hi = r + 8 < ntok;
            uint32_t pb[NT][2];
#pragma unroll
            for (int t = 0; t < NT; ++t) {
                if (t == 1 && !tile1) {
                    pb[t][0] = pb[t][1] = 0u;
                    continue;
                }
                float s0 = sa[t][0] + sb[t][0], s1 = sa[t][1] + sb[t][1];   // token r, heads 2cq, 2cq+1
                float s2 = sa[t][2] + sb[t][2], s3 = sa[t][3] + sb[t][3];   // token r + 8
                if constexpr (CAUSAL) {
                    const int tk = ch * CHUNK + r;
                    s0 = tk < lim[t][0] ? s0 : -INFINITY;
                    s1 = tk < lim[t][1] ? s1 : -INFINITY;
                    s2 = tk + 8 < lim[t][0] ? s2 : -INFINITY;
                    s3 = tk + 8 < lim[t][1] ? s3 : -INFINITY;
                } else if (tail) {
                    s0 = tok_lo ? s0 : -INFINITY;
                    s1 = tok_lo ? s1 : -INFINITY;
                    s2 = tok_hi ? s2 : -INFINITY;
                    s3 = tok_hi ? s3 : -INFINITY;
                }
                float mx0 = fmaxf(s0, s2), mx1 = fmaxf(s1, s3);
#pragma unroll
                for (int o = 4; o < 32; o <<= 1) {
                    mx0 = fmaxf(mx0, __shfl_xor_sync(0xffffffffu, mx0, o));
                    mx1 = fmaxf(mx1, __shfl_xor_sync(0xffffffffu, mx1, o));
                }
                mx0 *= sl2;
                mx1 *= sl2;
                // keep a stale maximum until a score exceeds it by 2^8; then rescale
                if (mx0 > m[t][0] + RESCALE_THRESHOLD || mx1 > m[t][1] + RESCALE_THRESHOLD) {
                    const float n0 = fmaxf(m[t][0], mx0), n1 = fmaxf(m[t][1], mx1);
                    const float al0 = fast_exp2(m[t][0] - n0), al1 = fast_exp2(m[t][1] - n1);
                    m[t][0] = n0;
                    m[t][1] = n1;
                    l[t][0] *= al0;
                    l[t][1] *= al1;
#pragma unroll
                    for (int i = 0; i < MT; ++i) {
                        acc[i][t][0] *= al0;
                        acc[i][t][1] *= al1;
                        acc[i][t][2] *= al0;
                        acc[i][t][3] *= al1;
                    }
                }
                const float p0 = fast_exp2(fmaf(s0, sl2, -m[t][0])), p1 = fast_exp2(fmaf(s1, sl2, -m[t][1]));
                const float p2 = fast_exp2(fmaf(s2, sl2, -m[t][0])), p3 = fast_exp2(fmaf(s3, sl2, -m[t][1]));
                l[t][0] += p0 + p2;
                l[t][1] += p1 + p3;
                // P^T rows (tokens r, r+8) -> B operand of P V (k = token, n = head) by transposition
                pb[t][0] = movmatrix_trans(pack_p<KV>(p0, p1));
                pb[t][1] = movmatrix_trans(pack_p<KV>(p2, p3));
            }
            const uint32_t vlo = (2 * cq < ntok ? 0x0000ffffu : 0u) | (2 * cq + 1 < ntok ? 0xffff0000u : 0u);
            const uint32_t vhi = (2 * cq + 8 < ntok ? 0x0000ffffu : 0u) | (2 * cq + 9 < ntok ? 0xffff0000u : 0u);
            if constexpr (C::FP8 && PA_FP8_LATE_V) {
                // V^T fragments of an fp8 tile (layout as in the early path),
                // converted just before their MMAs to keep few registers live
#pragma unroll
                for (int u = 0; u < MT / 2; ++u) {
                    uint32_t r4[4];
                    ldmatrix_x4_trans(vt + koff[u], r4[0], r4[1], r4[2], r4[3]);
#pragma unroll
                    for (int h = 0; h < 2; ++h) {
                        const uint32_t lo = __byte_perm(r4[2 * h], 0, 0x3120);
                        const uint32_t hi = __byte_perm(r4[2 * h + 1], 0, 0x3120);
                        uint32_t f[4] = {e4m3x2_lo_to_f16x2(lo), e4m3x2_hi_to_f16x2(lo), e4m3x2_lo_to_f16x2(hi),
                                         e4m3x2_hi_to_f16x2(hi)};
                        if (tail) {
                            f[0] &= vlo;
                            f[1] &= vlo;
                            f[2] &= vhi;
                            f[3] &= vhi;
                        }
#pragma unroll
                        for (int t = 0; t < NT; ++t)
                            if (t == 0 || tile1)
                            mma_kv<KV>(acc[2 * u + h][t][0], acc[2 * u + h][t][1], acc[2 * u + h][t][2],
                                       acc[2 * u + h][t][3], f[0], f[1], f[2], f[3], pb[t][0], pb[t][1]);
                    }
                }
            } else {
                if (tail) {   // stale or poisoned slots past the context must not reach O
#pragma unroll
                    for (int i = 0; i < MT; ++i) {
                        va[i][0] &= vlo;
                        va[i][1] &= vlo;
                        va[i][2] &= vhi;
                        va[i][3] &= vhi;
                    }
                }
                // O^T += V^T P^T
#pragma unroll
                for (int i = 0; i < MT; ++i)
#pragma unroll
                    for (int t = 0; t < NT; ++t)
                        if (t == 0 || tile1)
                            mma_kv<KV>(acc[i][t][0], acc[i][t][1], acc[i][t][2], acc[i][t][3], va[i][0], va[i][1],
                                       va[i][2], va[i][3], pb[t][0], pb[t][1]);
            }
            __syncwarp();
            if (lane == 0) mbar_arrive(smem_u32(&cs.empty[s]));   // stage free for the next copy
            ++stage;
            if (ch == 0 && owe) take_ticket();
        }

        // ---- item complete: row sums over the 8 token lanes, then write out
#pragma unroll
        for (int t = 0; t < NT; ++t)
#pragma unroll
            for (int e = 0; e < 2; ++e) {
                float v = l[t][e];
                v += __shfl_xor_sync(0xffffffffu, v, 4);
                v += __shfl_xor_sync(0xffffffffu, v, 8);
                v += __shfl_xor_sync(0xffffffffu, v, 16);
                l[t][e] = v;
            }
        const float qnan = __int_as_float(0x7fc00000);
        const ItemDesc dsc = *const_cast<const ItemDesc *>(dp);
        __syncwarp();
        if (lane == 0) mbar_arrive(smem_u32(&cs.qfree[q]));   // query slot and descriptor free again
        // per query row: member m = row / G of the item, head g = row % G;
        // P and the partial's row are the member's own
#pragma unroll
        for (int t = 0; t < NT; ++t)
#pragma unroll
            for (int e = 0; e < 2; ++e) {
                const int row = t * 8 + 2 * cq + e;
                if (row < dsc.nmem * a.G) {
                    const int mbr = row / a.G, g = row - mbr * a.G;
                    const int seq = dsc.seq0 + mbr;
                    int P = dsc.P0, canon = dsc.canon0;
                    if (dsc.canon0 < 0) {   // a shared-prefix item: every member has its own P and row
                        P = partitions_of(__ldg(&a.context_lens[seq]), dsc.shared, a.pt, a.pts);
                        canon = __ldg(&a.part_off[seq]) + dsc.pidx;
                    }
                    const int h = dsc.kvh * a.G + g;
                    // output dims of this thread's accumulator rows r and r + 8
                    // of m-tile i: 16 i + r and 16 i + r + 8, or for an fp8
                    // cache 16 i + 2 r and 16 i + 2 r + 1 (see the V loads)
                    constexpr int DSTEP = C::FP8 ? 1 : 8;
                    const int d0 = C::FP8 ? 2 * r : r;
                    const float vs = C::FP8 ? a.v_scale : 1.f;
                    if (P == 1) {
                        const float inv = dsc.bad ? qnan : vs / l[t][e];
                        uint16_t *orow = a.out + ((long long)seq * a.Hq + h) * D;
#pragma unroll
                        for (int i = 0; i < MT; ++i) {
                            orow[16 * i + d0] = out_bits<KV>(acc[i][t][e] * inv);
                            orow[16 * i + d0 + DSTEP] = out_bits<KV>(acc[i][t][e + 2] * inv);
                        }
                    } else {
                        const long long wrow = (long long)canon * a.Hq + h;
                        float *orow = a.ws_o + wrow * D;
#pragma unroll
                        for (int i = 0; i < MT; ++i) {
                            orow[16 * i + d0] = dsc.bad ? qnan : acc[i][t][e] * vs;
                            orow[16 * i + d0 + DSTEP] = dsc.bad ? qnan : acc[i][t][e + 2] * vs;
                        }
                        if (r == 0)
                            a.ws_ml[wrow] = dsc.bad ? make_float2(qnan, qnan) : make_float2(m[t][e], l[t][e]);
                    }
                }
            }
        // the tickets taken during this item: merge the groups they completed
        settle();
        if (lane < dsc.nmem) {   // tickets owed for this item's members
            owe_seq = dsc.seq0 + lane;
            owe_kvh = dsc.kvh;
            const int Lm = __ldg(&a.context_lens[owe_seq]);
            owe_P = dsc.canon0 < 0 ? partitions_of(Lm, dsc.shared, a.pt, a.pts) : dsc.P0;
            owe_T = a.tc_shared ? (Lm - dsc.shared + a.pt - 1) / a.pt : owe_P;
        }
        owe = __any_sync(0xffffffffu, owe_P > 1);
    }
}

template <int D, int NT, bool CAUSAL, int KV>
__global__ void __launch_bounds__(Cfg<D, NT, KV>::WARPS * 32, Cfg<D, NT, KV>::MINB)
    decode_kernel(const __grid_constant__ CUtensorMap tmk, const __grid_constant__ CUtensorMap tmv, const DecodeArgs a) {
    using C = Cfg<D, NT, KV>;
    extern __shared__ uint8_t smem_raw[];
    uint8_t *smem = reinterpret_cast<uint8_t *>((reinterpret_cast<uintptr_t>(smem_raw) + 1023) & ~uintptr_t(1023));
    const int warp = threadIdx.x >> 5;
    if (threadIdx.x == 0) {
        for (int c = 0; c < C::NCON; ++c) {
            const ConsumerSmem cs = consumer_smem<D, NT, KV>(smem, c);
            for (int s = 0; s < Cfg<D, NT, KV>::DEPTH; ++s) {
                mbar_init(smem_u32(&cs.full[s]), 1);
                mbar_init(smem_u32(&cs.empty[s]), 1);
            }
            mbar_init(smem_u32(&cs.qfree[0]), 1);
            mbar_init(smem_u32(&cs.qfree[1]), 1);
        }
        fence_mbar_init();
    }
    __syncthreads();
    if constexpr (C::SPLIT) {   // warpgroup 0: producers, warpgroup 1: their consumers
        if (warp < 4) {
            regs_decrease<C::PROD_REGS>();
            producer<D, NT, CAUSAL, KV>(smem, &tmk, &tmv, a, warp);
        } else {
            regs_increase<C::CONS_REGS>();
            consumer<D, NT, CAUSAL, KV>(smem, warp - 4, a);
        }
    } else {
        if (warp == 0)
            producer<D, NT, CAUSAL, KV>(smem, &tmk, &tmv, a, 0);
        else
            consumer<D, NT, CAUSAL, KV>(smem, warp - 1, a);
    }
}

template <int D, int NT, bool CAUSAL, int KV>
int launch_decode(const CUtensorMap &tmk, const CUtensorMap &tmv, const DecodeArgs &args, long long max_items,
                  cudaStream_t st) {
    using C = Cfg<D, NT, KV>;
    static int grid = 0;
    static bool usable = false;
    static std::once_flag once;
    static cudaError_t init_err = cudaSuccess;
    std::call_once(once, [] {
        init_err =
            cudaFuncSetAttribute(decode_kernel<D, NT, CAUSAL, KV>, cudaFuncAttributeMaxDynamicSharedMemorySize, C::SMEM);
        if (init_err != cudaSuccess) return;
        int dev = 0, sms = 0, per_sm = 0;
        cudaFuncAttributes fa;
        init_err = cudaGetDevice(&dev);
        if (init_err == cudaSuccess) init_err = cudaDeviceGetAttribute(&sms, cudaDevAttrMultiProcessorCount, dev);
        if (init_err == cudaSuccess)
            init_err = cudaOccupancyMaxActiveBlocksPerMultiprocessor(&per_sm, decode_kernel<D, NT, CAUSAL, KV>,
                                                                     C::WARPS * 32, C::SMEM);
        if (init_err == cudaSuccess) init_err = cudaFuncGetAttributes(&fa, decode_kernel<D, NT, CAUSAL, KV>);
        if (init_err == cudaSuccess) grid = sms * (per_sm > 0 ? per_sm : 1);
        // a register split is only run with the launch count it was sized for
        // (a larger split than the pool would make the consumers' increase
        // wait forever)
        usable = init_err == cudaSuccess && (!C::SPLIT || fa.numRegs == C::LAUNCH_REGS);
    });
    if (init_err != cudaSuccess || grid <= 0) return PA_ERR_CUDA;
    if (!usable) return PA_ERR_UNSUPPORTED;
    // no more CTAs than there can be items for their consumers
    const long long need = (max_items + C::NCON - 1) / C::NCON;
    const int g = (int)(need < grid ? (need > 0 ? need : 1) : grid);
    decode_kernel<D, NT, CAUSAL, KV><<<g, C::WARPS * 32, C::SMEM, st>>>(tmk, tmv, args);
    return cuda_status(cudaGetLastError());
}

}  // namespace

// One launch of the decode kernel for the cache element type of the
// translation unit that defines it (D, NT and CAUSAL picked at run time).
int launch_kv_f16(int D, int NT, bool causal, const CUtensorMap &tmk, const CUtensorMap &tmv,
                  const DecodeArgs &args, long long max_items, cudaStream_t st);
int launch_kv_bf16(int D, int NT, bool causal, const CUtensorMap &tmk, const CUtensorMap &tmv,
                   const DecodeArgs &args, long long max_items, cudaStream_t st);
int launch_kv_fp8(int D, int NT, bool causal, const CUtensorMap &tmk, const CUtensorMap &tmv,
                  const DecodeArgs &args, long long max_items, cudaStream_t st);

// The launch for one cache element type: D in {64, 128} (128 only for fp8),
// NT in {1, 2}; the multi-token form runs with PA_CAUSAL_NT head tiles.
template <int KV>
int launch_kv(int D, int NT, bool causal, const CUtensorMap &tmk, const CUtensorMap &tmv, const DecodeArgs &args,
              long long max_items, cudaStream_t st) {
    if (causal) {
        if (NT != PA_CAUSAL_NT) return PA_ERR_UNSUPPORTED;
        if (D == 128) return launch_decode<128, PA_CAUSAL_NT, true, KV>(tmk, tmv, args, max_items, st);
        if constexpr (KV != PA_KV_FP8_E4M3) return launch_decode<64, PA_CAUSAL_NT, true, KV>(tmk, tmv, args, max_items, st);
        return PA_ERR_UNSUPPORTED;
    }
    if (D == 128)
        return NT == 1 ? launch_decode<128, 1, false, KV>(tmk, tmv, args, max_items, st)
                       : launch_decode<128, 2, false, KV>(tmk, tmv, args, max_items, st);
    if constexpr (KV != PA_KV_FP8_E4M3)
        return NT == 1 ? launch_decode<64, 1, false, KV>(tmk, tmv, args, max_items, st)
                       : launch_decode<64, 2, false, KV>(tmk, tmv, args, max_items, st);
    return PA_ERR_UNSUPPORTED;
}

}  // namespace pa
