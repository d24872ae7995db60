// Paged single-token decode attention for sm_103a.
//
// What is computed: for sequence i, query head h and kv head g = h / G,
//   out[i][h] = sum_t softmax_t(scale * <q[i][h], K_t[g]>) * V_t[g],   t < L_i,
// where token t is gathered from physical block block_tables[i][t / bs] at
// offset t % bs.  The block table and the gather through it are section 2.2
// of "PagedAttention de vLLM : comment la gestion de la VRAM soutient
// l'inference des grands modeles" (deepsonar.com.cn) and section "La table de
// blocs en arriere-plan" of "PagedAttention : comment optimiser la memoire GPU
// lors de l'inference des LLM" (deeplearn.tn); GQA sharing (G consecutive
// query heads per kv head) is section 2.1 of the deepsonar page; the
// incremental, tile-by-tile softmax is section "PagedAttention vs.
// FlashAttention" of the deeplearn.tn page.
//
// How (two launches on the caller's stream):
//  1. decode_prep_kernel (one CTA): splits every sequence into partitions of
//     PT tokens (PT = 256, 512 or 1024, chosen from the shapes), writes the compact list of (sequence, partition)
//     work items into the workspace, zeroes the work and merge counters, and
//     writes the rows of empty (zero) and invalid (NaN) sequences.
//  2. decode_kernel (persistent, warp-specialised).  In every CTA one
//     producer warp takes work items (sequence, partition, kv head) from an
//     atomic counter on behalf of NC consumer warps and streams each item's
//     16-token chunks of K and V into that consumer's ring of DEPTH shared
//     memory stages with TMA: 2-D tiled copies through a tensor map over the
//     cache with a 128-byte swizzle, the gather being the TMA row coordinate
//     read from the block table.  Full/empty mbarriers pace the rings.
//     A consumer warp reduces one item at a time with m16n8k16 tensor-core
//     MMAs, tokens on M and the G query heads of the kv head on N:
//     S^T = K Q^T, an online softmax per head in fp32 (rescaling the running
//     sums only when the maximum grows by more than 2^8), then
//     O^T += V^T P^T, P^T moved into operand layout with movmatrix.  Each KV
//     tile crosses HBM once for the whole group.  A single-partition sequence
//     writes its fp16 output directly.  Otherwise the item stores (m, l,
//     unnormalised o) in the workspace and takes a ticket; the item that
//     completes its (sequence, kv head) group merges the group's partitions
//     by the log-sum-exp rule
//       M = max_p m_p,  w_p = 2^(m_p - M),  out = sum_p w_p o_p / sum_p w_p l_p.
//
// Results do not depend on the physical placement, on the block size or on
// which warp ran which item: every item is reduced by one warp in a fixed
// chunk order, and the merge runs over partitions in order.

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
#ifndef PA_DECODE_MINB_WIDE
#define PA_DECODE_MINB_WIDE 4
#endif
#ifndef PA_DECODE_DEPTH_WIDE
#define PA_DECODE_DEPTH_WIDE 5
#endif
#ifndef PA_DECODE_MINB
#define PA_DECODE_MINB 8
#endif
#ifndef PA_CAUSAL_L2
#define PA_CAUSAL_L2 0
#endif
#ifndef PA_CAUSAL_NT
#define PA_CAUSAL_NT 2
#endif

namespace pa {
namespace {

constexpr int MAX_PART_TOKENS = 1024;           // largest partition (one work item)
constexpr long long TARGET_ITEMS = 4096;        // work items wanted for load balance
constexpr int CHUNK = 16;                       // tokens per pipeline stage (one MMA K step of P V)
constexpr int NC = PA_DECODE_CONSUMERS;         // consumer warps per CTA
constexpr int NWARPS = NC + 1;                  // + the producer warp
constexpr long long WAIT_LIMIT = 1LL << 31;     // clock cycles (about a second): default wait bound, drain bound
constexpr int PREP_THREADS = 1024;
constexpr float RESCALE_THRESHOLD = 8.f;        // log2 units: rescale when the max grows by more than 2^8
constexpr int ENTRIES = MAX_PART_TOKENS / 8 / 32;   // block-table entries per lane for one item (block size >= 8)

// Partition size: the largest of 1024, 512, 256 tokens whose estimated item
// count (sequences x kv heads x partitions of the longest context) reaches
// TARGET_ITEMS, so that long batches get long, cheap items and short ones
// still spread over every SM.  It depends on the shapes only, so a given
// call always partitions the same way.
int part_tokens(int B, int Hkv, int max_ctx) {
    for (int pt = MAX_PART_TOKENS; pt > 256; pt /= 2)
        if ((long long)B * Hkv * ((max_ctx + pt - 1) / pt) >= TARGET_ITEMS) return pt;
    return 256;
}

struct WsHeader {
    int error;
    int total_items;
    int counter;
    int pad[61];
};
static_assert(sizeof(WsHeader) == 256, "header is one 256-byte line");

struct WsLayout {
    size_t part_off, gsize, gshared, items, grp, ml, o, total;
    int pmax, pt;
    long long item_cap;
};

inline size_t up256(size_t x) { return (x + 255) & ~size_t(255); }

// Workspace of one call.  grouped: sequences may share a prefix, which adds
// at most one partition per sequence and as many shared items again.
WsLayout ws_layout(int B, int Hq, int Hkv, int D, int max_ctx, bool grouped) {
    WsLayout w;
    w.pt = part_tokens(B, Hkv, max_ctx);
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
    w.total = off;
    return w;
}

// Workspace of one call of the multi-token (causal) form: NQ query rows of B
// sequences; per row its visible length and partial-row offset, per sequence
// the first of its member groups (ms consecutive rows read together), and a
// partial row per (query row, partition).
WsLayout ws_layout_causal(int B, int NQ, int Hq, int Hkv, int D, int max_ctx) {
    WsLayout w;
    const int G = Hq / Hkv;
    const int ms = 8 * PA_CAUSAL_NT / G > 1 ? 8 * PA_CAUSAL_NT / G : 1;
    w.pt = part_tokens(B, Hkv, max_ctx);
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
    __half *out;
    const __half *query;
    const int32_t *block_tables;
    const int32_t *context_lens;
    int Hq, Hkv, G, bs, mbps, pt, ms;
    long long num_blocks;
    long long wait_limit;   // bound of every pipeline wait, clock cycles
    float scale_log2;
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

template <int D, int NT>
struct Cfg {
    // pipeline stages per consumer: a two-tile consumer keeps fewer warps on
    // an SM (registers), so each keeps more bytes in flight
    static constexpr int DEPTH = NT == 1 ? PA_DECODE_DEPTH : PA_DECODE_DEPTH_WIDE;
    static constexpr int BOXES = D / 64;                   // 64-column (128-byte) boxes per tile row
    static constexpr int TILE = BOXES * CHUNK * 128;       // one 16-token K or V tile
    static constexpr int STAGE = 2 * TILE;                 // K tile then V tile
    static constexpr int QSLOT = NT * 8 * D * 2;           // the group's query rows
    static constexpr int DATA = DEPTH * STAGE + 2 * QSLOT; // per consumer, a multiple of 1024
    static constexpr int CTRL = 256;                       // per consumer: barriers and descriptors
    static constexpr int SMEM = NC * (DATA + CTRL) + 1024;
    static_assert(DATA % 1024 == 0, "stages must stay 1024-byte aligned for the 128-byte swizzle");
    static_assert((2 * DEPTH + 2) * 8 + 16 + 2 * 64 <= CTRL, "control block too small");
};

// Byte offset, inside a swizzled tile, of 16-byte column `col` (0 .. D/8-1)
// of row `row`: 64-column boxes of CHUNK rows x 128 bytes; chunk j of row r
// sits at position j ^ (r & 7) (the TMA 128-byte swizzle).
__host__ __device__ constexpr int swz(int row, int col) {
    return (col >> 3) * (CHUNK * 128) + row * 128 + (((col & 7) ^ (row & 7)) << 4);
}

// -------------------------------------------------------------- prep

// Block-wide exclusive scan of one int per thread (PREP_THREADS threads);
// returns the thread's exclusive prefix and writes the block total to *total.
__device__ __forceinline__ int block_exclusive_scan(int x, int *warp_sums, int *total) {
    const int lane = threadIdx.x & 31, wid = threadIdx.x >> 5;
    int inc = x;
#pragma unroll
    for (int o = 1; o < 32; o <<= 1) {
        const int y = __shfl_up_sync(0xffffffffu, inc, o);
        if (lane >= o) inc += y;
    }
    if (lane == 31) warp_sums[wid] = inc;
    __syncthreads();
    if (wid == 0) {
        int s = warp_sums[lane];
#pragma unroll
        for (int o = 1; o < 32; o <<= 1) {
            const int y = __shfl_up_sync(0xffffffffu, s, o);
            if (lane >= o) s += y;
        }
        warp_sums[lane] = s;
    }
    __syncthreads();
    const int excl = (wid ? warp_sums[wid - 1] : 0) + inc - x;
    *total = warp_sums[PREP_THREADS / 32 - 1];
    __syncthreads();
    return excl;
}

// Partitions of one sequence: its shared prefix [0, S) and its own range
// [S, L), each cut into pieces of pt tokens (S = 0 for a sequence that
// shares nothing).
__device__ __forceinline__ int partitions_of(int L, int S, int pt) {
    return (S + pt - 1) / pt + (L - S + pt - 1) / pt;
}

// Work list, longest first.  Items of full length (pt tokens) come first:
// shared-prefix items of every group, then each sequence's own partitions
// but its last, in sequence order; every sequence's last partition and the
// shorter shared items follow in decreasing length (a counting sort on
// 16-token buckets).  So the dynamically scheduled tail of the kernel runs
// the shortest items, and the merges, which follow a sequence's last
// partition, land mostly in that tail where consumers would idle anyway.  Partial results are
// stored at canonical rows part_off[seq] + partition, independent of the
// order.
//
// Groups (optional): sequence i names the leader of its group in lead[i];
// the group is the run of consecutive sequences from the leader that all name
// it, and shares the leader's shared_len[] tokens (rounded down to whole
// blocks, capped by every member's context).  A shared range is read once per
// item for up to ms members together.
__global__ void __launch_bounds__(PREP_THREADS) decode_prep_kernel(
    const int32_t *__restrict__ context_lens, const int32_t *__restrict__ lead,
    const int32_t *__restrict__ shared_len, int B, int Hq, int D, int Hkv, int bs, int max_ctx,
    long long max_table_tokens, int pt, int ms, WsHeader *hdr, int *part_off, int *gsize, int *gshared,
    ItemRec *items, int *grp, __half *out) {
    constexpr int NBK = MAX_PART_TOKENS / CHUNK;     // length buckets of the short items
    __shared__ int warp_sums[PREP_THREADS / 32];
    __shared__ int hist[NBK], cursor[NBK];
    int run_p = 0, run_f = 0;                        // uniform running totals
    for (int k = threadIdx.x; k < NBK; k += PREP_THREADS) hist[k] = cursor[k] = 0;
    if (grp)
        for (long long k = threadIdx.x; k < (long long)B * Hkv; k += PREP_THREADS) grp[k] = 0;
    auto valid_len = [&](int L) { return L >= 0 && L <= max_ctx && (long long)L <= max_table_tokens; };
    // pass 0: group sizes and shared lengths, at each leader
    if (lead)
        for (int i = threadIdx.x; i < B; i += PREP_THREADS) {
            int M = 0, S = 0;
            if (lead[i] == i) {
                S = shared_len[i] > 0 ? shared_len[i] / bs * bs : 0;
                bool ok = true;
                for (int j = i; j < B && lead[j] == i; ++j, ++M) {
                    const int L = context_lens[j];
                    ok = ok && valid_len(L) && L > 0;
                    S = min(S, ok ? L : 0);
                }
                S = S / bs * bs;   // whole blocks only, also after capping by a member's context
                if (!ok || M < 2) S = 0;
            }
            gsize[i] = M;
            gshared[i] = S;
        }
    __syncthreads();
    // the shared length of sequence i: its leader's, if i is in the leader's run
    auto shared_of = [&](int i, int &ld) -> int {
        ld = i;
        if (!lead) return 0;
        const int l = lead[i];
        if (l < 0 || l > i || i - l >= gsize[l] || gshared[l] == 0) return 0;
        ld = l;
        return gshared[l];
    };
    const int nbk = pt / CHUNK;
    // pass 1: partitions and canonical offsets; full-length items; histogram of the short ones
    for (int base = 0; base < B; base += PREP_THREADS) {
        const int i = base + threadIdx.x;
        int L = 0, P = 0, code = 0, S = 0, ld = i, nfull = 0;   // code 1: zero row, 2: NaN row
        int Ms = 0, Ps = 0;                                      // leader: members, shared partitions
        if (i < B) {
            L = context_lens[i];
            S = shared_of(i, ld);
            if (!valid_len(L))
                code = 2;
            else if (L == 0)
                code = 1;
            else
                P = partitions_of(L, S, pt);
            if (P > 0) {
                nfull = (L - S + pt - 1) / pt - 1;   // own partitions but the last
                if (ld == i && S > 0) {
                    Ms = gsize[i];
                    Ps = (S + pt - 1) / pt;
                    nfull += (S / pt) * ((Ms + ms - 1) / ms);
                }
            }
        }
        int tp, tf;
        const int ep = run_p + block_exclusive_scan(P, warp_sums, &tp);
        int ef = run_f + block_exclusive_scan(nfull, warp_sums, &tf);
        if (i < B) {
            part_off[i] = ep;
            if (P > 0) {
                const int ps_i = (S + pt - 1) / pt;
                if (Ps > 0) {   // leader: full shared items
                    for (int p = 0; p < S / pt; ++p)
                        for (int k = 0; k < Ms; k += ms) {
                            ItemRec r;
                            r.a = make_int4(i + k, min(ms, Ms - k), p * pt, (p + 1) * pt);
                            r.b = make_int4(p, S, L, -1);
                            items[ef++] = r;
                        }
                    if (S % pt) atomicAdd(&hist[(pt - S % pt) / CHUNK], (Ms + ms - 1) / ms);
                }
                const int pp = (L - S + pt - 1) / pt;      // own partitions
                for (int p = 0; p + 1 < pp; ++p) {         // all full but the last
                    ItemRec r;
                    r.a = make_int4(i, 1, S + p * pt, S + (p + 1) * pt);
                    r.b = make_int4(ps_i + p, S, L, ep + ps_i + p);
                    items[ef++] = r;
                }
                if (pp > 0) atomicAdd(&hist[(pt - (L - S - (pp - 1) * pt)) / CHUNK], 1);
            }
            if (code) {
                const uint32_t h = code == 1 ? 0u : 0x7e007e00u;
                uint4 fill = make_uint4(h, h, h, h);
                uint4 *row = reinterpret_cast<uint4 *>(out + (long long)i * Hq * D);
                for (int k = 0; k < Hq * D / 8; ++k) row[k] = fill;
            }
        }
        run_p += tp;
        run_f += tf;
    }
    __syncthreads();
    int total_items = run_f;
    if (threadIdx.x == 0) {
        int acc = run_f;
        for (int k = 0; k < nbk; ++k) {
            cursor[k] = acc;
            acc += hist[k];
        }
    }
    __syncthreads();
    // pass 2: short items, longest first
    for (int i = threadIdx.x; i < B; i += PREP_THREADS) {
        const int L = context_lens[i];
        if (L <= 0 || !valid_len(L)) continue;
        int ld;
        const int S = shared_of(i, ld);
        const int ps_i = (S + pt - 1) / pt;
        if (ld == i && S > 0 && S % pt) {
            const int Ms = gsize[i];
            for (int k = 0; k < Ms; k += ms) {
                ItemRec r;
                r.a = make_int4(i + k, min(ms, Ms - k), S / pt * pt, S);
                r.b = make_int4(ps_i - 1, S, L, -1);
                items[atomicAdd(&cursor[(pt - S % pt) / CHUNK], 1)] = r;
            }
        }
        const int pp = (L - S + pt - 1) / pt;
        if (pp > 0) {
            const int p = pp - 1;
            ItemRec r;
            r.a = make_int4(i, 1, S + p * pt, L);
            r.b = make_int4(ps_i + p, S, L, part_off[i] + ps_i + p);
            items[atomicAdd(&cursor[(pt - (L - S - p * pt)) / CHUNK], 1)] = r;
        }
    }
    __syncthreads();
    if (threadIdx.x == 0) {
        total_items = cursor[nbk - 1];
        part_off[B] = run_p;
        hdr->total_items = total_items * Hkv;
        hdr->counter = 0;
        hdr->error = 0;
    }
}

// Index of the last entry of the non-decreasing array a[0 .. n] that is <= x
// (a[0] <= x < a[n]): the sequence a query row or member group belongs to.
__device__ __forceinline__ int last_le(const int32_t *a, int n, int x) {
    int lo = 0, hi = n;
    while (hi - lo > 1) {
        const int mid = (lo + hi) >> 1;
        if (a[mid] <= x)   // plain load: the group offsets are written by the same kernel
            lo = mid;
        else
            hi = mid;
    }
    return lo;
}

// Work list of the multi-token form.  Sequence i computes T_i new tokens in
// one step (a chunk of its prompt, or speculative tokens: "PagedAttention de
// vLLM", section 2.5); they are the last T_i of its L_i positions and are
// query rows query_start[i] + j, row j seeing positions [0, L_i - T_i + j].
// Rows are cut into member groups of ms consecutive rows of one sequence; a
// group's items are the partitions [p pt, (p + 1) pt) of the range its last
// member sees, each for the group's members that see the partition's first
// token (so every member of an item sees at least one of its tokens).  A row
// sees ceil(vis / pt) partitions, stored at part_off[row] + p.  Items of full
// length first, every group's last item after them by decreasing length, as
// in the single-token form.  A sequence whose lengths are inconsistent gets
// NaN rows; a query_start that is not a non-decreasing cover of [0, NQ) makes
// every row NaN.
__global__ void __launch_bounds__(PREP_THREADS) causal_prep_kernel(
    const int32_t *__restrict__ context_lens, const int32_t *__restrict__ qs, int B, int NQ, int Hq, int D, int Hkv,
    int max_ctx, long long max_table_tokens, int pt, int ms, WsHeader *hdr, int *part_off, int *vlen, int *gstart,
    ItemRec *items, int *grp, __half *out) {
    constexpr int NBK = MAX_PART_TOKENS / CHUNK;
    __shared__ int warp_sums[PREP_THREADS / 32];
    __shared__ int hist[NBK], cursor[NBK];
    for (int k = threadIdx.x; k < NBK; k += PREP_THREADS) hist[k] = cursor[k] = 0;
    for (long long k = threadIdx.x; k < (long long)NQ * Hkv; k += PREP_THREADS) grp[k] = 0;
    bool ok = true;
    for (int i = threadIdx.x; i <= B; i += PREP_THREADS) {
        const int x = qs[i];
        ok = ok && (i > 0 || x == 0) && (i < B || x == NQ) && (i == B || x <= qs[i + 1]);
    }
    const bool qs_ok = __syncthreads_and(ok) != 0;
    auto seq_ok = [&](int i, int &L, int &T) {
        L = context_lens[i];
        T = qs[i + 1] - qs[i];
        return L >= 0 && L <= max_ctx && (long long)L <= max_table_tokens && T <= L;
    };
    // pass 1: visible length and partial-row offset of every query row
    int run = 0;
    for (int base = 0; base < NQ; base += PREP_THREADS) {
        const int v = base + threadIdx.x;
        int vl = -1;
        if (v < NQ && qs_ok) {
            const int i = last_le(qs, B, v);
            int L, T;
            if (seq_ok(i, L, T)) vl = L - T + (v - qs[i]) + 1;
        }
        int tot;
        const int e = run + block_exclusive_scan(vl > 0 ? (vl + pt - 1) / pt : 0, warp_sums, &tot);
        if (v < NQ) {
            vlen[v] = vl;
            part_off[v] = e;
            if (vl < 0) {
                uint4 fill = make_uint4(0x7e007e00u, 0x7e007e00u, 0x7e007e00u, 0x7e007e00u);
                uint4 *row = reinterpret_cast<uint4 *>(out + (long long)v * Hq * D);
                for (int k = 0; k < Hq * D / 8; ++k) row[k] = fill;
            }
        }
        run += tot;
    }
    // pass 2: member groups per sequence
    int run_g = 0;
    for (int base = 0; base < B; base += PREP_THREADS) {
        const int i = base + threadIdx.x;
        int n = 0, L, T;
        if (i < B && qs_ok && seq_ok(i, L, T)) n = (T + ms - 1) / ms;
        int tot;
        const int e = run_g + block_exclusive_scan(n, warp_sums, &tot);
        if (i < B) gstart[i] = e;
        run_g += tot;
    }
    if (threadIdx.x == 0) {
        gstart[B] = run_g;
        part_off[NQ] = run;
    }
    __syncthreads();
    const int NG = run_g;
    // group g: rows [r0 + jl, r0 + jh) of sequence i; C = L - T + 1 positions
    // seen by its first new token; the last member sees vis positions
    auto group = [&](int g, int &r0, int &jl, int &jh, int &C, int &vis, int &np, int &i) {
        i = last_le(gstart, B, g);
        const int L = context_lens[i];
        r0 = qs[i];
        const int T = qs[i + 1] - r0;
        jl = (g - gstart[i]) * ms;
        jh = min(jl + ms, T);
        C = L - T + 1;
        vis = C + jh - 1;
        np = (vis + pt - 1) / pt;
    };
    // pass 3: full-length items, and a histogram of every group's last item
    int run_f = 0;
    for (int base = 0; base < NG; base += PREP_THREADS) {
        const int g = base + threadIdx.x;
        int r0 = 0, jl = 0, jh = 0, C = 0, vis = 0, np = 0, i = 0;
        if (g < NG) group(g, r0, jl, jh, C, vis, np, i);
        int tot;
        int ef = run_f + block_exclusive_scan(g < NG ? np - 1 : 0, warp_sums, &tot);
        if (g < NG) {
            for (int p = 0; p + 1 < np; ++p) {
                const int t0 = p * pt, j0 = max(jl, t0 - C + 1);
                ItemRec r;
                r.a = make_int4(r0 + j0, jh - j0, t0, t0 + pt);
                r.b = make_int4(p, 0, i, -1);
                items[ef++] = r;
            }
            atomicAdd(&hist[(pt - (vis - (np - 1) * pt)) / CHUNK], 1);
        }
        run_f += tot;
    }
    __syncthreads();
    if (threadIdx.x == 0) {
        int acc = run_f;
        for (int k = 0; k < pt / CHUNK; ++k) {
            cursor[k] = acc;
            acc += hist[k];
        }
    }
    __syncthreads();
    // pass 4: every group's last item, longest first
    for (int g = threadIdx.x; g < NG; g += PREP_THREADS) {
        int r0, jl, jh, C, vis, np, i;
        group(g, r0, jl, jh, C, vis, np, i);
        const int p = np - 1, t0 = p * pt, j0 = max(jl, t0 - C + 1);
        ItemRec r;
        r.a = make_int4(r0 + j0, jh - j0, t0, vis);
        r.b = make_int4(p, 0, i, -1);
        items[atomicAdd(&cursor[(pt - (vis - t0)) / CHUNK], 1)] = r;
    }
    __syncthreads();
    if (threadIdx.x == 0) {
        hdr->total_items = cursor[pt / CHUNK - 1] * Hkv;
        hdr->counter = 0;
        hdr->error = 0;
    }
}

// ------------------------------------------------------------ decode

struct ConsumerSmem {
    uint32_t data;        // shared address of the consumer's stages and query slots
    uint64_t *full;       // [DEPTH]: stage loaded (producer arrive + TMA bytes)
    uint64_t *empty;      // [DEPTH]: stage consumed (consumer arrive)
    uint64_t *qfree;      // [2]: query slot / descriptor free again
    ItemDesc *desc;       // [2]
};

template <int D, int NT>
__device__ __forceinline__ ConsumerSmem consumer_smem(uint8_t *smem, int c) {
    using C = Cfg<D, NT>;
    constexpr int DEPTH = C::DEPTH;
    uint8_t *ctrl = smem + NC * C::DATA + c * C::CTRL;
    ConsumerSmem s;
    s.data = smem_u32(smem + c * C::DATA);
    s.full = reinterpret_cast<uint64_t *>(ctrl);
    s.empty = s.full + DEPTH;
    s.qfree = s.empty + DEPTH;
    s.desc = reinterpret_cast<ItemDesc *>(ctrl + (2 * DEPTH + 2) * 8 + 16);
    return s;
}

// Producer warp: hands items to the consumers round-robin and keeps their
// rings full.  All lanes run the loop; lane 0 issues the copies.
template <int D, int NT, bool CAUSAL>
__device__ void producer(uint8_t *smem, const CUtensorMap *tmk, const CUtensorMap *tmv, const DecodeArgs &a) {
    using C = Cfg<D, NT>;
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
            const ConsumerSmem cs = consumer_smem<D, NT>(smem, c);
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
            const ConsumerSmem cs = consumer_smem<D, NT>(smem, c);
            const int s = sc[c] % DEPTH;
            const uint32_t full = smem_u32(&cs.full[s]);
            bool ok = mbar_wait_bounded(smem_u32(&cs.empty[s]), ((sc[c] / DEPTH) & 1) ^ 1, a.wait_limit);
            bool first = false;
            if (ok && chunk[c] == nch[c]) {          // the consumer needs its next item
                const int q = ic[c] & 1;
                ok = mbar_wait_bounded(smem_u32(&cs.qfree[q]), ((ic[c] >> 1) & 1) ^ 1, a.wait_limit);
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
                        d.P0 = CAUSAL ? 0 : partitions_of(n_rec.b.z, n_rec.b.y, a.pt);
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
                        tma_load_2d(kdst + b * CHUNK * 128, tmk, 64 * b, y, full, pol);
                        tma_load_2d(vdst + b * CHUNK * 128, tmv, 64 * b, y, full, pol);
                    }
                    if (two) {
#pragma unroll
                        for (int b = 0; b < C::BOXES; ++b) {
                            tma_load_2d(kdst + b * CHUNK * 128 + a.bs * 128, tmk, 64 * b, yb, full, pol);
                            tma_load_2d(vdst + b * CHUNK * 128 + a.bs * 128, tmv, 64 * b, yb, full, pol);
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
template <int D>
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
    __half *orow = a.out + ((long long)seq * a.Hq + h0) * D;
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
                h.x = pack_half2(acc[i].x, acc[i].y);
                h.y = pack_half2(acc[i].z, acc[i].w);
                *reinterpret_cast<uint2 *>(orow + 4 * k[i]) = h;
            }
    }
}

// Consumer warp c: reduces the items its producer hands it.  CAUSAL: the
// item's query rows may see different lengths of its token range (several
// new tokens of one sequence); scores past a row's own position are masked.
template <int D, int NT, bool CAUSAL>
__device__ void consumer(uint8_t *smem, int c, const DecodeArgs &a) {
    using C = Cfg<D, NT>;
    constexpr int DEPTH = C::DEPTH;
    constexpr int KS = D / 16;     // MMA k-steps of S^T = K Q^T
    constexpr int MT = D / 16;     // MMA m-tiles of O^T = V^T P^T
    const int lane = threadIdx.x & 31;
    const int r = lane >> 2, cq = lane & 3;
    const ConsumerSmem cs = consumer_smem<D, NT>(smem, c);

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
    bool owe = false;
    int owe_seq = 0, owe_kvh = 0, owe_P = 0;          // per lane: member lane
    int pend_ticket = 0, pend_seq = 0, pend_kvh = 0, pend_P = 0;
    auto take_ticket = [&]() {
        __syncwarp();
        __threadfence();
        pend_ticket = 0;
        if (owe_P > 1) pend_ticket = atomicAdd(&a.grp[owe_seq * a.Hkv + owe_kvh], 1);
        pend_seq = owe_seq;
        pend_kvh = owe_kvh;
        pend_P = owe_P;
        owe = false;
        owe_P = 0;
    };
    auto settle = [&]() {
        unsigned last = __ballot_sync(0xffffffffu, pend_P > 1 && pend_ticket == pend_P - 1);
        if (last) __threadfence();
        while (last) {
            const int l0 = __ffs(last) - 1;
            last &= last - 1;
            merge_group<D>(a, __shfl_sync(0xffffffffu, pend_seq, l0), __shfl_sync(0xffffffffu, pend_kvh, l0),
                           __shfl_sync(0xffffffffu, pend_P, l0));
        }
        pend_P = 0;
    };

    int stage = 0;
    for (int item = 0;; ++item) {
        const int q = item & 1;
        int s = stage % DEPTH;
        if (!mbar_wait_bounded(smem_u32(&cs.full[s]), (stage / DEPTH) & 1, a.wait_limit)) {
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
        uint32_t qb[NT][KS][2];
        {
            const __half *qs = reinterpret_cast<const __half *>(smem + c * C::DATA + DEPTH * C::STAGE + q * C::QSLOT);
#pragma unroll
            for (int t = 0; t < NT; ++t)
#pragma unroll
                for (int k = 0; k < KS; ++k) {
                    const __half *row = qs + (t * 8 + r) * D + 16 * k + 2 * cq;
                    qb[t][k][0] = *reinterpret_cast<const uint32_t *>(row);
                    qb[t][k][1] = *reinterpret_cast<const uint32_t *>(row + 8);
                }
        }
        const int nchunks = dp->nchunks;
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
                if (!mbar_wait_bounded(smem_u32(&cs.full[s]), (stage / DEPTH) & 1, a.wait_limit)) {
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
#pragma unroll
            for (int k = 0; k < KS; ++k) {
                uint32_t a0, a1, a2, a3;
                ldmatrix_x4(kt + (k >> 2) * (C::BOXES > 1 ? CHUNK * 128 : 0) + koff[k & 3], a0, a1, a2, a3);
#pragma unroll
                for (int t = 0; t < NT; ++t) {
                    float *acc_s = (k & 1) ? sb[t] : sa[t];
                    mma_16816(acc_s[0], acc_s[1], acc_s[2], acc_s[3], a0, a1, a2, a3, qb[t][k][0], qb[t][k][1],
                              acc_s[0], acc_s[1], acc_s[2], acc_s[3]);
                }
            }
            // V^T fragments, loaded ahead of the softmax
            uint32_t va[MT][4];
#pragma unroll
            for (int i = 0; i < MT; ++i)
                ldmatrix_x4_trans(vt + (i >> 2) * (C::BOXES > 1 ? CHUNK * 128 : 0) + voff[i & 3], va[i][0], va[i][1],
                                  va[i][2], va[i][3]);

            // softmax per head column; thread holds tokens r, r + 8
            const bool tail = ntok < CHUNK;
            const bool tok_lo = r < ntok, tok_hi = r + 8 < ntok;
            uint32_t pb[NT][2];
#pragma unroll
            for (int t = 0; t < NT; ++t) {
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
                pb[t][0] = movmatrix_trans(pack_half2(p0, p1));
                pb[t][1] = movmatrix_trans(pack_half2(p2, p3));
            }
            if (tail) {   // stale or poisoned slots past the context must not reach O
                const uint32_t lo = (2 * cq < ntok ? 0x0000ffffu : 0u) | (2 * cq + 1 < ntok ? 0xffff0000u : 0u);
                const uint32_t hi = (2 * cq + 8 < ntok ? 0x0000ffffu : 0u) | (2 * cq + 9 < ntok ? 0xffff0000u : 0u);
#pragma unroll
                for (int i = 0; i < MT; ++i) {
                    va[i][0] &= lo;
                    va[i][1] &= lo;
                    va[i][2] &= hi;
                    va[i][3] &= hi;
                }
            }
            // O^T += V^T P^T
#pragma unroll
            for (int i = 0; i < MT; ++i)
#pragma unroll
                for (int t = 0; t < NT; ++t)
                    mma_16816(acc[i][t][0], acc[i][t][1], acc[i][t][2], acc[i][t][3], va[i][0], va[i][1], va[i][2],
                              va[i][3], pb[t][0], pb[t][1], acc[i][t][0], acc[i][t][1], acc[i][t][2], acc[i][t][3]);
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
                        P = partitions_of(__ldg(&a.context_lens[seq]), dsc.shared, a.pt);
                        canon = __ldg(&a.part_off[seq]) + dsc.pidx;
                    }
                    const int h = dsc.kvh * a.G + g;
                    if (P == 1) {
                        const float inv = dsc.bad ? qnan : 1.f / l[t][e];
                        __half *orow = a.out + ((long long)seq * a.Hq + h) * D;
#pragma unroll
                        for (int i = 0; i < MT; ++i) {
                            orow[16 * i + r] = __float2half_rn(acc[i][t][e] * inv);
                            orow[16 * i + r + 8] = __float2half_rn(acc[i][t][e + 2] * inv);
                        }
                    } else {
                        const long long wrow = (long long)canon * a.Hq + h;
                        float *orow = a.ws_o + wrow * D;
#pragma unroll
                        for (int i = 0; i < MT; ++i) {
                            orow[16 * i + r] = dsc.bad ? qnan : acc[i][t][e];
                            orow[16 * i + r + 8] = dsc.bad ? qnan : acc[i][t][e + 2];
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
            owe_P = dsc.canon0 < 0 ? partitions_of(__ldg(&a.context_lens[owe_seq]), dsc.shared, a.pt) : dsc.P0;
        }
        owe = __any_sync(0xffffffffu, owe_P > 1);
    }
}

template <int D, int NT, bool CAUSAL>
__global__ void __launch_bounds__(NWARPS * 32, NT == 1 ? PA_DECODE_MINB : PA_DECODE_MINB_WIDE) decode_kernel(const __grid_constant__ CUtensorMap tmk,
                                                             const __grid_constant__ CUtensorMap tmv,
                                                             const DecodeArgs a) {
    extern __shared__ uint8_t smem_raw[];
    uint8_t *smem = reinterpret_cast<uint8_t *>((reinterpret_cast<uintptr_t>(smem_raw) + 1023) & ~uintptr_t(1023));
    const int warp = threadIdx.x >> 5;
    if (threadIdx.x == 0) {
        for (int c = 0; c < NC; ++c) {
            const ConsumerSmem cs = consumer_smem<D, NT>(smem, c);
            for (int s = 0; s < Cfg<D, NT>::DEPTH; ++s) {
                mbar_init(smem_u32(&cs.full[s]), 1);
                mbar_init(smem_u32(&cs.empty[s]), 1);
            }
            mbar_init(smem_u32(&cs.qfree[0]), 1);
            mbar_init(smem_u32(&cs.qfree[1]), 1);
        }
        fence_mbar_init();
    }
    __syncthreads();
    if (warp == 0)
        producer<D, NT, CAUSAL>(smem, &tmk, &tmv, a);
    else
        consumer<D, NT, CAUSAL>(smem, warp - 1, a);
}

// ------------------------------------------------------------ host side

PFN_cuTensorMapEncodeTiled_v12000 tensor_map_encoder() {
    static PFN_cuTensorMapEncodeTiled_v12000 fn = nullptr;
    static std::once_flag once;
    std::call_once(once, [] {
        void *p = nullptr;
        cudaDriverEntryPointQueryResult q;
        if (cudaGetDriverEntryPointByVersion("cuTensorMapEncodeTiled", &p, 12000, cudaEnableDefault, &q) ==
                cudaSuccess &&
            q == cudaDriverEntryPointSuccess)
            fn = reinterpret_cast<PFN_cuTensorMapEncodeTiled_v12000>(p);
    });
    return fn;
}

struct MapKey {
    const void *base;
    long long rows;
    int D, box_rows;
    bool operator==(const MapKey &o) const {
        return base == o.base && rows == o.rows && D == o.D && box_rows == o.box_rows;
    }
};

// 2-D view of a cache as [rows = num_blocks * Hkv * bs][D] fp16, boxes of
// 64 columns x box_rows rows, 128-byte swizzle.  Encoded maps are cached.
bool cache_tensor_map(CUtensorMap *map, const void *base, long long rows, int D, int box_rows) {
    static std::mutex mu;
    static std::vector<std::pair<MapKey, CUtensorMap>> cache;
    const MapKey key{base, rows, D, box_rows};
    std::lock_guard<std::mutex> lock(mu);
    for (auto &e : cache)
        if (e.first == key) {
            *map = e.second;
            return true;
        }
    auto enc = tensor_map_encoder();
    if (!enc) return false;
    cuuint64_t dims[2] = {(cuuint64_t)D, (cuuint64_t)rows};
    cuuint64_t strides[1] = {(cuuint64_t)D * 2};
    cuuint32_t box[2] = {64u, (cuuint32_t)box_rows};
    cuuint32_t estr[2] = {1u, 1u};
    CUresult res = enc(map, CU_TENSOR_MAP_DATA_TYPE_FLOAT16, 2, const_cast<void *>(base), dims, strides, box, estr,
                       CU_TENSOR_MAP_INTERLEAVE_NONE, CU_TENSOR_MAP_SWIZZLE_128B, CU_TENSOR_MAP_L2_PROMOTION_L2_256B,
                       CU_TENSOR_MAP_FLOAT_OOB_FILL_NONE);
    if (res != CUDA_SUCCESS) return false;
    if (cache.size() >= 32) cache.erase(cache.begin());
    cache.emplace_back(key, *map);
    return true;
}

template <int D, int NT, bool CAUSAL>
int launch_decode(const CUtensorMap &tmk, const CUtensorMap &tmv, const DecodeArgs &args, long long max_items,
                  cudaStream_t st) {
    using C = Cfg<D, NT>;
    static int grid = 0;
    static std::once_flag once;
    static cudaError_t init_err = cudaSuccess;
    std::call_once(once, [] {
        init_err =
            cudaFuncSetAttribute(decode_kernel<D, NT, CAUSAL>, cudaFuncAttributeMaxDynamicSharedMemorySize, C::SMEM);
        if (init_err != cudaSuccess) return;
        int dev = 0, sms = 0, per_sm = 0;
        init_err = cudaGetDevice(&dev);
        if (init_err == cudaSuccess) init_err = cudaDeviceGetAttribute(&sms, cudaDevAttrMultiProcessorCount, dev);
        if (init_err == cudaSuccess)
            init_err = cudaOccupancyMaxActiveBlocksPerMultiprocessor(&per_sm, decode_kernel<D, NT, CAUSAL>,
                                                                     NWARPS * 32, C::SMEM);
        if (init_err == cudaSuccess) grid = sms * (per_sm > 0 ? per_sm : 1);
    });
    if (init_err != cudaSuccess || grid <= 0) return PA_ERR_CUDA;
    // no more CTAs than there can be items for their consumers
    const long long need = (max_items + NC - 1) / NC;
    const int g = (int)(need < grid ? (need > 0 ? need : 1) : grid);
    decode_kernel<D, NT, CAUSAL><<<g, NWARPS * 32, C::SMEM, st>>>(tmk, tmv, args);
    return cuda_status(cudaGetLastError());
}

}  // namespace
}  // namespace pa

using namespace pa;

namespace pa {
namespace {

// Bound of the kernel's pipeline waits: about a second, or the value of
// PA_WAIT_LIMIT_CYCLES (read once) -- a small value makes the waits give up,
// which is how the timeout path is tested without a fault or a hang.
long long wait_limit_cycles() {
    static const long long v = [] {
        const char *e = std::getenv("PA_WAIT_LIMIT_CYCLES");
        const long long x = e ? std::atoll(e) : 0;
        return x > 0 ? x : WAIT_LIMIT;
    }();
    return v;
}

// One decode call; lead/shared_len are null for pa_decode.
int decode_impl(uint16_t *out, const uint16_t *query, const uint16_t *k_cache, const uint16_t *v_cache,
                const int32_t *block_tables, const int32_t *context_lens, const int32_t *lead,
                const int32_t *shared_len, int num_seqs, int num_heads, int num_kv_heads, int head_dim, int block_size,
                int64_t num_blocks, int max_blocks_per_seq, int max_context_len, float scale, void *workspace,
                size_t workspace_bytes, cudaStream_t st) {
    const bool grouped = lead != nullptr;
    if (num_seqs < 0 || num_heads <= 0 || num_kv_heads <= 0 || num_heads % num_kv_heads != 0 ||
        max_context_len < 0 || max_blocks_per_seq <= 0 || num_blocks <= 0 || !std::isfinite(scale) || !(scale > 0.f))
        return PA_ERR_INVALID_ARG;
    const int G = num_heads / num_kv_heads;
    if ((head_dim != 64 && head_dim != 128) || (block_size != 8 && block_size != 16 && block_size != 32) || G > 16)
        return PA_ERR_UNSUPPORTED;
    if (num_seqs == 0) return PA_OK;
    if (!out || !query || !k_cache || !v_cache || !block_tables || !context_lens || (grouped && !shared_len))
        return PA_ERR_INVALID_ARG;
    if (!aligned16(out) || !aligned16(query) || !aligned16(k_cache) || !aligned16(v_cache))
        return PA_ERR_INVALID_ARG;
    const long long rows = (long long)num_blocks * num_kv_heads * block_size;
    if (rows >= (1LL << 31)) return PA_ERR_UNSUPPORTED;
    const WsLayout L = ws_layout(num_seqs, num_heads, num_kv_heads, head_dim, max_context_len, grouped);
    if (!workspace || (reinterpret_cast<uintptr_t>(workspace) & 255u) || workspace_bytes < L.total)
        return PA_ERR_WORKSPACE;
    if (debug_validate()) {
        std::vector<int32_t> lens((size_t)num_seqs), tab((size_t)num_seqs * max_blocks_per_seq);
        std::vector<int32_t> ld, sl;
        if (cudaMemcpyAsync(lens.data(), context_lens, sizeof(int32_t) * lens.size(), cudaMemcpyDeviceToHost, st) !=
                cudaSuccess ||
            cudaMemcpyAsync(tab.data(), block_tables, sizeof(int32_t) * tab.size(), cudaMemcpyDeviceToHost, st) !=
                cudaSuccess)
            return PA_ERR_CUDA;
        if (grouped) {
            ld.resize((size_t)num_seqs);
            sl.resize((size_t)num_seqs);
            if (cudaMemcpyAsync(ld.data(), lead, sizeof(int32_t) * ld.size(), cudaMemcpyDeviceToHost, st) !=
                    cudaSuccess ||
                cudaMemcpyAsync(sl.data(), shared_len, sizeof(int32_t) * sl.size(), cudaMemcpyDeviceToHost, st) !=
                    cudaSuccess)
                return PA_ERR_CUDA;
        }
        if (cudaStreamSynchronize(st) != cudaSuccess) return PA_ERR_CUDA;
        for (int i = 0; i < num_seqs; ++i) {
            const int len = lens[(size_t)i];
            if (len < 0 || len > max_context_len || (long long)len > (long long)max_blocks_per_seq * block_size)
                return PA_ERR_INVALID_ARG;
            for (int b = 0; b < (len + block_size - 1) / block_size; ++b) {
                const int32_t id = tab[(size_t)i * max_blocks_per_seq + b];
                if (id < 0 || id >= num_blocks) return PA_ERR_INVALID_ARG;
            }
            if (grouped) {   // a member's shared blocks must be its leader's
                const int l = ld[(size_t)i];
                if (l < 0 || l > i || (l < i && ld[(size_t)i - 1] != l)) return PA_ERR_INVALID_ARG;
                if (l == i && sl[(size_t)i] < 0) return PA_ERR_INVALID_ARG;
                const int S = sl[(size_t)l] / block_size * block_size;
                if (l < i && S > len) return PA_ERR_INVALID_ARG;
                for (int b = 0; l < i && b < S / block_size; ++b)
                    if (tab[(size_t)i * max_blocks_per_seq + b] != tab[(size_t)l * max_blocks_per_seq + b])
                        return PA_ERR_INVALID_ARG;
            }
        }
    }
    const int box_rows = block_size < CHUNK ? block_size : CHUNK;
    CUtensorMap tmk, tmv;
    if (!cache_tensor_map(&tmk, k_cache, rows, head_dim, box_rows) ||
        !cache_tensor_map(&tmv, v_cache, rows, head_dim, box_rows))
        return PA_ERR_CUDA;

    // query rows per item: one sequence's G heads, or, for a shared range,
    // as many members' G heads as two head tiles hold
    const int NT = (G > 8 || grouped) ? 2 : 1;
    const int ms = grouped ? (16 / G > 1 ? 16 / G : 1) : 1;

    uint8_t *ws = static_cast<uint8_t *>(workspace);
    WsHeader *hdr = reinterpret_cast<WsHeader *>(ws);
    int *part_off = reinterpret_cast<int *>(ws + L.part_off);
    int *gsize = grouped ? reinterpret_cast<int *>(ws + L.gsize) : nullptr;
    int *gshared = grouped ? reinterpret_cast<int *>(ws + L.gshared) : nullptr;
    ItemRec *items = reinterpret_cast<ItemRec *>(ws + L.items);
    const bool multi = L.pmax > 1 || grouped;
    int *grp = multi ? reinterpret_cast<int *>(ws + L.grp) : nullptr;
    float2 *ws_ml = reinterpret_cast<float2 *>(ws + L.ml);
    float *ws_o = reinterpret_cast<float *>(ws + L.o);
    __half *hout = reinterpret_cast<__half *>(out);

    decode_prep_kernel<<<1, PREP_THREADS, 0, st>>>(context_lens, lead, shared_len, num_seqs, num_heads, head_dim,
                                                   num_kv_heads, block_size, max_context_len,
                                                   (long long)max_blocks_per_seq * block_size, L.pt, ms, hdr,
                                                   part_off, gsize, gshared, items, grp, hout);
    if (cudaGetLastError() != cudaSuccess) return PA_ERR_CUDA;

    DecodeArgs args;
    args.out = hout;
    args.query = reinterpret_cast<const __half *>(query);
    args.block_tables = block_tables;
    args.context_lens = context_lens;
    args.Hq = num_heads;
    args.Hkv = num_kv_heads;
    args.G = G;
    args.bs = block_size;
    args.mbps = max_blocks_per_seq;
    args.pt = L.pt;
    args.ms = ms;
    args.num_blocks = num_blocks;
    args.wait_limit = wait_limit_cycles();
    args.scale_log2 = scale * 1.4426950408889634f;
    args.hdr = hdr;
    args.part_off = part_off;
    args.items = items;
    args.grp = grp;
    args.ws_ml = ws_ml;
    args.ws_o = ws_o;
    const long long max_items = L.item_cap * num_kv_heads;
    if (head_dim == 128)
        return NT == 1 ? launch_decode<128, 1, false>(tmk, tmv, args, max_items, st)
                       : launch_decode<128, 2, false>(tmk, tmv, args, max_items, st);
    return NT == 1 ? launch_decode<64, 1, false>(tmk, tmv, args, max_items, st)
                   : launch_decode<64, 2, false>(tmk, tmv, args, max_items, st);
}

// One multi-token (causal) call.
int causal_impl(uint16_t *out, const uint16_t *query, const uint16_t *k_cache, const uint16_t *v_cache,
                const int32_t *block_tables, const int32_t *context_lens, const int32_t *query_start, int num_seqs,
                int num_query_tokens, int num_heads, int num_kv_heads, int head_dim, int block_size,
                int64_t num_blocks, int max_blocks_per_seq, int max_context_len, float scale, void *workspace,
                size_t workspace_bytes, cudaStream_t st) {
    if (num_seqs < 0 || num_query_tokens < 0 || num_heads <= 0 || num_kv_heads <= 0 ||
        num_heads % num_kv_heads != 0 || max_context_len < 0 || max_blocks_per_seq <= 0 || num_blocks <= 0 ||
        !std::isfinite(scale) || !(scale > 0.f))
        return PA_ERR_INVALID_ARG;
    const int G = num_heads / num_kv_heads;
    if ((head_dim != 64 && head_dim != 128) || (block_size != 8 && block_size != 16 && block_size != 32) || G > 16)
        return PA_ERR_UNSUPPORTED;
    if (num_query_tokens == 0) return PA_OK;
    if (num_seqs == 0) return PA_ERR_INVALID_ARG;
    if (!out || !query || !k_cache || !v_cache || !block_tables || !context_lens || !query_start)
        return PA_ERR_INVALID_ARG;
    if (!aligned16(out) || !aligned16(query) || !aligned16(k_cache) || !aligned16(v_cache))
        return PA_ERR_INVALID_ARG;
    const long long rows = (long long)num_blocks * num_kv_heads * block_size;
    if (rows >= (1LL << 31)) return PA_ERR_UNSUPPORTED;
    const WsLayout L = ws_layout_causal(num_seqs, num_query_tokens, num_heads, num_kv_heads, head_dim,
                                        max_context_len);
    // item and partial-row indices are 32-bit
    if (L.item_cap * num_kv_heads >= (1LL << 31) || (long long)num_query_tokens * L.pmax >= (1LL << 31))
        return PA_ERR_UNSUPPORTED;
    if (!workspace || (reinterpret_cast<uintptr_t>(workspace) & 255u) || workspace_bytes < L.total)
        return PA_ERR_WORKSPACE;
    if (debug_validate()) {
        std::vector<int32_t> lens((size_t)num_seqs), tab((size_t)num_seqs * max_blocks_per_seq),
            qs((size_t)num_seqs + 1);
        if (cudaMemcpyAsync(lens.data(), context_lens, sizeof(int32_t) * lens.size(), cudaMemcpyDeviceToHost, st) !=
                cudaSuccess ||
            cudaMemcpyAsync(tab.data(), block_tables, sizeof(int32_t) * tab.size(), cudaMemcpyDeviceToHost, st) !=
                cudaSuccess ||
            cudaMemcpyAsync(qs.data(), query_start, sizeof(int32_t) * qs.size(), cudaMemcpyDeviceToHost, st) !=
                cudaSuccess ||
            cudaStreamSynchronize(st) != cudaSuccess)
            return PA_ERR_CUDA;
        if (qs[0] != 0 || qs[(size_t)num_seqs] != num_query_tokens) return PA_ERR_INVALID_ARG;
        for (int i = 0; i < num_seqs; ++i) {
            const int len = lens[(size_t)i];
            const int T = qs[(size_t)i + 1] - qs[(size_t)i];
            if (T < 0 || T > len || len > max_context_len ||
                (long long)len > (long long)max_blocks_per_seq * block_size)
                return PA_ERR_INVALID_ARG;
            for (int b = 0; b < (len + block_size - 1) / block_size; ++b) {
                const int32_t id = tab[(size_t)i * max_blocks_per_seq + b];
                if (id < 0 || id >= num_blocks) return PA_ERR_INVALID_ARG;
            }
        }
    }
    const int box_rows = block_size < CHUNK ? block_size : CHUNK;
    CUtensorMap tmk, tmv;
    if (!cache_tensor_map(&tmk, k_cache, rows, head_dim, box_rows) ||
        !cache_tensor_map(&tmv, v_cache, rows, head_dim, box_rows))
        return PA_ERR_CUDA;
    // query rows of up to ms new tokens fill the head tiles
    const int ms = 8 * PA_CAUSAL_NT / G > 1 ? 8 * PA_CAUSAL_NT / G : 1;
    if (PA_CAUSAL_NT == 1 && G > 8) return PA_ERR_UNSUPPORTED;

    uint8_t *ws = static_cast<uint8_t *>(workspace);
    WsHeader *hdr = reinterpret_cast<WsHeader *>(ws);
    int *part_off = reinterpret_cast<int *>(ws + L.part_off);
    int *vlen = reinterpret_cast<int *>(ws + L.gsize);
    int *gstart = reinterpret_cast<int *>(ws + L.gshared);
    ItemRec *items = reinterpret_cast<ItemRec *>(ws + L.items);
    int *grp = reinterpret_cast<int *>(ws + L.grp);
    __half *hout = reinterpret_cast<__half *>(out);
    causal_prep_kernel<<<1, PREP_THREADS, 0, st>>>(context_lens, query_start, num_seqs, num_query_tokens, num_heads,
                                                   head_dim, num_kv_heads, max_context_len,
                                                   (long long)max_blocks_per_seq * block_size, L.pt, ms, hdr,
                                                   part_off, vlen, gstart, items, grp, hout);
    if (cudaGetLastError() != cudaSuccess) return PA_ERR_CUDA;

    DecodeArgs args;
    args.out = hout;
    args.query = reinterpret_cast<const __half *>(query);
    args.block_tables = block_tables;
    args.context_lens = vlen;   // per query row: the positions it sees
    args.Hq = num_heads;
    args.Hkv = num_kv_heads;
    args.G = G;
    args.bs = block_size;
    args.mbps = max_blocks_per_seq;
    args.pt = L.pt;
    args.ms = ms;
    args.num_blocks = num_blocks;
    args.wait_limit = wait_limit_cycles();
    args.scale_log2 = scale * 1.4426950408889634f;
    args.hdr = hdr;
    args.part_off = part_off;
    args.items = items;
    args.grp = grp;
    args.ws_ml = reinterpret_cast<float2 *>(ws + L.ml);
    args.ws_o = reinterpret_cast<float *>(ws + L.o);
    const long long max_items = L.item_cap * num_kv_heads;
    if (head_dim == 128) return launch_decode<128, PA_CAUSAL_NT, true>(tmk, tmv, args, max_items, st);
    return launch_decode<64, PA_CAUSAL_NT, true>(tmk, tmv, args, max_items, st);
}

}  // namespace
}  // namespace pa

extern "C" size_t pa_decode_workspace_size(int num_seqs, int num_heads, int num_kv_heads, int head_dim,
                                           int max_context_len) {
    if (num_seqs < 0 || num_heads <= 0 || num_kv_heads <= 0 || head_dim <= 0 || max_context_len < 0) return 0;
    return ws_layout(num_seqs, num_heads, num_kv_heads, head_dim, max_context_len, false).total;
}

extern "C" size_t pa_decode_shared_prefix_workspace_size(int num_seqs, int num_heads, int num_kv_heads, int head_dim,
                                                         int max_context_len) {
    if (num_seqs < 0 || num_heads <= 0 || num_kv_heads <= 0 || head_dim <= 0 || max_context_len < 0) return 0;
    return ws_layout(num_seqs, num_heads, num_kv_heads, head_dim, max_context_len, true).total;
}

extern "C" int pa_workspace_status(const void *workspace, int *status_out, void *stream) {
    if (!workspace || !status_out) return PA_ERR_INVALID_ARG;
    cudaStream_t st = static_cast<cudaStream_t>(stream);
    int err = 0;
    if (cudaMemcpyAsync(&err, workspace, sizeof(int), cudaMemcpyDeviceToHost, st) != cudaSuccess ||
        cudaStreamSynchronize(st) != cudaSuccess)
        return PA_ERR_CUDA;
    *status_out = err;
    return PA_OK;
}

extern "C" int pa_decode(uint16_t *out, const uint16_t *query, const uint16_t *k_cache, const uint16_t *v_cache,
                         const int32_t *block_tables, const int32_t *context_lens, int num_seqs, int num_heads,
                         int num_kv_heads, int head_dim, int block_size, int64_t num_blocks, int max_blocks_per_seq,
                         int max_context_len, float scale, void *workspace, size_t workspace_bytes, void *stream) {
    return decode_impl(out, query, k_cache, v_cache, block_tables, context_lens, nullptr, nullptr, num_seqs,
                       num_heads, num_kv_heads, head_dim, block_size, num_blocks, max_blocks_per_seq, max_context_len,
                       scale, workspace, workspace_bytes, static_cast<cudaStream_t>(stream));
}

extern "C" int pa_decode_shared_prefix(uint16_t *out, const uint16_t *query, const uint16_t *k_cache,
                                       const uint16_t *v_cache, const int32_t *block_tables,
                                       const int32_t *context_lens, const int32_t *group_leader,
                                       const int32_t *shared_len, int num_seqs, int num_heads, int num_kv_heads,
                                       int head_dim, int block_size, int64_t num_blocks, int max_blocks_per_seq,
                                       int max_context_len, float scale, void *workspace, size_t workspace_bytes,
                                       void *stream) {
    if (!group_leader) return PA_ERR_INVALID_ARG;
    return decode_impl(out, query, k_cache, v_cache, block_tables, context_lens, group_leader, shared_len, num_seqs,
                       num_heads, num_kv_heads, head_dim, block_size, num_blocks, max_blocks_per_seq, max_context_len,
                       scale, workspace, workspace_bytes, static_cast<cudaStream_t>(stream));
}

extern "C" size_t pa_attention_causal_workspace_size(int num_seqs, int num_query_tokens, int num_heads,
                                                     int num_kv_heads, int head_dim, int max_context_len) {
    if (num_seqs < 0 || num_query_tokens < 0 || num_heads <= 0 || num_kv_heads <= 0 ||
        num_heads % num_kv_heads != 0 || head_dim <= 0 || max_context_len < 0)
        return 0;
    return ws_layout_causal(num_seqs, num_query_tokens, num_heads, num_kv_heads, head_dim, max_context_len).total;
}

extern "C" int pa_attention_causal(uint16_t *out, const uint16_t *query, const uint16_t *k_cache,
                                   const uint16_t *v_cache, const int32_t *block_tables, const int32_t *context_lens,
                                   const int32_t *query_start, int num_seqs, int num_query_tokens, int num_heads,
                                   int num_kv_heads, int head_dim, int block_size, int64_t num_blocks,
                                   int max_blocks_per_seq, int max_context_len, float scale, void *workspace,
                                   size_t workspace_bytes, void *stream) {
    return causal_impl(out, query, k_cache, v_cache, block_tables, context_lens, query_start, num_seqs,
                       num_query_tokens, num_heads, num_kv_heads, head_dim, block_size, num_blocks,
                       max_blocks_per_seq, max_context_len, scale, workspace, workspace_bytes,
                       static_cast<cudaStream_t>(stream));
}

// ------------------------------------------------ failure-detection self-test

namespace pa {
namespace {

// Waits, with the decode pipeline's bounded wait, on an mbarrier that nothing
// ever completes; the wait must give up after `limit` cycles.
__global__ void selftest_wait_kernel(long long limit, int *status) {
    __shared__ uint64_t bar;
    if (threadIdx.x == 0) {
        mbar_init(smem_u32(&bar), 1);
        fence_mbar_init();
    }
    __syncthreads();
    const bool ok = mbar_wait_bounded(smem_u32(&bar), 0, limit);
    if (threadIdx.x == 0) *status = ok ? PA_OK : PA_ERR_TIMEOUT;
}

}  // namespace
}  // namespace pa

extern "C" int pa_selftest_wait_timeout(long long limit_cycles, int *status_device, void *stream) {
    if (!status_device || limit_cycles <= 0 || limit_cycles > WAIT_LIMIT) return PA_ERR_INVALID_ARG;
    selftest_wait_kernel<<<1, 32, 0, static_cast<cudaStream_t>(stream)>>>(limit_cycles, status_device);
    return cuda_status(cudaGetLastError());
}

// ------------------------------------------------ decode without allocation

// Scratch for pa_decode_static_ws: a file-scope device array, so that callers
// that may not allocate device memory still have somewhere for the partition
// results.  In host code the name g_static_ws is only a stand-in; its device
// address comes from cudaGetSymbolAddress, once per device.
static __device__ __align__(256) uint8_t g_static_ws[PA_DECODE_STATIC_WS_BYTES];

namespace pa {
namespace {

constexpr int MAX_DEVICES = 64;

// Device address of g_static_ws on the current device, looked up on the first
// call for that device; nullptr if the lookup fails.
void *static_ws_address(int device) {
    static std::mutex mu;
    static void *addr[MAX_DEVICES] = {};
    if (device < 0 || device >= MAX_DEVICES) return nullptr;
    std::lock_guard<std::mutex> lock(mu);
    if (!addr[device]) {
        void *p = nullptr;
        if (cudaGetSymbolAddress(&p, g_static_ws) != cudaSuccess || !p) return nullptr;
        addr[device] = p;
    }
    return addr[device];
}

}  // namespace
}  // namespace pa

extern "C" int pa_decode_static_ws(uint16_t *out, const uint16_t *query, const uint16_t *k_cache,
                                   const uint16_t *v_cache, const int32_t *block_tables,
                                   const int32_t *context_lens, int num_seqs, int num_heads, int num_kv_heads,
                                   int head_dim, int block_size, int64_t num_blocks, int max_blocks_per_seq,
                                   int max_context_len, float scale, void *stream) {
    if (num_seqs < 0 || num_heads <= 0 || num_kv_heads <= 0 || head_dim <= 0 || max_context_len < 0)
        return PA_ERR_INVALID_ARG;
    if (ws_layout(num_seqs, num_heads, num_kv_heads, head_dim, max_context_len, false).total >
        (size_t)PA_DECODE_STATIC_WS_BYTES)
        return PA_ERR_WORKSPACE;
    if (num_seqs == 0) return PA_OK;
    int device = -1;
    if (cudaGetDevice(&device) != cudaSuccess) return PA_ERR_CUDA;
    void *ws = static_ws_address(device);
    if (!ws) return PA_ERR_CUDA;
    return pa_decode(out, query, k_cache, v_cache, block_tables, context_lens, num_seqs, num_heads, num_kv_heads,
                     head_dim, block_size, num_blocks, max_blocks_per_seq, max_context_len, scale, ws,
                     (size_t)PA_DECODE_STATIC_WS_BYTES, stream);
}
