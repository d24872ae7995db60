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
#include <mutex>
#include <vector>

#include "common.cuh"

#ifndef PA_DECODE_CONSUMERS
#define PA_DECODE_CONSUMERS 1
#endif
#ifndef PA_DECODE_DEPTH
#define PA_DECODE_DEPTH 2
#endif
#ifndef PA_DECODE_MINB
#define PA_DECODE_MINB 8
#endif

namespace pa {
namespace {

constexpr int MAX_PART_TOKENS = 1024;           // largest partition (one work item)
constexpr long long TARGET_ITEMS = 4096;        // work items wanted for load balance
constexpr int CHUNK = 16;                       // tokens per pipeline stage (one MMA K step of P V)
constexpr int NC = PA_DECODE_CONSUMERS;         // consumer warps per CTA
constexpr int DEPTH = PA_DECODE_DEPTH;          // pipeline stages per consumer
constexpr int NWARPS = NC + 1;                  // + the producer warp
constexpr long long WAIT_LIMIT = 1LL << 31;     // clock cycles (about a second)
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
    size_t part_off, sp_info, grp, ml, o, total;
    int pmax, pt;
};

inline size_t up256(size_t x) { return (x + 255) & ~size_t(255); }

WsLayout ws_layout(int B, int Hq, int Hkv, int D, int max_ctx) {
    WsLayout w;
    w.pt = part_tokens(B, Hkv, max_ctx);
    w.pmax = max_ctx > 0 ? (max_ctx + w.pt - 1) / w.pt : 1;
    size_t off = sizeof(WsHeader);
    w.part_off = off;
    off += up256(sizeof(int) * ((size_t)B + 1));
    w.sp_info = off;
    off += up256(sizeof(int4) * (size_t)B * w.pmax);
    w.grp = off;
    if (w.pmax > 1) off += up256(sizeof(int) * (size_t)B * Hq);
    w.ml = off;
    if (w.pmax > 1) off += up256(sizeof(float2) * (size_t)B * w.pmax * Hq);
    w.o = off;
    if (w.pmax > 1) off += up256(sizeof(float) * (size_t)B * w.pmax * Hq * D);
    w.total = off;
    return w;
}

struct DecodeArgs {
    __half *out;
    const __half *query;
    const int32_t *block_tables;
    int Hq, Hkv, G, bs, mbps, pt;
    long long num_blocks;
    float scale_log2;
    WsHeader *hdr;
    const int *part_off;
    const int4 *sp_info;
    int *grp;
    float2 *ws_ml;
    float *ws_o;
};

// What the producer tells a consumer about its next item (32 bytes).
struct ItemDesc {
    int seq, kvh, sp, P, nchunks, ntok_last, bad, end;
};

template <int D, int NT>
struct Cfg {
    static constexpr int BOXES = D / 64;                   // 64-column (128-byte) boxes per tile row
    static constexpr int TILE = BOXES * CHUNK * 128;       // one 16-token K or V tile
    static constexpr int STAGE = 2 * TILE;                 // K tile then V tile
    static constexpr int QSLOT = NT * 8 * D * 2;           // the group's query rows
    static constexpr int DATA = DEPTH * STAGE + 2 * QSLOT; // per consumer, a multiple of 1024
    static constexpr int CTRL = 256;                       // per consumer: barriers and descriptors
    static constexpr int SMEM = NC * (DATA + CTRL) + 1024;
    static_assert(DATA % 1024 == 0, "stages must stay 1024-byte aligned for the 128-byte swizzle");
    static_assert((2 * DEPTH + 2) * 8 + 2 * 32 <= CTRL, "control block too small");
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

// Work list, longest first: every sequence's partitions but its last are
// full (pt tokens) and come first, in sequence order; the last partitions
// follow in decreasing length (a counting sort on 16-token buckets), so
// that the dynamically scheduled tail of the kernel runs the shortest items.
// An item record is {seq, partition, L, canonical index}; partial results
// are stored at the canonical index part_off[seq] + partition, independent
// of the order.
__global__ void __launch_bounds__(PREP_THREADS) decode_prep_kernel(
    const int32_t *__restrict__ context_lens, int B, int Hq, int D, int Hkv, int max_ctx, long long max_table_tokens,
    int pt, WsHeader *hdr, int *part_off, int4 *sp_info, int *grp, __half *out) {
    constexpr int NBK = MAX_PART_TOKENS / CHUNK;     // length buckets of the last partitions
    __shared__ int warp_sums[PREP_THREADS / 32];
    __shared__ int hist[NBK], cursor[NBK];
    int run_p = 0, run_f = 0;                        // uniform running totals
    for (int k = threadIdx.x; k < NBK; k += PREP_THREADS) hist[k] = cursor[k] = 0;
    if (grp)
        for (long long k = threadIdx.x; k < (long long)B * Hkv; k += PREP_THREADS) grp[k] = 0;
    __syncthreads();
    const int nbk = pt / CHUNK;
    // pass 1: partition counts, canonical offsets, full items, bucket histogram
    for (int base = 0; base < B; base += PREP_THREADS) {
        const int i = base + threadIdx.x;
        int L = 0, P = 0, code = 0;                  // code 1: zero row, 2: NaN row
        if (i < B) {
            L = context_lens[i];
            if (L < 0 || L > max_ctx || (long long)L > max_table_tokens)
                code = 2;
            else if (L == 0)
                code = 1;
            else
                P = (L + pt - 1) / pt;
        }
        int tp, tf;
        const int ep = run_p + block_exclusive_scan(P, warp_sums, &tp);
        const int ef = run_f + block_exclusive_scan(P > 0 ? P - 1 : 0, warp_sums, &tf);
        if (i < B) {
            part_off[i] = ep;
            for (int p = 0; p + 1 < P; ++p) sp_info[ef + p] = make_int4(i, p, L, ep + p);
            if (P > 0) atomicAdd(&hist[(pt - (L - (P - 1) * pt)) / CHUNK], 1);
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
    // bucket starts, largest last partitions first
    if (threadIdx.x == 0) {
        int acc = run_f;
        for (int k = 0; k < nbk; ++k) {
            cursor[k] = acc;
            acc += hist[k];
        }
    }
    __syncthreads();
    // pass 2: place the last partitions
    for (int i = threadIdx.x; i < B; i += PREP_THREADS) {
        const int L = context_lens[i];
        if (L <= 0 || L > max_ctx || (long long)L > max_table_tokens) continue;
        const int P = (L + pt - 1) / pt;
        const int slot = atomicAdd(&cursor[(pt - (L - (P - 1) * pt)) / CHUNK], 1);
        sp_info[slot] = make_int4(i, P - 1, L, part_off[i] + P - 1);
    }
    if (threadIdx.x == 0) {
        part_off[B] = run_p;
        hdr->total_items = run_p * Hkv;
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
    uint8_t *ctrl = smem + NC * C::DATA + c * C::CTRL;
    ConsumerSmem s;
    s.data = smem_u32(smem + c * C::DATA);
    s.full = reinterpret_cast<uint64_t *>(ctrl);
    s.empty = s.full + DEPTH;
    s.qfree = s.empty + DEPTH;
    s.desc = reinterpret_cast<ItemDesc *>(ctrl + (2 * DEPTH + 2) * 8);
    return s;
}

// Producer warp: hands items to the consumers round-robin and keeps their
// rings full.  All lanes run the loop; lane 0 issues the copies.
template <int D, int NT>
__device__ void producer(uint8_t *smem, const CUtensorMap *tmk, const CUtensorMap *tmv, const DecodeArgs &a) {
    using C = Cfg<D, NT>;
    const int lane = threadIdx.x & 31;
    const int total = a.hdr->total_items;
    const uint64_t pol = policy_evict_first();
    const int box_rows = a.bs < CHUNK ? a.bs : CHUNK;

    // Items are prefetched in three depths so that no latency is waited on
    // when a consumer needs its next item: the work-counter ticket three items
    // ahead (lane 0), the item record two ahead, and one ahead the item's
    // fields plus, per lane, its block-table entries lane and lane + 32.
    int raw = 0;
    int nn_item = -1;
    int4 nn_inf = make_int4(0, 0, 0, 0);
    int n_item = -1, n_seq = 0, n_p = 0, n_L = 0, n_P = 0, n_fb = 0, n_canon = 0;
    int n_e[ENTRIES];
#pragma unroll
    for (int e = 0; e < ENTRIES; ++e) n_e[e] = 0;
    auto advance = [&]() {
        n_item = nn_item;
        if (n_item >= 0) {
            n_seq = nn_inf.x;
            n_p = nn_inf.y;
            n_L = nn_inf.z;
            n_canon = nn_inf.w;
            n_P = (n_L + a.pt - 1) / a.pt;
            const int t0 = n_p * a.pt;
            const int t1 = min(n_L, t0 + a.pt);
            n_fb = t0 / a.bs;
            const int nb = (t1 + a.bs - 1) / a.bs - n_fb;
            const int32_t *row = a.block_tables + (long long)n_seq * a.mbps + n_fb;
#pragma unroll
            for (int e = 0; e < ENTRIES; ++e) n_e[e] = lane + 32 * e < nb ? row[lane + 32 * e] : 0;
        }
        const int j = __shfl_sync(0xffffffffu, raw, 0);
        nn_item = j < total ? j : -1;
        if (nn_item >= 0) nn_inf = a.sp_info[nn_item / a.Hkv];
        if (lane == 0) raw = atomicAdd(&a.hdr->counter, 1);
    };

    // per-consumer state (NC is small and the loops over it are unrolled)
    int sc[NC], ic[NC], chunk[NC], nch[NC], t0[NC], t1[NC], fb[NC], y[NC][ENTRIES], qrow[NC];
    bool done[NC], bad[NC];
#pragma unroll
    for (int c = 0; c < NC; ++c) {
        sc[c] = ic[c] = chunk[c] = nch[c] = t0[c] = t1[c] = fb[c] = qrow[c] = 0;
#pragma unroll
        for (int e = 0; e < ENTRIES; ++e) y[c][e] = 0;
        done[c] = bad[c] = false;
    }
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
            bool ok = mbar_wait_bounded(smem_u32(&cs.empty[s]), ((sc[c] / DEPTH) & 1) ^ 1, WAIT_LIMIT);
            bool first = false;
            if (ok && chunk[c] == nch[c]) {          // the consumer needs its next item
                const int q = ic[c] & 1;
                ok = mbar_wait_bounded(smem_u32(&cs.qfree[q]), ((ic[c] >> 1) & 1) ^ 1, WAIT_LIMIT);
                if (ok && n_item < 0) {              // nothing left: tell the consumer to stop
                    if (lane == 0) {
                        ItemDesc e = {0, 0, 0, 0, 0, 0, 0, 1};
                        cs.desc[q] = e;
                        mbar_arrive(full);
                    }
                    done[c] = true;
                    --live;
                    continue;
                }
                if (ok) {
                    const int sp = n_item / a.Hkv;
                    const int kvh = n_item - sp * a.Hkv;
                    t0[c] = n_p * a.pt;
                    t1[c] = min(n_L, t0[c] + a.pt);
                    fb[c] = n_fb;
                    nch[c] = (t1[c] - t0[c] + CHUNK - 1) / CHUNK;
                    const int nb = (t1[c] + a.bs - 1) / a.bs - n_fb;
                    bool bad_any = false;
#pragma unroll
                    for (int e = 0; e < ENTRIES; ++e) {
                        bad_any |= lane + 32 * e < nb && (n_e[e] < 0 || n_e[e] >= a.num_blocks);
                        y[c][e] = (int)(((long long)n_e[e] * a.Hkv + kvh) * a.bs);
                    }
                    bad[c] = __any_sync(0xffffffffu, bad_any);
                    qrow[c] = n_seq * a.Hq + kvh * a.G;
                    chunk[c] = 0;
                    if (lane == 0) {
                        ItemDesc d;
                        d.seq = n_seq;
                        d.kvh = kvh;
                        d.sp = n_canon;
                        d.P = n_P;
                        d.nchunks = nch[c];
                        d.ntok_last = t1[c] - (t0[c] + (nch[c] - 1) * CHUNK);
                        d.bad = bad[c] ? 1 : 0;
                        d.end = 0;
                        cs.desc[q] = d;
                    }
                    ++ic[c];
                    first = true;
                    advance();
                }
            }
            if (!ok) {   // a consumer stopped answering: record it and stop feeding everyone
                if (lane == 0) atomicExch(&a.hdr->error, PA_ERR_TIMEOUT);
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
                if (first && !bad[c]) bytes += (uint32_t)(a.G * D * 2);
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
                    if (first)
                        bulk_load(cs.data + DEPTH * C::STAGE + ((ic[c] - 1) & 1) * C::QSLOT,
                                  a.query + (long long)qrow[c] * D, (uint32_t)(a.G * D * 2), full);
                }
            }
            ++chunk[c];
            ++sc[c];
        }
    }
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

// Consumer warp c: reduces the items its producer hands it.
template <int D, int NT>
__device__ void consumer(uint8_t *smem, int c, const DecodeArgs &a) {
    using C = Cfg<D, NT>;
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

    // Merge tickets.  After an item of a multi-partition sequence has stored
    // its partial, it owes a ticket for its (sequence, kv head) group: the
    // ticket is taken after the next item's first chunk (by then the partial's
    // stores have drained, so the fence is cheap) and inspected at that item's
    // end (so the atomic's latency is hidden); the warp holding the group's
    // last ticket merges the group then.
    bool owe = false;
    int owe_seq = 0, owe_kvh = 0, owe_P = 0;
    int pend_ticket = 0, pend_seq = 0, pend_kvh = 0, pend_P = 0;
    auto take_ticket = [&]() {
        __syncwarp();
        __threadfence();
        pend_ticket = 0;
        if (lane == 0) pend_ticket = atomicAdd(&a.grp[owe_seq * a.Hkv + owe_kvh], 1);
        pend_seq = owe_seq;
        pend_kvh = owe_kvh;
        pend_P = owe_P;
        owe = false;
    };
    auto settle = [&]() {
        const int t = __shfl_sync(0xffffffffu, pend_ticket, 0);
        if (pend_P > 0 && t == pend_P - 1) {
            __threadfence();
            merge_group<D>(a, pend_seq, pend_kvh, pend_P);
        }
        pend_P = 0;
    };

    int stage = 0;
    for (int item = 0;; ++item) {
        const int q = item & 1;
        int s = stage % DEPTH;
        if (!mbar_wait_bounded(smem_u32(&cs.full[s]), (stage / DEPTH) & 1, WAIT_LIMIT)) {
            if (lane == 0) atomicExch(&a.hdr->error, PA_ERR_TIMEOUT);
            return;
        }
        const ItemDesc dsc = cs.desc[q];
        if (dsc.end) {
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
        __syncwarp();
        if (lane == 0) mbar_arrive(smem_u32(&cs.qfree[q]));   // query slot and descriptor read

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

        for (int ch = 0; ch < dsc.nchunks; ++ch) {
            if (ch > 0) {
                s = stage % DEPTH;
                if (!mbar_wait_bounded(smem_u32(&cs.full[s]), (stage / DEPTH) & 1, WAIT_LIMIT)) {
                    if (lane == 0) atomicExch(&a.hdr->error, PA_ERR_TIMEOUT);
                    return;
                }
            }
            const uint32_t kt = cs.data + s * C::STAGE;
            const uint32_t vt = kt + C::TILE;
            const int ntok = ch == dsc.nchunks - 1 ? dsc.ntok_last : CHUNK;

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
                if (tail) {
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
        if (dsc.P == 1) {
#pragma unroll
            for (int t = 0; t < NT; ++t)
#pragma unroll
                for (int e = 0; e < 2; ++e) {
                    const int g = t * 8 + 2 * cq + e;
                    if (g < a.G) {
                        const float inv = dsc.bad ? qnan : 1.f / l[t][e];
                        __half *orow = a.out + ((long long)dsc.seq * a.Hq + dsc.kvh * a.G + g) * D;
#pragma unroll
                        for (int i = 0; i < MT; ++i) {
                            orow[16 * i + r] = __float2half_rn(acc[i][t][e] * inv);
                            orow[16 * i + r + 8] = __float2half_rn(acc[i][t][e + 2] * inv);
                        }
                    }
                }
        } else {
#pragma unroll
            for (int t = 0; t < NT; ++t)
#pragma unroll
                for (int e = 0; e < 2; ++e) {
                    const int g = t * 8 + 2 * cq + e;
                    if (g < a.G) {
                        const long long wrow = (long long)dsc.sp * a.Hq + dsc.kvh * a.G + g;
                        float *orow = a.ws_o + wrow * D;
#pragma unroll
                        for (int i = 0; i < MT; ++i) {
                            orow[16 * i + r] = dsc.bad ? qnan : acc[i][t][e];
                            orow[16 * i + r + 8] = dsc.bad ? qnan : acc[i][t][e + 2];
                        }
                        if (r == 0) a.ws_ml[wrow] = dsc.bad ? make_float2(qnan, qnan) : make_float2(m[t][e], l[t][e]);
                    }
                }
        }
        // the ticket taken during this item: merge its group if it was the last
        settle();
        if (dsc.P > 1) {
            owe = true;
            owe_seq = dsc.seq;
            owe_kvh = dsc.kvh;
            owe_P = dsc.P;
        }
    }
}

template <int D, int NT>
__global__ void __launch_bounds__(NWARPS * 32, NT == 1 ? PA_DECODE_MINB : PA_DECODE_MINB / 2) decode_kernel(const __grid_constant__ CUtensorMap tmk,
                                                             const __grid_constant__ CUtensorMap tmv,
                                                             const DecodeArgs a) {
    extern __shared__ uint8_t smem_raw[];
    uint8_t *smem = reinterpret_cast<uint8_t *>((reinterpret_cast<uintptr_t>(smem_raw) + 1023) & ~uintptr_t(1023));
    const int warp = threadIdx.x >> 5;
    if (threadIdx.x == 0) {
        for (int c = 0; c < NC; ++c) {
            const ConsumerSmem cs = consumer_smem<D, NT>(smem, c);
            for (int s = 0; s < DEPTH; ++s) {
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
        producer<D, NT>(smem, &tmk, &tmv, a);
    else
        consumer<D, NT>(smem, warp - 1, a);
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

template <int D, int NT>
int launch_decode(const CUtensorMap &tmk, const CUtensorMap &tmv, const DecodeArgs &args, long long max_items,
                  cudaStream_t st) {
    using C = Cfg<D, NT>;
    static int grid = 0;
    static std::once_flag once;
    static cudaError_t init_err = cudaSuccess;
    std::call_once(once, [] {
        init_err = cudaFuncSetAttribute(decode_kernel<D, NT>, cudaFuncAttributeMaxDynamicSharedMemorySize, C::SMEM);
        if (init_err != cudaSuccess) return;
        int dev = 0, sms = 0, per_sm = 0;
        init_err = cudaGetDevice(&dev);
        if (init_err == cudaSuccess) init_err = cudaDeviceGetAttribute(&sms, cudaDevAttrMultiProcessorCount, dev);
        if (init_err == cudaSuccess)
            init_err = cudaOccupancyMaxActiveBlocksPerMultiprocessor(&per_sm, decode_kernel<D, NT>, NWARPS * 32,
                                                                     C::SMEM);
        if (init_err == cudaSuccess) grid = sms * (per_sm > 0 ? per_sm : 1);
    });
    if (init_err != cudaSuccess || grid <= 0) return PA_ERR_CUDA;
    // no more CTAs than there can be items for their consumers
    const long long need = (max_items + NC - 1) / NC;
    const int g = (int)(need < grid ? (need > 0 ? need : 1) : grid);
    decode_kernel<D, NT><<<g, NWARPS * 32, C::SMEM, st>>>(tmk, tmv, args);
    return cuda_status(cudaGetLastError());
}

}  // namespace
}  // namespace pa

using namespace pa;

extern "C" size_t pa_decode_workspace_size(int num_seqs, int num_heads, int num_kv_heads, int head_dim,
                                           int max_context_len) {
    if (num_seqs < 0 || num_heads <= 0 || num_kv_heads <= 0 || head_dim <= 0 || max_context_len < 0) return 0;
    return ws_layout(num_seqs, num_heads, num_kv_heads, head_dim, max_context_len).total;
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
    if (num_seqs < 0 || num_heads <= 0 || num_kv_heads <= 0 || num_heads % num_kv_heads != 0 ||
        max_context_len < 0 || max_blocks_per_seq <= 0 || num_blocks <= 0 || !std::isfinite(scale) || !(scale > 0.f))
        return PA_ERR_INVALID_ARG;
    const int G = num_heads / num_kv_heads;
    if ((head_dim != 64 && head_dim != 128) || (block_size != 8 && block_size != 16 && block_size != 32) || G > 16)
        return PA_ERR_UNSUPPORTED;
    if (num_seqs == 0) return PA_OK;
    if (!out || !query || !k_cache || !v_cache || !block_tables || !context_lens) return PA_ERR_INVALID_ARG;
    if (!aligned16(out) || !aligned16(query) || !aligned16(k_cache) || !aligned16(v_cache))
        return PA_ERR_INVALID_ARG;
    const long long rows = (long long)num_blocks * num_kv_heads * block_size;
    if (rows >= (1LL << 31)) return PA_ERR_UNSUPPORTED;
    const WsLayout L = ws_layout(num_seqs, num_heads, num_kv_heads, head_dim, max_context_len);
    if (!workspace || (reinterpret_cast<uintptr_t>(workspace) & 255u) || workspace_bytes < L.total)
        return PA_ERR_WORKSPACE;
    cudaStream_t st = static_cast<cudaStream_t>(stream);
    if (debug_validate()) {
        std::vector<int32_t> lens((size_t)num_seqs), tab((size_t)num_seqs * max_blocks_per_seq);
        if (cudaMemcpyAsync(lens.data(), context_lens, sizeof(int32_t) * lens.size(), cudaMemcpyDeviceToHost, st) !=
                cudaSuccess ||
            cudaMemcpyAsync(tab.data(), block_tables, sizeof(int32_t) * tab.size(), cudaMemcpyDeviceToHost, st) !=
                cudaSuccess ||
            cudaStreamSynchronize(st) != cudaSuccess)
            return PA_ERR_CUDA;
        for (int i = 0; i < num_seqs; ++i) {
            const int len = lens[(size_t)i];
            if (len < 0 || len > max_context_len || (long long)len > (long long)max_blocks_per_seq * block_size)
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

    uint8_t *ws = static_cast<uint8_t *>(workspace);
    WsHeader *hdr = reinterpret_cast<WsHeader *>(ws);
    int *part_off = reinterpret_cast<int *>(ws + L.part_off);
    int4 *sp_info = reinterpret_cast<int4 *>(ws + L.sp_info);
    int *grp = L.pmax > 1 ? reinterpret_cast<int *>(ws + L.grp) : nullptr;
    float2 *ws_ml = reinterpret_cast<float2 *>(ws + L.ml);
    float *ws_o = reinterpret_cast<float *>(ws + L.o);
    __half *hout = reinterpret_cast<__half *>(out);

    decode_prep_kernel<<<1, PREP_THREADS, 0, st>>>(context_lens, num_seqs, num_heads, head_dim, num_kv_heads,
                                                   max_context_len, (long long)max_blocks_per_seq * block_size, L.pt,
                                                   hdr, part_off, sp_info, grp, hout);
    if (cudaGetLastError() != cudaSuccess) return PA_ERR_CUDA;

    DecodeArgs args;
    args.out = hout;
    args.query = reinterpret_cast<const __half *>(query);
    args.block_tables = block_tables;
    args.Hq = num_heads;
    args.Hkv = num_kv_heads;
    args.G = G;
    args.bs = block_size;
    args.mbps = max_blocks_per_seq;
    args.pt = L.pt;
    args.num_blocks = num_blocks;
    args.scale_log2 = scale * 1.4426950408889634f;
    args.hdr = hdr;
    args.part_off = part_off;
    args.sp_info = sp_info;
    args.grp = grp;
    args.ws_ml = ws_ml;
    args.ws_o = ws_o;
    const long long max_items = (long long)num_seqs * num_kv_heads * L.pmax;
    int rc;
    if (head_dim == 128)
        rc = G <= 8 ? launch_decode<128, 1>(tmk, tmv, args, max_items, st)
                    : launch_decode<128, 2>(tmk, tmv, args, max_items, st);
    else
        rc = G <= 8 ? launch_decode<64, 1>(tmk, tmv, args, max_items, st)
                    : launch_decode<64, 2>(tmk, tmv, args, max_items, st);
    if (rc != PA_OK) return rc;
    return PA_OK;
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
    if (ws_layout(num_seqs, num_heads, num_kv_heads, head_dim, max_context_len).total >
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
