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

#include <cmath>
#include <cstdlib>
#include <mutex>
#include <vector>

#include "decode_common.cuh"
#include "prefill.h"

namespace pa {
namespace {

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
    long long max_table_tokens, int pt, int pts, int ms, WsHeader *hdr, int *part_off, int *gsize, int *gshared,
    ItemRec *items, int *grp, uint16_t *out, uint32_t nan2, int mt, int4 *sitems) {
    constexpr int NBK = MAX_PART_TOKENS / CHUNK;     // length buckets of the short items
    __shared__ int warp_sums[PREP_THREADS / 32];
    __shared__ int hist[NBK], cursor[NBK];
    int run_p = 0, run_f = 0, run_s = 0;             // uniform running totals
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
                    S = min(S, ok ? L - 1 : 0);   // every member keeps at least one token of its own
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
                P = partitions_of(L, S, pt, pts);
            if (P > 0) {
                nfull = (L - S + pt - 1) / pt - 1;   // own partitions but the last
                if (ld == i && S > 0) {
                    Ms = gsize[i];
                    Ps = (S + pts - 1) / pts;
                    if (!mt) nfull += (S / pts) * ((Ms + ms - 1) / ms);
                }
            }
        }
        int tp, tf, ts;
        const int ep = run_p + block_exclusive_scan(P, warp_sums, &tp);
        int ef = run_f + block_exclusive_scan(nfull, warp_sums, &tf);
        // shared ranges on the tensor cores: every partition of a leader's
        // shared range, for up to mt members at a time
        const int nsh = mt && Ps > 0 ? Ps * ((Ms + mt - 1) / mt) : 0;
        int es = run_s + block_exclusive_scan(nsh, warp_sums, &ts);
        if (i < B) {
            part_off[i] = ep;
            if (P > 0) {
                const int ps_i = (S + pts - 1) / pts;
                if (Ps > 0 && mt) {   // leader: its shared ranges, for the tensor-core kernel
                    for (int p = 0; p < Ps; ++p)
                        for (int k = 0; k < Ms; k += mt)
                            sitems[es++] = make_int4(i + k, min(mt, Ms - k), p * pts, min((p + 1) * pts, S));
                } else if (Ps > 0) {   // leader: full shared items (pts == pt here)
                    for (int p = 0; p < S / pts; ++p)
                        for (int k = 0; k < Ms; k += ms) {
                            ItemRec r;
                            r.a = make_int4(i + k, min(ms, Ms - k), p * pts, (p + 1) * pts);
                            r.b = make_int4(p, S, L, -1);
                            items[ef++] = r;
                        }
                    if (S % pts) atomicAdd(&hist[(pts - S % pts) / CHUNK], (Ms + ms - 1) / ms);
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
                const uint32_t h = code == 1 ? 0u : nan2;
                uint4 fill = make_uint4(h, h, h, h);
                uint4 *row = reinterpret_cast<uint4 *>(out + (long long)i * Hq * D);
                for (int k = 0; k < Hq * D / 8; ++k) row[k] = fill;
            }
        }
        run_p += tp;
        run_f += tf;
        run_s += ts;
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
        const int ps_i = (S + pts - 1) / pts;
        if (!mt && ld == i && S > 0 && S % pts) {
            const int Ms = gsize[i];
            for (int k = 0; k < Ms; k += ms) {
                ItemRec r;
                r.a = make_int4(i + k, min(ms, Ms - k), S / pts * pts, S);
                r.b = make_int4(ps_i - 1, S, L, -1);
                items[atomicAdd(&cursor[(pts - S % pts) / CHUNK], 1)] = r;
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
        hdr->pf_items = run_s * Hkv;
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
// A sequence with at least pf_min_rows query rows (new tokens x G; 0: none)
// goes to the tensor-core prefill kernels instead: it gets no items here.  Its
// ceil(T G / 128) row tiles, last rows first, are listed in ptiles when there
// is one (or when pairs is 0), otherwise in pptiles as pairs of neighbouring
// tiles {seq, tile, tile - 1, 0} (an odd one out as {seq, 0, -1, 0}) -- unless
// its rows number at most nr_max (0: never), then it is listed in ntiles
// ({seq, 0, 0, 0}) for the narrow kernel.  Its N = (listed sequences x Hkv)
// items run on nw_grid CTAs; when the last round is partial (R = N mod
// nw_grid items), those R items are split into k = nw_grid / R pieces of their
// KV ranges (at least two KV tiles each), which the kernel merges.
__global__ void __launch_bounds__(PREP_THREADS) causal_prep_kernel(
    const int32_t *__restrict__ context_lens, const int32_t *__restrict__ qs, int B, int NQ, int Hq, int D, int Hkv,
    int max_ctx, long long max_table_tokens, int pt, int ms, WsHeader *hdr, int *part_off, int *vlen, int *gstart,
    ItemRec *items, int *grp, uint16_t *out, uint32_t nan2, int pf_min_rows, int4 *ptiles, int4 *pptiles,
    int pairs, int nr_max, int4 *ntiles, int nw_grid, int *ntickets) {
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
    const int G = Hq / Hkv;
    auto prefill = [&](int T) { return pf_min_rows > 0 && (long long)T * G >= pf_min_rows; };
    // pass 1: visible length and partial-row offset of every query row
    int run = 0;
    for (int base = 0; base < NQ; base += PREP_THREADS) {
        const int v = base + threadIdx.x;
        int vl = -1;
        if (v < NQ && qs_ok) {
            const int i = last_le(qs, B, v);
            int L, T;
            if (seq_ok(i, L, T)) vl = prefill(T) ? 0 : L - T + (v - qs[i]) + 1;   // 0: the prefill kernel's row
        }
        int tot;
        const int e = run + block_exclusive_scan(vl > 0 ? (vl + pt - 1) / pt : 0, warp_sums, &tot);
        if (v < NQ) {
            vlen[v] = vl;
            part_off[v] = e;
            if (vl < 0) {
                uint4 fill = make_uint4(nan2, nan2, nan2, nan2);
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
        if (i < B && qs_ok && seq_ok(i, L, T) && !prefill(T)) n = (T + ms - 1) / ms;
        int tot;
        const int e = run_g + block_exclusive_scan(n, warp_sums, &tot);
        if (i < B) gstart[i] = e;
        run_g += tot;
    }
    // pass 2b: row tiles of the prefill kernels
    int run_t = 0, run_p = 0, run_n = 0;
    for (int base = 0; base < B; base += PREP_THREADS) {
        const int i = base + threadIdx.x;
        int n = 0, nn = 0, L, T;
        if (i < B && qs_ok && seq_ok(i, L, T) && prefill(T)) {
            if ((long long)T * G <= nr_max)
                nn = 1;
            else
                n = (int)(((long long)T * G + 127) / 128);
        }
        const bool paired = pairs && n >= 2;
        const int ns = paired ? 0 : n, np = paired ? (n + 1) / 2 : 0;
        int tot, totp, totn;
        const int e = run_t + block_exclusive_scan(ns, warp_sums, &tot);
        const int ep = run_p + block_exclusive_scan(np, warp_sums, &totp);
        const int en = run_n + block_exclusive_scan(nn, warp_sums, &totn);
        for (int k = 0; k < ns; ++k) ptiles[e + k] = make_int4(i, n - 1 - k, 0, 0);
        for (int k = 0; k < np; ++k) pptiles[ep + k] = make_int4(i, n - 1 - 2 * k, n - 2 - 2 * k, 0);
        if (nn) ntiles[en] = make_int4(i, 0, 0, 0);
        run_t += tot;
        run_p += totp;
        run_n += totn;
    }
    if (threadIdx.x == 0) {
        gstart[B] = run_g;
        part_off[NQ] = run;
        hdr->pf_items = run_t * Hkv;
        hdr->pf2_items = run_p * Hkv;
        hdr->pfn_items = run_n * Hkv;
    }
    __syncthreads();
    if (threadIdx.x == 0 && nw_grid > 0) {
        const int N = run_n * Hkv;
        int whole = N, k = 1;
        const int F = N / nw_grid, R = N - F * nw_grid;
        if (R > 0) {
            int kk = nw_grid / R;
            // every piece at least two KV tiles: capped by the shortest split item
            for (int x = N - R; x < N && kk >= 2; x += Hkv - (x % Hkv)) {
                const int nkv = (context_lens[ntiles[x / Hkv].x] + 127) / 128;
                kk = min(kk, nkv / 2);
            }
            if (kk >= 2) whole = F * nw_grid, k = kk;
        }
        hdr->pfn_whole = whole;
        hdr->pfn_split = k;
        hdr->pfn_items = whole + (N - whole) * k;
        for (int j = 0; j < NW_MAX_CTAS; ++j) ntickets[j] = 0;
    }
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
    int D, box_rows, kv;
    bool operator==(const MapKey &o) const {
        return base == o.base && rows == o.rows && D == o.D && box_rows == o.box_rows && kv == o.kv;
    }
};

// 2-D view of a cache as [rows = num_blocks * Hkv * bs][D] fp16, boxes of
// 64 columns x box_rows rows, 128-byte swizzle.  Encoded maps are cached.
bool cache_tensor_map(CUtensorMap *map, const void *base, long long rows, int D, int box_rows, int kv) {
    static std::mutex mu;
    static std::vector<std::pair<MapKey, CUtensorMap>> cache;
    const MapKey key{base, rows, D, box_rows, kv};
    std::lock_guard<std::mutex> lock(mu);
    for (auto &e : cache)
        if (e.first == key) {
            *map = e.second;
            return true;
        }
    auto enc = tensor_map_encoder();
    if (!enc) return false;
    cuuint64_t dims[2] = {(cuuint64_t)D, (cuuint64_t)rows};
    const bool fp8 = kv == PA_KV_FP8_E4M3;
    cuuint64_t strides[1] = {(cuuint64_t)D * (fp8 ? 1 : 2)};
    cuuint32_t box[2] = {fp8 ? 128u : 64u, (cuuint32_t)box_rows};   // 128-byte box rows
    cuuint32_t estr[2] = {1u, 1u};
    const CUtensorMapDataType dt = fp8 ? CU_TENSOR_MAP_DATA_TYPE_UINT8
                                   : kv == PA_KV_BF16 ? CU_TENSOR_MAP_DATA_TYPE_BFLOAT16
                                                      : CU_TENSOR_MAP_DATA_TYPE_FLOAT16;
    CUresult res = enc(map, dt, 2, const_cast<void *>(base), dims, strides, box, estr,
                       CU_TENSOR_MAP_INTERLEAVE_NONE, CU_TENSOR_MAP_SWIZZLE_128B, CU_TENSOR_MAP_L2_PROMOTION_L2_256B,
                       CU_TENSOR_MAP_FLOAT_OOB_FILL_NONE);
    if (res != CUDA_SUCCESS) return false;
    if (cache.size() >= 32) cache.erase(cache.begin());
    cache.emplace_back(key, *map);
    return true;
}

}  // namespace

int launch_kv_f16(int D, int NT, bool causal, const CUtensorMap &tmk, const CUtensorMap &tmv, const DecodeArgs &args,
                  long long max_items, cudaStream_t st) {
    return launch_kv<PA_KV_F16>(D, NT, causal, tmk, tmv, args, max_items, st);
}

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

// The tensor-core kernel for long runs of new tokens is used unless
// PA_PREFILL=0 (read once; then every sequence takes the decode pipeline).
bool prefill_enabled() {
    static const bool on = [] {
        const char *e = std::getenv("PA_PREFILL");
        return !(e && e[0] == '0');
    }();
    return on;
}

// Whether sequences with several row tiles take them in pairs on the two-tile
// tensor-core kernel (unless PA_PREFILL_PAIRS=0, read once).
bool prefill_pairs_enabled() {
    static const bool on = [] {
        const char *e = std::getenv("PA_PREFILL_PAIRS");
        return !(e && e[0] == '0');
    }();
    return on;
}

// Whether sequences (and shared ranges) of at most NARROW_ROWS query rows go to
// the narrow tensor-core kernel (unless PA_NARROW=0, read once).
bool narrow_enabled() {
    static const bool on = [] {
        const char *e = std::getenv("PA_NARROW");
        return !(e && e[0] == '0');
    }();
    return on;
}

// Shared-range pieces on the tensor cores span this many decode partitions
// (PA_SHARED_PIECE, read once; default 4: on the parallel-sampling workload a
// whole 2048-token prompt per piece, 1 % faster than pieces of one partition).
int shared_piece_factor() {
    static const int f = [] {
        const char *e = std::getenv("PA_SHARED_PIECE");
        const int v = e ? std::atoi(e) : 4;
        return v >= 1 && v <= 64 ? v : 4;
    }();
    return f;
}

// Whether shared ranges of at most NARROW_ROWS rows go to the narrow kernel
// (only with PA_NARROW_SHARED=1, read once).
bool narrow_shared_enabled() {
    static const bool on = [] {
        const char *e = std::getenv("PA_NARROW_SHARED");
        return e && e[0] == '1' && narrow_enabled();
    }();
    return on;
}

// ------------------------- the decode pipeline beside the tensor-core kernels

// A multi-token call with both kinds of sequence runs the decode pipeline (an
// HBM-bound kernel) on a second stream beside the tensor-core kernels (bound
// by the tensor cores and L2), forked from and joined back into the caller's
// stream with events.  The tensor-core kernels are launched first and take
// one SM each; the decode pipeline's CTAs take the SMs their last round leaves
// idle instead of waiting for all of them.  One stream and two events per
// device, created by the first such call on the device (before any stream
// capture); a mutex keeps each call's record / wait pairs together when
// several host threads call at once.  PA_PREFILL_SIDE=0 (read once) keeps
// everything on the caller's stream.
struct Side {
    std::mutex mu;
    cudaStream_t stream = nullptr;
    cudaEvent_t fork = nullptr, join = nullptr;
    bool ok = false, tried = false;
};

constexpr int MAX_SIDE_DEVICES = 64;

Side *side_of(int dev) {
    static std::mutex mu;
    static Side sides[MAX_SIDE_DEVICES];
    static const bool on = [] {
        const char *e = std::getenv("PA_PREFILL_SIDE");
        return !(e && e[0] == '0');
    }();
    if (!on || dev < 0 || dev >= MAX_SIDE_DEVICES) return nullptr;
    std::lock_guard<std::mutex> lock(mu);
    Side &sd = sides[dev];
    if (!sd.tried) {
        sd.tried = true;
        sd.ok = cudaStreamCreateWithFlags(&sd.stream, cudaStreamNonBlocking) == cudaSuccess &&
                cudaEventCreateWithFlags(&sd.fork, cudaEventDisableTiming) == cudaSuccess &&
                cudaEventCreateWithFlags(&sd.join, cudaEventDisableTiming) == cudaSuccess;
    }
    return sd.ok ? &sd : nullptr;
}

// Whether a grouped decode reduces its shared ranges on the tensor cores
// (unless PA_SHARED_TC=0, read once).
bool shared_tc_enabled() {
    static const bool on = [] {
        const char *e = std::getenv("PA_SHARED_TC");
        return !(e && e[0] == '0');
    }();
    return on;
}

// Checks of the cache element type and its scales; 0 when valid.
int check_kv(int kv, int head_dim, float k_scale, float v_scale) {
    if (kv != PA_KV_F16 && kv != PA_KV_BF16 && kv != PA_KV_FP8_E4M3) return PA_ERR_INVALID_ARG;
    if (kv == PA_KV_FP8_E4M3) {
        if (!std::isfinite(k_scale) || !(k_scale > 0.f) || !std::isfinite(v_scale) || !(v_scale > 0.f))
            return PA_ERR_INVALID_ARG;
        if (head_dim != 128) return PA_ERR_UNSUPPORTED;
    }
    return 0;
}

// The decode kernel's launch for a cache element type.
int launch_kv_any(int kv, int D, int NT, bool causal, const CUtensorMap &tmk, const CUtensorMap &tmv,
                  const DecodeArgs &args, long long max_items, cudaStream_t st) {
    if (kv == PA_KV_BF16) return launch_kv_bf16(D, NT, causal, tmk, tmv, args, max_items, st);
    if (kv == PA_KV_FP8_E4M3) return launch_kv_fp8(D, NT, causal, tmk, tmv, args, max_items, st);
    return launch_kv_f16(D, NT, causal, tmk, tmv, args, max_items, st);
}

// NaN in the output's 16-bit type, twice.
uint32_t nan_pair(int kv) { return kv == PA_KV_BF16 ? 0x7fc07fc0u : 0x7e007e00u; }

// What decode_checks returns for a valid call with no work (num_seqs = 0).
constexpr int NOTHING_TO_DO = 1;

// The host-side checks of a decode call that need neither device data nor the
// workspace, in the order the calls report them: PA_OK to go on,
// NOTHING_TO_DO, or the error status.
int decode_checks(const void *out, const void *query, const void *k_cache, const void *v_cache,
                  const int32_t *block_tables, const int32_t *context_lens, bool grouped, const int32_t *shared_len,
                  int num_seqs, int num_heads, int num_kv_heads, int head_dim, int block_size, int64_t num_blocks,
                  int max_blocks_per_seq, int max_context_len, float scale, int kv, float k_scale, float v_scale) {
    if (num_seqs < 0 || num_heads <= 0 || num_kv_heads <= 0 || num_heads % num_kv_heads != 0 ||
        max_context_len < 0 || max_blocks_per_seq <= 0 || num_blocks <= 0 || !std::isfinite(scale) || !(scale > 0.f))
        return PA_ERR_INVALID_ARG;
    const int G = num_heads / num_kv_heads;
    if ((head_dim != 64 && head_dim != 128) || (block_size != 8 && block_size != 16 && block_size != 32) || G > 16)
        return PA_ERR_UNSUPPORTED;
    if (const int e = check_kv(kv, head_dim, k_scale, v_scale)) return e;
    if (num_seqs == 0) return NOTHING_TO_DO;
    if (!out || !query || !k_cache || !v_cache || !block_tables || !context_lens || (grouped && !shared_len))
        return PA_ERR_INVALID_ARG;
    if (!aligned16(out) || !aligned16(query) || !aligned16(k_cache) || !aligned16(v_cache))
        return PA_ERR_INVALID_ARG;
    if ((long long)num_blocks * num_kv_heads * block_size >= (1LL << 31)) return PA_ERR_UNSUPPORTED;
    return PA_OK;
}

// One decode call; lead/shared_len are null for pa_decode.
int decode_impl(uint16_t *out, const uint16_t *query, const void *k_cache, const void *v_cache,
                const int32_t *block_tables, const int32_t *context_lens, const int32_t *lead,
                const int32_t *shared_len, int num_seqs, int num_heads, int num_kv_heads, int head_dim, int block_size,
                int64_t num_blocks, int max_blocks_per_seq, int max_context_len, float scale, int kv, float k_scale,
                float v_scale, void *workspace, size_t workspace_bytes, cudaStream_t st) {
    const bool grouped = lead != nullptr;
    if (const int c = decode_checks(out, query, k_cache, v_cache, block_tables, context_lens, grouped, shared_len,
                                    num_seqs, num_heads, num_kv_heads, head_dim, block_size, num_blocks,
                                    max_blocks_per_seq, max_context_len, scale, kv, k_scale, v_scale))
        return c == NOTHING_TO_DO ? PA_OK : c;
    const int G = num_heads / num_kv_heads;
    const long long rows = (long long)num_blocks * num_kv_heads * block_size;
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
    if (!cache_tensor_map(&tmk, k_cache, rows, head_dim, box_rows, kv) ||
        !cache_tensor_map(&tmv, v_cache, rows, head_dim, box_rows, kv))
        return PA_ERR_CUDA;

    // Shared ranges of a grouped call go to the tensor-core kernel (fp16 cache,
    // head_dim 128, G dividing its 128-row tile), up to 128 / G members per
    // item; the decode kernel then reduces each member's own partitions only.
    const bool tc = grouped && kv == PA_KV_F16 && head_dim == 128 && PF_ROWS % G == 0 && prefill_enabled() &&
                    shared_tc_enabled();
    // up to NARROW_ROWS / G members on the narrow kernel when that is at least 4
    // (only with PA_NARROW_SHARED=1: on the parallel-sampling workload the
    // 128-row kernel is faster)
    const bool tcn = tc && narrow_shared_enabled() && NARROW_ROWS % G == 0 && NARROW_ROWS / G >= 4 &&
                     narrow_usable(PA_KV_F16);
    const int mt = tcn ? NARROW_ROWS / G : tc ? PF_ROWS / G : 0;
    // query rows per decode item: one sequence's G heads, or, for a shared
    // range on this kernel, as many members' G heads as two head tiles hold
    const int NT = (G > 8 || (grouped && !tc)) ? 2 : 1;
    const int ms = grouped && !tc ? (16 / G > 1 ? 16 / G : 1) : 1;

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
    uint16_t *hout = out;

    int4 *sitems = reinterpret_cast<int4 *>(ws + L.ptiles);
    // shared ranges on the tensor cores are cut into longer pieces than the
    // decode partitions: each piece is a tensor-core item with its start-up and
    // epilogue, and each member merges one partial per piece
    const int pts = tc ? L.pt * shared_piece_factor() : L.pt;
    decode_prep_kernel<<<1, PREP_THREADS, 0, st>>>(context_lens, lead, shared_len, num_seqs, num_heads, head_dim,
                                                   num_kv_heads, block_size, max_context_len,
                                                   (long long)max_blocks_per_seq * block_size, L.pt, pts, ms, hdr,
                                                   part_off, gsize, gshared, items, grp, hout, nan_pair(kv), mt,
                                                   sitems);
    if (cudaGetLastError() != cudaSuccess) return PA_ERR_CUDA;
    if (tc) {   // the shared ranges' partial rows, before the decode kernel merges them
        PrefillArgs pa_{};
        pa_.out = hout;
        pa_.query = query;
        pa_.block_tables = block_tables;
        pa_.context_lens = context_lens;
        pa_.query_start = nullptr;
        pa_.tiles = sitems;
        pa_.pairs = nullptr;
        pa_.hdr = hdr;
        pa_.Hq = num_heads;
        pa_.Hkv = num_kv_heads;
        pa_.G = G;
        pa_.bs = block_size;
        pa_.mbps = max_blocks_per_seq;
        pa_.num_blocks = num_blocks;
        pa_.scale_log2 = scale * 1.4426950408889634f;
        pa_.v_scale = 1.f;
        pa_.wait_limit = wait_limit_cycles();
        pa_.part_off = part_off;
        pa_.ws_ml = ws_ml;
        pa_.ws_o = ws_o;
        pa_.pt = pts;
        pa_.scratch = ws + L.nscr;
        const int rc = tcn ? launch_narrow_shared(tmk, tmv, pa_, L.ptile_cap * num_kv_heads, st)
                           : launch_shared_ranges(tmk, tmv, pa_, L.ptile_cap * num_kv_heads, st);
        if (rc != PA_OK) return rc;
    }

    DecodeArgs args;
    args.out = hout;
    args.query = query;
    args.block_tables = block_tables;
    args.context_lens = context_lens;
    args.Hq = num_heads;
    args.Hkv = num_kv_heads;
    args.G = G;
    args.bs = block_size;
    args.mbps = max_blocks_per_seq;
    args.pt = L.pt;
    args.pts = pts;
    args.ms = ms;
    args.num_blocks = num_blocks;
    args.wait_limit = wait_limit_cycles();
    args.scale_log2 = scale * (kv == PA_KV_FP8_E4M3 ? k_scale : 1.f) * 1.4426950408889634f;
    args.v_scale = kv == PA_KV_FP8_E4M3 ? v_scale : 1.f;
    args.tc_shared = tc ? 1 : 0;
    args.hdr = hdr;
    args.part_off = part_off;
    args.items = items;
    args.grp = grp;
    args.ws_ml = ws_ml;
    args.ws_o = ws_o;
    const long long max_items = L.item_cap * num_kv_heads;
    return launch_kv_any(kv, head_dim, NT, false, tmk, tmv, args, max_items, st);
}

// One multi-token (causal) call.
int causal_impl(uint16_t *out, const uint16_t *query, const void *k_cache, const void *v_cache,
                const int32_t *block_tables, const int32_t *context_lens, const int32_t *query_start, int num_seqs,
                int num_query_tokens, int num_heads, int num_kv_heads, int head_dim, int block_size,
                int64_t num_blocks, int max_blocks_per_seq, int max_context_len, float scale, int kv, float k_scale,
                float v_scale, void *workspace, size_t workspace_bytes, cudaStream_t st) {
    if (num_seqs < 0 || num_query_tokens < 0 || num_heads <= 0 || num_kv_heads <= 0 ||
        num_heads % num_kv_heads != 0 || max_context_len < 0 || max_blocks_per_seq <= 0 || num_blocks <= 0 ||
        !std::isfinite(scale) || !(scale > 0.f))
        return PA_ERR_INVALID_ARG;
    const int G = num_heads / num_kv_heads;
    if ((head_dim != 64 && head_dim != 128) || (block_size != 8 && block_size != 16 && block_size != 32) || G > 16)
        return PA_ERR_UNSUPPORTED;
    if (const int e = check_kv(kv, head_dim, k_scale, v_scale)) return e;
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
    if (!cache_tensor_map(&tmk, k_cache, rows, head_dim, box_rows, kv) ||
        !cache_tensor_map(&tmv, v_cache, rows, head_dim, box_rows, kv))
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
    uint16_t *hout = out;
    // sequences with many new tokens go to the tensor-core prefill kernel
    // (head_dim 128, G dividing the 128-row tile; FP8 codes become fp16 tiles on chip)
    const bool pf = prefill_enabled() && head_dim == 128 && PF_ROWS % G == 0 &&
                    (long long)num_query_tokens * G >= PF_MIN_ROWS && prefill_usable(kv);
    int4 *ptiles = reinterpret_cast<int4 *>(ws + L.ptiles);
    int4 *ppairs = reinterpret_cast<int4 *>(ws + L.ppairs);
    // sequences with several row tiles take them two at a time (16-bit caches)
    const bool pairs = pf && kv != PA_KV_FP8_E4M3 && prefill_pairs_enabled() && prefill2_usable(kv);
    // sequences of at most NARROW_ROWS rows go to the narrow kernel
    const bool narrow = pf && narrow_enabled() && narrow_usable(kv);
    int4 *ntiles = reinterpret_cast<int4 *>(ws + L.ntiles);
    causal_prep_kernel<<<1, PREP_THREADS, 0, st>>>(context_lens, query_start, num_seqs, num_query_tokens, num_heads,
                                                   head_dim, num_kv_heads, max_context_len,
                                                   (long long)max_blocks_per_seq * block_size, L.pt, ms, hdr,
                                                   part_off, vlen, gstart, items, grp, hout, nan_pair(kv),
                                                   pf ? PF_MIN_ROWS : 0, ptiles, ppairs, pairs ? 1 : 0,
                                                   narrow ? NARROW_ROWS : 0, ntiles, narrow ? narrow_grid() : 0,
                                                   narrow ? nw_split_area(ws + L.nscr).tickets : nullptr);
    if (cudaGetLastError() != cudaSuccess) return PA_ERR_CUDA;

    DecodeArgs args;
    args.out = hout;
    args.query = query;
    args.block_tables = block_tables;
    args.context_lens = vlen;   // per query row: the positions it sees
    args.Hq = num_heads;
    args.Hkv = num_kv_heads;
    args.G = G;
    args.bs = block_size;
    args.mbps = max_blocks_per_seq;
    args.pt = L.pt;
    args.pts = L.pt;
    args.ms = ms;
    args.num_blocks = num_blocks;
    args.wait_limit = wait_limit_cycles();
    args.scale_log2 = scale * (kv == PA_KV_FP8_E4M3 ? k_scale : 1.f) * 1.4426950408889634f;
    args.v_scale = kv == PA_KV_FP8_E4M3 ? v_scale : 1.f;
    args.tc_shared = 0;
    args.hdr = hdr;
    args.part_off = part_off;
    args.items = items;
    args.grp = grp;
    args.ws_ml = reinterpret_cast<float2 *>(ws + L.ml);
    args.ws_o = reinterpret_cast<float *>(ws + L.o);
    const long long max_items = L.item_cap * num_kv_heads;
    if (!pf) return launch_kv_any(kv, head_dim, PA_CAUSAL_NT, true, tmk, tmv, args, max_items, st);
    PrefillArgs pa_{};
    pa_.out = hout;
    pa_.query = query;
    pa_.block_tables = block_tables;
    pa_.context_lens = context_lens;
    pa_.query_start = query_start;
    pa_.tiles = ptiles;
    pa_.pairs = ppairs;
    pa_.hdr = hdr;
    pa_.Hq = num_heads;
    pa_.Hkv = num_kv_heads;
    pa_.G = G;
    pa_.bs = block_size;
    pa_.mbps = max_blocks_per_seq;
    pa_.num_blocks = num_blocks;
    pa_.scale_log2 = args.scale_log2;   // with the K scale of an FP8 cache
    pa_.v_scale = args.v_scale;
    pa_.wait_limit = wait_limit_cycles();
    // the tensor-core kernels on `on`: pairs (the long chunks) first, then
    // the narrow items and the sequences of one row tile.  The host does not
    // know which lists are empty; a kernel with none still claims a whole SM
    // per CTA while it starts, so an empty one launched ahead of a busy one
    // waits for the decode pipeline's CTAs on the side stream to leave the SMs
    // and the busy one with it.  Of the narrow and one-tile lists, the one more
    // likely to be empty goes last: the narrow kernel first when sequences
    // average at most NARROW_ROWS query rows, otherwise after the one-tile
    // kernel (ahead of it, empty, it cost the chunked-prefill step 4 %).
    const bool narrow_first = (long long)num_query_tokens * G <= (long long)NARROW_ROWS * num_seqs;
    auto tensor_core = [&](cudaStream_t on) {
        if (pairs) {
            const int rc2 = launch_prefill2(kv, tmk, tmv, pa_, (L.ptile_cap + 1) / 2 * num_kv_heads, on);
            if (rc2 != PA_OK) return rc2;
        }
        auto narrow_launch = [&]() {
            PrefillArgs na = pa_;
            na.tiles = ntiles;
            na.scratch = ws + L.nscr;
            return launch_narrow(kv, tmk, tmv, na, narrow_grid(), on);
        };
        if (narrow && narrow_first) {
            const int rcn = narrow_launch();
            if (rcn != PA_OK) return rcn;
        }
        const int rc1 = launch_prefill(kv, tmk, tmv, pa_, L.ptile_cap * num_kv_heads, on);
        if (rc1 != PA_OK || !narrow || narrow_first) return rc1;
        return narrow_launch();
    };
    int dev = -1;
    Side *side = cudaGetDevice(&dev) == cudaSuccess ? side_of(dev) : nullptr;
    if (!side) {   // one stream: the decode pipeline, then the tensor-core kernels
        const int rc = launch_kv_any(kv, head_dim, PA_CAUSAL_NT, true, tmk, tmv, args, max_items, st);
        return rc != PA_OK ? rc : tensor_core(st);
    }
    std::lock_guard<std::mutex> lock(side->mu);
    if (cudaEventRecord(side->fork, st) != cudaSuccess) return PA_ERR_CUDA;   // after the prep kernel
    int rc = tensor_core(st);
    if (rc != PA_OK) return rc;
    if (cudaStreamWaitEvent(side->stream, side->fork, 0) != cudaSuccess) return PA_ERR_CUDA;
    rc = launch_kv_any(kv, head_dim, PA_CAUSAL_NT, true, tmk, tmv, args, max_items, side->stream);
    if (cudaEventRecord(side->join, side->stream) != cudaSuccess ||
        cudaStreamWaitEvent(st, side->join, 0) != cudaSuccess)
        return PA_ERR_CUDA;
    return rc;
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
                       scale, PA_KV_F16, 1.f, 1.f, workspace, workspace_bytes, static_cast<cudaStream_t>(stream));
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
                       scale, PA_KV_F16, 1.f, 1.f, workspace, workspace_bytes, static_cast<cudaStream_t>(stream));
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
                       max_blocks_per_seq, max_context_len, scale, PA_KV_F16, 1.f, 1.f, workspace, workspace_bytes,
                       static_cast<cudaStream_t>(stream));
}

extern "C" int pa_decode_typed(void *out, const void *query, const void *k_cache, const void *v_cache,
                               const int32_t *block_tables, const int32_t *context_lens, int num_seqs, int num_heads,
                               int num_kv_heads, int head_dim, int block_size, int64_t num_blocks,
                               int max_blocks_per_seq, int max_context_len, float scale, int kv_dtype, float k_scale,
                               float v_scale, void *workspace, size_t workspace_bytes, void *stream) {
    return decode_impl(static_cast<uint16_t *>(out), static_cast<const uint16_t *>(query), k_cache, v_cache,
                       block_tables, context_lens, nullptr, nullptr, num_seqs, num_heads, num_kv_heads, head_dim,
                       block_size, num_blocks, max_blocks_per_seq, max_context_len, scale, kv_dtype, k_scale, v_scale,
                       workspace, workspace_bytes, static_cast<cudaStream_t>(stream));
}

extern "C" int pa_attention_causal_typed(void *out, const void *query, const void *k_cache, const void *v_cache,
                                         const int32_t *block_tables, const int32_t *context_lens,
                                         const int32_t *query_start, int num_seqs, int num_query_tokens,
                                         int num_heads, int num_kv_heads, int head_dim, int block_size,
                                         int64_t num_blocks, int max_blocks_per_seq, int max_context_len, float scale,
                                         int kv_dtype, float k_scale, float v_scale, void *workspace,
                                         size_t workspace_bytes, void *stream) {
    return causal_impl(static_cast<uint16_t *>(out), static_cast<const uint16_t *>(query), k_cache, v_cache,
                       block_tables, context_lens, query_start, num_seqs, num_query_tokens, num_heads, num_kv_heads,
                       head_dim, block_size, num_blocks, max_blocks_per_seq, max_context_len, scale, kv_dtype, k_scale,
                       v_scale, workspace, workspace_bytes, static_cast<cudaStream_t>(stream));
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
    // pa_decode's own argument checks first, so that both calls report the same status
    const int c = decode_checks(out, query, k_cache, v_cache, block_tables, context_lens, false, nullptr, num_seqs,
                                num_heads, num_kv_heads, head_dim, block_size, num_blocks, max_blocks_per_seq,
                                max_context_len, scale, PA_KV_F16, 1.f, 1.f);
    if (c < 0) return c;
    if (ws_layout(num_seqs, num_heads, num_kv_heads, head_dim, max_context_len, false).total >
        (size_t)PA_DECODE_STATIC_WS_BYTES)
        return PA_ERR_WORKSPACE;
    if (c == NOTHING_TO_DO) return PA_OK;
    int device = -1;
    if (cudaGetDevice(&device) != cudaSuccess) return PA_ERR_CUDA;
    void *ws = static_ws_address(device);
    if (!ws) return PA_ERR_CUDA;
    return pa_decode(out, query, k_cache, v_cache, block_tables, context_lens, num_seqs, num_heads, num_kv_heads,
                     head_dim, block_size, num_blocks, max_blocks_per_seq, max_context_len, scale, ws,
                     (size_t)PA_DECODE_STATIC_WS_BYTES, stream);
}

extern "C" int pa_decode_static_ws_status(int *status_out, void *stream) {
    if (!status_out) return PA_ERR_INVALID_ARG;
    int device = -1;
    if (cudaGetDevice(&device) != cudaSuccess) return PA_ERR_CUDA;
    void *ws = static_ws_address(device);
    if (!ws) return PA_ERR_CUDA;
    return pa_workspace_status(ws, status_out, stream);
}
