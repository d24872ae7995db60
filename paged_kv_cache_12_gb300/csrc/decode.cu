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
// How (three launches on the caller's stream):
//  1. decode_prep_kernel (one CTA): splits every sequence into partitions of
//     PART_TOKENS tokens, writes the compact list of (sequence, partition)
//     work items into the workspace, zeroes the work counter, and writes the
//     rows of empty (zero) and invalid (NaN) sequences.
//  2. decode_kernel (persistent, one warp = one independent pipeline):
//     each warp takes work items (sequence, partition, kv head) from an atomic
//     counter.  For an item it streams 16-token chunks of the K and V tiles
//     through a DEPTH-deep ring of shared-memory stages with TMA (2-D tiled
//     copies through a tensor map over the cache, 128-byte swizzle), the
//     gather being the per-chunk TMA y coordinate taken from the block table.
//     The G query heads of the kv head ride on the M dimension of
//     m16n8k16 tensor-core MMAs: S = Q K^T (heads x tokens) and O += P V,
//     with ldmatrix from the swizzled tiles (bank-conflict free) and an
//     online softmax in fp32 registers.  Each KV tile is read from HBM once
//     for the whole group.  A single-partition sequence writes its fp16
//     output directly; otherwise the item writes (m, l, unnormalised o) to
//     the workspace.
//  3. decode_merge_kernel: log-sum-exp merge of the partitions of every
//     multi-partition sequence: M = max m_p, w_p = 2^(m_p - M),
//     out = sum_p w_p o_p / sum_p w_p l_p.
//
// Results do not depend on the physical placement, on the block size or on
// which warp ran which item: every item is reduced by one warp in a fixed
// chunk order, and the merge runs over partitions in order.

#include <cudaTypedefs.h>

#include <cmath>
#include <mutex>
#include <vector>

#include "common.cuh"

namespace pa {
namespace {

constexpr int PART_TOKENS = 512;       // tokens per partition (one work item)
constexpr int CHUNK = 16;              // tokens per pipeline stage
constexpr int NWARPS = 2;              // independent warps per CTA
constexpr int DEPTH = 4;               // pipeline stages per warp
constexpr long long WAIT_LIMIT = 1LL << 31;   // clock cycles (about a second)
constexpr int PREP_THREADS = 1024;

struct WsHeader {
    int error;
    int total_items;
    int counter;
    int pad[61];
};
static_assert(sizeof(WsHeader) == 256, "header is one 256-byte line");

struct WsLayout {
    size_t part_off, sp_info, ml, o, total;
    int pmax;
};

inline size_t up256(size_t x) { return (x + 255) & ~size_t(255); }

WsLayout ws_layout(int B, int Hq, int D, int max_ctx) {
    WsLayout w;
    w.pmax = max_ctx > 0 ? (max_ctx + PART_TOKENS - 1) / PART_TOKENS : 1;
    size_t off = sizeof(WsHeader);
    w.part_off = off;
    off += up256(sizeof(int) * ((size_t)B + 1));
    w.sp_info = off;
    off += up256(sizeof(int4) * (size_t)B * w.pmax);
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
    int Hq, Hkv, G, bs, mbps;
    long long num_blocks;
    float scale_log2;
    WsHeader *hdr;
    const int4 *sp_info;
    float2 *ws_ml;
    float *ws_o;
};

struct StageMeta {
    int chunk, ntok, qslot, flags;     // flags: 1 = first chunk of the item, 2 = last
};
struct ItemInfo {
    int seq, kvh, sp, P, bad, pad0, pad1, pad2;
};

template <int D, int GPAD>
struct Cfg {
    static constexpr int BOXES = D / 64;                  // 64-column (128-byte) boxes per tile row
    static constexpr int TILE = BOXES * CHUNK * 128;      // one 16-token K or V tile
    static constexpr int STAGE = 2 * TILE;                // K tile then V tile
    static constexpr int QSLOT = GPAD * D * 2;
    static constexpr int DATA = DEPTH * STAGE + 2 * QSLOT;   // per warp, multiple of 1024
    static constexpr int CTRL = 256;                      // per warp: barriers, stage meta, item info
    static constexpr int SMEM = NWARPS * (DATA + CTRL) + 1024;
    static_assert(DATA % 1024 == 0, "stages must stay 1024-byte aligned for the 128-byte swizzle");
    static_assert(DEPTH * 8 + DEPTH * 16 + 2 * 32 <= CTRL, "control block too small");
};

// Address of 16-byte column `col` (0 .. D/8-1) of row `row` of a swizzled
// tile: 64-column boxes of CHUNK rows x 128 bytes, chunk j of row r stored at
// position j ^ (r & 7) (the TMA 128-byte swizzle).
__device__ __forceinline__ uint32_t swz(uint32_t tile, int row, int col) {
    return tile + (uint32_t)((col >> 3) * (CHUNK * 128) + row * 128 + (((col & 7) ^ (row & 7)) << 4));
}

// -------------------------------------------------------------- prep

__global__ void __launch_bounds__(PREP_THREADS) decode_prep_kernel(
    const int32_t *__restrict__ context_lens, int B, int Hq, int D, int Hkv, int max_ctx, long long max_table_tokens,
    WsHeader *hdr, int *part_off, int4 *sp_info, __half *out) {
    __shared__ int warp_sums[PREP_THREADS / 32];
    __shared__ int running;
    const int lane = threadIdx.x & 31, wid = threadIdx.x >> 5;
    if (threadIdx.x == 0) running = 0;
    __syncthreads();
    for (int base = 0; base < B; base += PREP_THREADS) {
        const int i = base + threadIdx.x;
        int L = 0, P = 0, code = 0;   // code 1: zero row, 2: NaN row
        if (i < B) {
            L = context_lens[i];
            if (L < 0 || L > max_ctx || (long long)L > max_table_tokens)
                code = 2;
            else if (L == 0)
                code = 1;
            else
                P = (L + PART_TOKENS - 1) / PART_TOKENS;
        }
        int x = P;
#pragma unroll
        for (int o = 1; o < 32; o <<= 1) {
            const int y = __shfl_up_sync(0xffffffffu, x, o);
            if (lane >= o) x += y;
        }
        if (lane == 31) warp_sums[wid] = x;
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
        const int excl = running + (wid ? warp_sums[wid - 1] : 0) + x - P;
        if (i < B) {
            part_off[i] = excl;
            for (int p = 0; p < P; ++p) sp_info[excl + p] = make_int4(i, p, L, P);
            if (code) {
                const uint32_t h = code == 1 ? 0u : 0x7e007e00u;
                uint4 fill = make_uint4(h, h, h, h);
                uint4 *row = reinterpret_cast<uint4 *>(out + (long long)i * Hq * D);
                for (int k = 0; k < Hq * D / 8; ++k) row[k] = fill;
            }
        }
        __syncthreads();
        if (threadIdx.x == 0) running += warp_sums[PREP_THREADS / 32 - 1];
        __syncthreads();
    }
    if (threadIdx.x == 0) {
        part_off[B] = running;
        hdr->total_items = running * Hkv;
        hdr->counter = 0;
        hdr->error = 0;
    }
}

// ------------------------------------------------------------ decode

template <int D, int GPAD>
__global__ void __launch_bounds__(NWARPS * 32) decode_kernel(const __grid_constant__ CUtensorMap tmk,
                                                             const __grid_constant__ CUtensorMap tmv,
                                                             const DecodeArgs a) {
    using C = Cfg<D, GPAD>;
    constexpr bool TWO = GPAD == 16;             // query heads 8..15 of the group present
    constexpr int KS = D / 16;                    // k-steps of Q K^T
    constexpr int ND = D / 8;                     // n-tiles of P V
    constexpr int NA = TWO ? 4 : 2;               // accumulator registers per n-tile
    extern __shared__ uint8_t smem_raw[];
    const int lane = threadIdx.x & 31, warp = threadIdx.x >> 5;
    const int r = lane >> 2, c = lane & 3;        // mma fragment row / column pair

    uint8_t *smem = reinterpret_cast<uint8_t *>((reinterpret_cast<uintptr_t>(smem_raw) + 1023) & ~uintptr_t(1023));
    uint8_t *wdata = smem + warp * C::DATA;
    uint8_t *wctrl = smem + NWARPS * C::DATA + warp * C::CTRL;
    const uint32_t sdata = smem_u32(wdata);
    uint64_t *bars = reinterpret_cast<uint64_t *>(wctrl);
    StageMeta *meta = reinterpret_cast<StageMeta *>(wctrl + DEPTH * 8);
    ItemInfo *info = reinterpret_cast<ItemInfo *>(wctrl + DEPTH * 8 + DEPTH * 16);
    const uint32_t qslot0 = sdata + DEPTH * C::STAGE;

    if (lane == 0) {
        for (int s = 0; s < DEPTH; ++s) mbar_init(smem_u32(&bars[s]), 1);
        fence_mbar_init();
    }
    __syncwarp();

    const int total = a.hdr->total_items;
    const uint64_t pol = policy_evict_first();
    const int box_rows = a.bs < CHUNK ? a.bs : CHUNK;

    // ---- issue side: the item being issued (c_*) and the prefetched next one (n_*)
    int n_item = -1, n_seq = 0, n_p = 0, n_L = 0, n_P = 0, n_fb = 0, n_tb0 = -1, n_tb1 = -1;
    auto fetch_next = [&]() {
        int j = 0;
        if (lane == 0) j = atomicAdd(&a.hdr->counter, 1);
        j = __shfl_sync(0xffffffffu, j, 0);
        if (j >= total) {
            n_item = -1;
            return;
        }
        n_item = j;
        const int4 inf = a.sp_info[j / a.Hkv];
        n_seq = inf.x;
        n_p = inf.y;
        n_L = inf.z;
        n_P = inf.w;
        const int t0 = n_p * PART_TOKENS;
        const int t1 = min(n_L, t0 + PART_TOKENS);
        n_fb = t0 / a.bs;
        const int nb = (t1 + a.bs - 1) / a.bs - n_fb;
        const int32_t *row = a.block_tables + (long long)n_seq * a.mbps + n_fb;
        n_tb0 = lane < nb ? row[lane] : -1;
        n_tb1 = lane + 32 < nb ? row[lane + 32] : -1;
    };

    int c_seq = 0, c_kvh = 0, c_t0 = 0, c_t1 = 0, c_fb = 0, c_tb0 = -1, c_tb1 = -1;
    int c_chunk = 0, c_nchunks = 0, c_qslot = 0;
    int started = 0, in_flight = 0, issued = 0, computed = 0;
    bool done_issuing = false;

    fetch_next();

    // ---- compute side
    float m0 = -INFINITY, l0 = 0.f, m1 = -INFINITY, l1 = 0.f;
    float acc[ND][TWO ? 4 : 2];
    uint32_t qf[KS][TWO ? 4 : 2];
#pragma unroll
    for (int n = 0; n < ND; ++n)
#pragma unroll
        for (int e = 0; e < (TWO ? 4 : 2); ++e) acc[n][e] = 0.f;
#pragma unroll
    for (int k = 0; k < KS; ++k)
#pragma unroll
        for (int e = 0; e < (TWO ? 4 : 2); ++e) qf[k][e] = 0u;

    while (true) {
        // -------- fill the ring
        while (!done_issuing && issued - computed < DEPTH) {
            if (c_chunk == c_nchunks) {
                if (in_flight == 2) break;           // both query slots busy
                if (n_item < 0) {
                    done_issuing = true;
                    break;
                }
                const int sp = n_item / a.Hkv;
                c_kvh = n_item - sp * a.Hkv;
                c_seq = n_seq;
                c_t0 = n_p * PART_TOKENS;
                c_t1 = min(n_L, c_t0 + PART_TOKENS);
                c_fb = n_fb;
                c_tb0 = n_tb0;
                c_tb1 = n_tb1;
                c_chunk = 0;
                c_nchunks = (c_t1 - c_t0 + CHUNK - 1) / CHUNK;
                c_qslot = started & 1;
                ++started;
                ++in_flight;
                if (lane == 0) {
                    ItemInfo ii;
                    ii.seq = n_seq;
                    ii.kvh = c_kvh;
                    ii.sp = sp;
                    ii.P = n_P;
                    ii.bad = 0;
                    ii.pad0 = ii.pad1 = ii.pad2 = 0;
                    info[c_qslot] = ii;
                }
                fetch_next();
            }
            const int s = issued % DEPTH;
            const int tok0 = c_t0 + c_chunk * CHUNK;
            const int ntok = min(CHUNK, c_t1 - tok0);
            const int lb0 = tok0 / a.bs - c_fb;
            const int phys0 = __shfl_sync(0xffffffffu, lb0 < 32 ? c_tb0 : c_tb1, lb0 & 31);
            const bool two_blocks = a.bs < CHUNK && ntok > a.bs;
            const int lb1 = lb0 + 1;
            const int phys1 = __shfl_sync(0xffffffffu, lb1 < 32 ? c_tb0 : c_tb1, lb1 & 31);
            if (lane == 0) {
                const bool bad = phys0 < 0 || phys0 >= a.num_blocks ||
                                 (two_blocks && (phys1 < 0 || phys1 >= a.num_blocks));
                const bool first = c_chunk == 0;
                const bool last = c_chunk == c_nchunks - 1;
                uint32_t bytes = 0;
                if (!bad) bytes = 2u * C::BOXES * box_rows * 128u * (two_blocks ? 2u : 1u);
                if (first) bytes += (uint32_t)(a.G * D * 2);
                StageMeta mt;
                mt.chunk = c_chunk;
                mt.ntok = ntok;
                mt.qslot = c_qslot;
                mt.flags = (first ? 1 : 0) | (last ? 2 : 0);
                meta[s] = mt;
                if (bad) info[c_qslot].bad = 1;
                const uint32_t bar = smem_u32(&bars[s]);
                const uint32_t kdst = sdata + s * C::STAGE;
                const uint32_t vdst = kdst + C::TILE;
                mbar_arrive_expect_tx(bar, bytes);
                if (!bad) {
                    const int row0 = tok0 % a.bs;
                    const int y0 = (int)(((long long)phys0 * a.Hkv + c_kvh) * a.bs + row0);
#pragma unroll
                    for (int b = 0; b < C::BOXES; ++b) {
                        tma_load_2d(kdst + b * CHUNK * 128, &tmk, 64 * b, y0, bar, pol);
                        tma_load_2d(vdst + b * CHUNK * 128, &tmv, 64 * b, y0, bar, pol);
                    }
                    if (two_blocks) {
                        const int y1 = (int)(((long long)phys1 * a.Hkv + c_kvh) * a.bs);
#pragma unroll
                        for (int b = 0; b < C::BOXES; ++b) {
                            tma_load_2d(kdst + b * CHUNK * 128 + a.bs * 128, &tmk, 64 * b, y1, bar, pol);
                            tma_load_2d(vdst + b * CHUNK * 128 + a.bs * 128, &tmv, 64 * b, y1, bar, pol);
                        }
                    }
                }
                if (first) {
                    const __half *qsrc = a.query + ((long long)c_seq * a.Hq + (long long)c_kvh * a.G) * D;
                    bulk_load(qslot0 + c_qslot * C::QSLOT, qsrc, (uint32_t)(a.G * D * 2), bar);
                }
            }
            ++c_chunk;
            ++issued;
        }
        __syncwarp();
        if (computed == issued) break;

        // -------- compute one stage
        const int s = computed % DEPTH;
        if (!mbar_wait_bounded(smem_u32(&bars[s]), (uint32_t)((computed / DEPTH) & 1), WAIT_LIMIT)) {
            if (lane == 0) atomicExch(&a.hdr->error, PA_ERR_TIMEOUT);
            // let this warp's other copies land (bounded) before leaving
            for (int k = computed + 1; k < issued; ++k)
                mbar_wait_bounded(smem_u32(&bars[k % DEPTH]), (uint32_t)((k / DEPTH) & 1), WAIT_LIMIT >> 4);
            return;
        }
        const StageMeta mt = meta[s];
        const uint32_t kt = sdata + s * C::STAGE;
        const uint32_t vt = kt + C::TILE;

        if (mt.flags & 1) {   // new item: load the group's query rows, reset the running state
            const __half *q = reinterpret_cast<const __half *>(wdata + DEPTH * C::STAGE + mt.qslot * C::QSLOT);
#pragma unroll
            for (int k = 0; k < KS; ++k) {
                qf[k][0] = *reinterpret_cast<const uint32_t *>(q + r * D + 16 * k + 2 * c);
                qf[k][1] = *reinterpret_cast<const uint32_t *>(q + r * D + 16 * k + 8 + 2 * c);
                if constexpr (TWO) {
                    qf[k][TWO ? 2 : 0] = *reinterpret_cast<const uint32_t *>(q + (r + 8) * D + 16 * k + 2 * c);
                    qf[k][TWO ? 3 : 0] = *reinterpret_cast<const uint32_t *>(q + (r + 8) * D + 16 * k + 8 + 2 * c);
                }
            }
            m0 = m1 = -INFINITY;
            l0 = l1 = 0.f;
#pragma unroll
            for (int n = 0; n < ND; ++n)
#pragma unroll
                for (int e = 0; e < (TWO ? 4 : 2); ++e) acc[n][e] = 0.f;
        }

        // S = Q K^T for the 16 tokens of the chunk: two n-tiles of 8 tokens
        float sc[2][4];
#pragma unroll
        for (int nt = 0; nt < 2; ++nt) {
            sc[nt][0] = sc[nt][1] = sc[nt][2] = sc[nt][3] = 0.f;
#pragma unroll
            for (int kp = 0; kp < D / 32; ++kp) {
                uint32_t b0, b1, b2, b3;
                ldmatrix_x4(swz(kt, nt * 8 + (lane & 7), kp * 4 + (lane >> 3)), b0, b1, b2, b3);
#pragma unroll
                for (int h2 = 0; h2 < 2; ++h2) {
                    const int k = 2 * kp + h2;
                    uint32_t a1 = 0u, a3 = 0u;
                    if constexpr (TWO) {
                        a1 = qf[k][TWO ? 2 : 0];
                        a3 = qf[k][TWO ? 3 : 0];
                    }
                    float d2, d3;
                    mma_16816(sc[nt][0], sc[nt][1], d2, d3, qf[k][0], a1, qf[k][1], a3, h2 ? b2 : b0, h2 ? b3 : b1,
                              sc[nt][0], sc[nt][1], sc[nt][2], sc[nt][3]);
                    if constexpr (TWO) {
                        sc[nt][2] = d2;
                        sc[nt][3] = d3;
                    }
                }
            }
        }

        // online softmax (base 2), rows r and r + 8
        const int ntok = mt.ntok;
        const float sl2 = a.scale_log2;
#pragma unroll
        for (int nt = 0; nt < 2; ++nt)
#pragma unroll
            for (int e = 0; e < 4; ++e) {
                const int tok = nt * 8 + 2 * c + (e & 1);
                sc[nt][e] = tok < ntok ? sc[nt][e] * sl2 : -INFINITY;
            }
        uint32_t pa0, pa1 = 0u, pa2, pa3 = 0u;
        {
            float mx = fmaxf(fmaxf(sc[0][0], sc[0][1]), fmaxf(sc[1][0], sc[1][1]));
            mx = fmaxf(mx, __shfl_xor_sync(0xffffffffu, mx, 1));
            mx = fmaxf(mx, __shfl_xor_sync(0xffffffffu, mx, 2));
            const float mn = fmaxf(m0, mx);
            const float alpha = exp2f(m0 - mn);
            const float p00 = exp2f(sc[0][0] - mn), p01 = exp2f(sc[0][1] - mn);
            const float p10 = exp2f(sc[1][0] - mn), p11 = exp2f(sc[1][1] - mn);
            l0 = l0 * alpha + ((p00 + p01) + (p10 + p11));
            m0 = mn;
#pragma unroll
            for (int n = 0; n < ND; ++n) {
                acc[n][0] *= alpha;
                acc[n][1] *= alpha;
            }
            pa0 = pack_half2(p00, p01);
            pa2 = pack_half2(p10, p11);
        }
        if constexpr (TWO) {
            float mx = fmaxf(fmaxf(sc[0][2], sc[0][3]), fmaxf(sc[1][2], sc[1][3]));
            mx = fmaxf(mx, __shfl_xor_sync(0xffffffffu, mx, 1));
            mx = fmaxf(mx, __shfl_xor_sync(0xffffffffu, mx, 2));
            const float mn = fmaxf(m1, mx);
            const float alpha = exp2f(m1 - mn);
            const float p00 = exp2f(sc[0][2] - mn), p01 = exp2f(sc[0][3] - mn);
            const float p10 = exp2f(sc[1][2] - mn), p11 = exp2f(sc[1][3] - mn);
            l1 = l1 * alpha + ((p00 + p01) + (p10 + p11));
            m1 = mn;
#pragma unroll
            for (int n = 0; n < ND; ++n) {
                acc[n][TWO ? 2 : 0] *= alpha;
                acc[n][TWO ? 3 : 0] *= alpha;
            }
            pa1 = pack_half2(p00, p01);
            pa3 = pack_half2(p10, p11);
        }

        // O += P V: V^T fragments by transposing ldmatrix; masked tokens zeroed
        // so that stale or poisoned slots past the context never reach O
        uint32_t vmask_lo = 0xffffffffu, vmask_hi = 0xffffffffu;
        if (ntok < CHUNK) {
            vmask_lo = (2 * c < ntok ? 0x0000ffffu : 0u) | (2 * c + 1 < ntok ? 0xffff0000u : 0u);
            vmask_hi = (2 * c + 8 < ntok ? 0x0000ffffu : 0u) | (2 * c + 9 < ntok ? 0xffff0000u : 0u);
        }
#pragma unroll
        for (int np = 0; np < D / 16; ++np) {
            const int mi = lane >> 3;
            uint32_t v0, v1, v2, v3;
            ldmatrix_x4_trans(swz(vt, ((mi & 1) << 3) + (lane & 7), 2 * np + (mi >> 1)), v0, v1, v2, v3);
            v0 &= vmask_lo;
            v2 &= vmask_lo;
            v1 &= vmask_hi;
            v3 &= vmask_hi;
#pragma unroll
            for (int h2 = 0; h2 < 2; ++h2) {
                const int n = 2 * np + h2;
                float c2 = 0.f, c3 = 0.f, d2, d3;
                if constexpr (TWO) {
                    c2 = acc[n][TWO ? 2 : 0];
                    c3 = acc[n][TWO ? 3 : 0];
                }
                mma_16816(acc[n][0], acc[n][1], d2, d3, pa0, pa1, pa2, pa3, h2 ? v2 : v0, h2 ? v3 : v1, acc[n][0],
                          acc[n][1], c2, c3);
                if constexpr (TWO) {
                    acc[n][TWO ? 2 : 0] = d2;
                    acc[n][TWO ? 3 : 0] = d3;
                }
            }
        }

        if (mt.flags & 2) {   // item complete: write it out
            const ItemInfo ii = info[mt.qslot];
            float lr0 = l0 + __shfl_xor_sync(0xffffffffu, l0, 1);
            lr0 += __shfl_xor_sync(0xffffffffu, lr0, 2);
            float lr1 = 0.f;
            if constexpr (TWO) {
                lr1 = l1 + __shfl_xor_sync(0xffffffffu, l1, 1);
                lr1 += __shfl_xor_sync(0xffffffffu, lr1, 2);
            }
            const float nanf_ = __int_as_float(0x7fc00000);
#pragma unroll
            for (int half_ = 0; half_ < (TWO ? 2 : 1); ++half_) {
                const int row = r + 8 * half_;
                if (row < a.G) {
                    const int h = ii.kvh * a.G + row;
                    const float lr = half_ ? lr1 : lr0;
                    const float mrow = half_ ? m1 : m0;
                    if (ii.P == 1) {
                        const float inv = ii.bad ? nanf_ : 1.f / lr;
                        __half *orow = a.out + ((long long)ii.seq * a.Hq + h) * D;
#pragma unroll
                        for (int n = 0; n < ND; ++n)
                            *reinterpret_cast<uint32_t *>(orow + 8 * n + 2 * c) =
                                pack_half2(acc[n][(2 * half_) % NA] * inv, acc[n][(2 * half_ + 1) % NA] * inv);
                    } else {
                        const long long wrow = (long long)ii.sp * a.Hq + h;
                        float *orow = a.ws_o + wrow * D;
#pragma unroll
                        for (int n = 0; n < ND; ++n)
                            *reinterpret_cast<float2 *>(orow + 8 * n + 2 * c) =
                                ii.bad ? make_float2(nanf_, nanf_)
                                       : make_float2(acc[n][(2 * half_) % NA], acc[n][(2 * half_ + 1) % NA]);
                        if (c == 0) a.ws_ml[wrow] = ii.bad ? make_float2(nanf_, nanf_) : make_float2(mrow, lr);
                    }
                }
            }
            --in_flight;
        }
        __syncwarp();
        fence_proxy_async_smem();   // this stage's reads before the next TMA write into it
        ++computed;
    }
}

// ------------------------------------------------------------- merge

template <int D>
__global__ void __launch_bounds__(256) decode_merge_kernel(const int *__restrict__ part_off,
                                                           const float2 *__restrict__ ws_ml,
                                                           const float *__restrict__ ws_o, __half *__restrict__ out,
                                                           int B, int Hq) {
    constexpr int PER = D / 32;   // elements per lane
    const long long row = (long long)blockIdx.x * (blockDim.x / 32) + (threadIdx.x >> 5);
    const int lane = threadIdx.x & 31;
    if (row >= (long long)B * Hq) return;
    const int seq = (int)(row / Hq), h = (int)(row % Hq);
    const int p0 = part_off[seq];
    const int P = part_off[seq + 1] - p0;
    if (P <= 1) return;
    float M = -INFINITY;
    for (int p = 0; p < P; ++p) M = fmaxf(M, ws_ml[(long long)(p0 + p) * Hq + h].x);
    float acc[PER];
#pragma unroll
    for (int e = 0; e < PER; ++e) acc[e] = 0.f;
    float lsum = 0.f;
    for (int p = 0; p < P; ++p) {
        const long long wrow = (long long)(p0 + p) * Hq + h;
        const float2 ml = ws_ml[wrow];
        const float w = exp2f(ml.x - M);
        lsum += w * ml.y;
        const float *o = ws_o + wrow * D + lane * PER;
        if constexpr (PER == 4) {
            const float4 v = *reinterpret_cast<const float4 *>(o);
            acc[0] += w * v.x;
            acc[1] += w * v.y;
            acc[2] += w * v.z;
            acc[3] += w * v.w;
        } else {
            const float2 v = *reinterpret_cast<const float2 *>(o);
            acc[0] += w * v.x;
            acc[1] += w * v.y;
        }
    }
    const float inv = 1.f / lsum;
    __half *orow = out + ((long long)seq * Hq + h) * D + lane * PER;
#pragma unroll
    for (int e = 0; e < PER; e += 2)
        *reinterpret_cast<uint32_t *>(orow + e) = pack_half2(acc[e] * inv, acc[e + 1] * inv);
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

struct Launch {
    int grid = 0;
};

template <int D, int GPAD>
int launch_decode(const CUtensorMap &tmk, const CUtensorMap &tmv, const DecodeArgs &args, cudaStream_t st) {
    using C = Cfg<D, GPAD>;
    static int grid = 0;
    static std::once_flag once;
    static cudaError_t init_err = cudaSuccess;
    std::call_once(once, [] {
        init_err = cudaFuncSetAttribute(decode_kernel<D, GPAD>, cudaFuncAttributeMaxDynamicSharedMemorySize, C::SMEM);
        if (init_err != cudaSuccess) return;
        int dev = 0, sms = 0, per_sm = 0;
        init_err = cudaGetDevice(&dev);
        if (init_err == cudaSuccess) init_err = cudaDeviceGetAttribute(&sms, cudaDevAttrMultiProcessorCount, dev);
        if (init_err == cudaSuccess)
            init_err = cudaOccupancyMaxActiveBlocksPerMultiprocessor(&per_sm, decode_kernel<D, GPAD>, NWARPS * 32,
                                                                     C::SMEM);
        if (init_err == cudaSuccess) grid = sms * (per_sm > 0 ? per_sm : 1);
    });
    if (init_err != cudaSuccess || grid <= 0) return PA_ERR_CUDA;
    decode_kernel<D, GPAD><<<grid, NWARPS * 32, C::SMEM, st>>>(tmk, tmv, args);
    return cuda_status(cudaGetLastError());
}

}  // namespace
}  // namespace pa

using namespace pa;

extern "C" size_t pa_decode_workspace_size(int num_seqs, int num_heads, int head_dim, int max_context_len) {
    if (num_seqs < 0 || num_heads <= 0 || head_dim <= 0 || max_context_len < 0) return 0;
    return ws_layout(num_seqs, num_heads, head_dim, max_context_len).total;
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
        max_context_len < 0 || max_blocks_per_seq <= 0 || num_blocks <= 0 || !std::isfinite(scale))
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
    const WsLayout L = ws_layout(num_seqs, num_heads, head_dim, max_context_len);
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
    float2 *ws_ml = reinterpret_cast<float2 *>(ws + L.ml);
    float *ws_o = reinterpret_cast<float *>(ws + L.o);
    __half *hout = reinterpret_cast<__half *>(out);

    decode_prep_kernel<<<1, PREP_THREADS, 0, st>>>(context_lens, num_seqs, num_heads, head_dim, num_kv_heads,
                                                   max_context_len, (long long)max_blocks_per_seq * block_size, hdr,
                                                   part_off, sp_info, hout);
    cudaError_t e = cudaGetLastError();
    if (e != cudaSuccess) return PA_ERR_CUDA;

    DecodeArgs args;
    args.out = hout;
    args.query = reinterpret_cast<const __half *>(query);
    args.block_tables = block_tables;
    args.Hq = num_heads;
    args.Hkv = num_kv_heads;
    args.G = G;
    args.bs = block_size;
    args.mbps = max_blocks_per_seq;
    args.num_blocks = num_blocks;
    args.scale_log2 = scale * 1.4426950408889634f;
    args.hdr = hdr;
    args.sp_info = sp_info;
    args.ws_ml = ws_ml;
    args.ws_o = ws_o;
    int rc;
    if (head_dim == 128)
        rc = G <= 8 ? launch_decode<128, 8>(tmk, tmv, args, st) : launch_decode<128, 16>(tmk, tmv, args, st);
    else
        rc = G <= 8 ? launch_decode<64, 8>(tmk, tmv, args, st) : launch_decode<64, 16>(tmk, tmv, args, st);
    if (rc != PA_OK) return rc;

    if (L.pmax > 1) {
        const long long rows_out = (long long)num_seqs * num_heads;
        const int per_cta = 8;
        const unsigned grid = (unsigned)((rows_out + per_cta - 1) / per_cta);
        if (head_dim == 128)
            decode_merge_kernel<128><<<grid, 32 * per_cta, 0, st>>>(part_off, ws_ml, ws_o, hout, num_seqs, num_heads);
        else
            decode_merge_kernel<64><<<grid, 32 * per_cta, 0, st>>>(part_off, ws_ml, ws_o, hout, num_seqs, num_heads);
        if (cudaGetLastError() != cudaSuccess) return PA_ERR_CUDA;
    }
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
    if (num_seqs < 0 || num_heads <= 0 || head_dim <= 0 || max_context_len < 0) return PA_ERR_INVALID_ARG;
    if (ws_layout(num_seqs, num_heads, head_dim, max_context_len).total > (size_t)PA_DECODE_STATIC_WS_BYTES)
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
