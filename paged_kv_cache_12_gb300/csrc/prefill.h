// Paged causal attention for long runs of new tokens on tcgen05 (prefill.cu):
// arguments and launch, used by the multi-token entry points in decode.cu.
#pragma once

#include <cudaTypedefs.h>
#include <stdint.h>

#include "decode_common.cuh"

namespace pa {

struct PrefillArgs {
    uint16_t *out;                    // fp16 (bf16 for a bf16 cache) [num_query_tokens][Hq][128]
    const uint16_t *query;            // same layout
    const int32_t *block_tables;
    const int32_t *context_lens;
    const int32_t *query_start;
    const int4 *tiles;                // one-tile kernel: {sequence, row tile, 0, 0}, longest first
    const int4 *pairs;                // two-tile kernel: {sequence, row tile, the tile before it or -1, 0}
    WsHeader *hdr;                    // error word; pf_items / pf2_items = work items (entries x Hkv)
    int Hq, Hkv, G, bs, mbps;
    long long num_blocks;
    float scale_log2;                 // softmax scale (times the K scale of an FP8 cache) x log2(e)
    float v_scale;                    // V scale of an FP8 cache (1 otherwise)
    long long wait_limit;
    // shared-prefix mode: tiles holds {first member, members, t0, t1} (t0 a
    // multiple of pt), and partial rows go to the decode kernel's workspace
    const int *part_off;
    float2 *ws_ml;
    float *ws_o;
    int pt;
    // narrow kernel: merge scratch, NW_SCRATCH_PER_CTA bytes per CTA
    uint8_t *scratch;
};

// Query rows per work tile, and the smallest number of query rows
// (new tokens x G) for which a sequence goes to the tensor-core kernels: more
// than the 16 rows one decode-pipeline item holds, so that the pipeline never
// reads a sequence's KV range twice (a 3-token speculative step at G = 8, 24
// rows: 1.07 ms as two 16-row items, 0.56 ms on the tensor-core kernel).
#ifndef PA_PF_MIN_ROWS
#define PA_PF_MIN_ROWS 17
#endif
constexpr int PF_ROWS = 128;
constexpr int PF_MIN_ROWS = PA_PF_MIN_ROWS;

// Launch the one-tile prefill kernel on `st` (fp16, bf16 or FP8 E4M3 caches,
// head_dim 128); it reads its item count from the workspace header; max_items
// is a host bound that trims the grid.  tmk / tmv: the caches' tensor maps.
int launch_prefill(int kv, const CUtensorMap &tmk, const CUtensorMap &tmv, const PrefillArgs &args,
                   long long max_items, cudaStream_t st);

// Launch the one-tile kernel in its shared-prefix mode (fp16 cache, head_dim
// 128): each work item is up to 128 / G members of a shared-prefix group over
// one partition [t0, t1) of their shared blocks, all members' query rows in one
// tile, each shared K/V tile read once for all of them.  It writes each
// member's partial row (m, l, unnormalised O) of that partition; the decode
// kernel, launched after it on the same stream, merges them with the
// members' own partitions.  Item count: pf_items in the workspace header.
int launch_shared_ranges(const CUtensorMap &tmk, const CUtensorMap &tmv, const PrefillArgs &args,
                         long long max_items, cudaStream_t st);

// The narrow kernel (narrow.cu): work items of at most NARROW_ROWS query rows
// (new tokens x G of one sequence, or members x G of a shared range), with the
// KV tokens on the MMAs' M side.  launch_narrow: the causal rows of the
// sequences listed in args.tiles ({sequence, 0, 0, 0}; pfn_items in the
// header), any cache type; launch_narrow_shared: the shared-prefix mode of
// launch_shared_ranges (fp16 cache), item count pf_items.
constexpr int NARROW_ROWS = 32;
int launch_narrow(int kv, const CUtensorMap &tmk, const CUtensorMap &tmv, const PrefillArgs &args,
                  long long max_items, cudaStream_t st);
int launch_narrow_shared(const CUtensorMap &tmk, const CUtensorMap &tmv, const PrefillArgs &args,
                         long long max_items, cudaStream_t st);
// Whether the narrow kernel can run for this cache type; checked once.
bool narrow_usable(int kv);

// CTAs the narrow kernel launches (one per SM, at most NW_MAX_CTAS); the
// causal prep kernel splits the items of the last, partial round into pieces
// for this many CTAs.
int narrow_grid();

// Whether the one-tile kernel can run for this cache type (for an FP8 cache:
// built with the register count its register split assumes); checked once.
bool prefill_usable(int kv);

// Whether the two-tile kernel can run for this cache type (fp16 or bf16, and
// built with the register count its register split assumes); checked once.
bool prefill2_usable(int kv);

// Launch the two-tile prefill kernel (fp16 or bf16 caches): each work item is
// two neighbouring row tiles of one sequence and kv head, which share every
// K/V tile the CTA loads.
int launch_prefill2(int kv, const CUtensorMap &tmk, const CUtensorMap &tmv, const PrefillArgs &args,
                    long long max_items, cudaStream_t st);

}  // namespace pa
