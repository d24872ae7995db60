/*
 * pa.h -- C ABI of the paged KV cache decode path (GB300, sm_103a).
 *
 * One shared library, libpa.so, exports everything declared here.  Plain C
 * types only: fp16 tensors are passed as pointers to their IEEE binary16 bit
 * patterns (uint16_t), CUDA streams as void* (a cudaStream_t; NULL is the
 * legacy default stream).
 *
 * Conventions for every call that touches the GPU
 *  - All tensor pointers are DEVICE pointers owned by the caller; tensors are
 *    dense and row-major in the shapes stated.  The library allocates no
 *    device memory: scratch space is the caller's workspace buffer.
 *  - Work is enqueued on `stream` and the call returns without waiting for
 *    it.  Argument checks that need no device data run on the host before any
 *    launch; a failed check returns PA_ERR_INVALID_ARG (or
 *    PA_ERR_UNSUPPORTED / PA_ERR_WORKSPACE) and launches nothing.  A launch
 *    failure returns PA_ERR_CUDA.
 *  - Values that live on the device (slot numbers, block ids, context
 *    lengths) are checked by the kernels: an entry out of range is never
 *    dereferenced.  What happens instead is stated per call.
 *  - With the environment variable PA_DEBUG_VALIDATE=1 the calls also copy
 *    their device-side index arguments to the host (synchronising `stream`)
 *    and return PA_ERR_INVALID_ARG on any out-of-range or conflicting entry.
 *  - No exception crosses this boundary.
 *
 * Cache layout (the pages fix none; this library's choice): k_cache and
 * v_cache are fp16 [num_blocks][num_kv_heads][block_size][head_dim].  Token
 * slot s lives in physical block s / block_size at offset s % block_size, so
 * every (block, kv head) tile is one contiguous block_size x head_dim run.
 *
 * Sources: "PagedAttention de vLLM : comment la gestion de la VRAM soutient
 * l'inference des grands modeles" (deepsonar.com.cn) sections 2.1-2.4, 2.6 and
 * VII; "PagedAttention : comment optimiser la memoire GPU lors de l'inference
 * des LLM" (deeplearn.tn), sections "Comment fonctionne PagedAttention", "Un
 * exemple concret d'allocation", "La table de blocs en arriere-plan";
 * "vLLM transforme la memoire GPU en systeme d'exploitation pour LLM"
 * (chester-dev.com), section "PagedAttention transforme l'historique en blocs
 * reutilisables".
 */
#ifndef PA_H
#define PA_H

#include <stddef.h>
#include <stdint.h>

#if defined(__GNUC__)
#define PA_API __attribute__((visibility("default")))
#else
#define PA_API
#endif

#ifdef __cplusplus
extern "C" {
#endif

/* ---------------------------------------------------------------- status */

enum {
    PA_OK = 0,
    PA_ERR_INVALID_ARG = -1,   /* a bad shape, pointer, id or index */
    PA_ERR_OUT_OF_BLOCKS = -2, /* the free queue cannot cover the request; nothing changed */
    PA_ERR_STATE = -3,         /* allocator bookkeeping found an inconsistency */
    PA_ERR_WORKSPACE = -4,     /* workspace missing, misaligned or too small */
    PA_ERR_CUDA = -5,          /* a CUDA runtime call or launch failed */
    PA_ERR_UNSUPPORTED = -6,   /* valid but not built: head_dim, block_size or group size;
                                * also a decode kernel whose compiled register count
                                * is not the one its register split was sized for
                                * (a build of other sources or another compiler; it
                                * is never launched then) */
    PA_ERR_TIMEOUT = -7        /* a kernel gave up waiting on its own copies (see pa_workspace_status) */
};

/* Element type of the K and V caches (the "typed" calls below).  The pages
 * keep the cache in fp16 (deepsonar page section 2.1: two bytes per element
 * in the cache-size count); bf16 keeps two bytes, fp8 E4M3 halves them.
 *   PA_KV_F16       fp16 cache; fp16 query and output
 *   PA_KV_BF16      bf16 cache; bf16 query and output
 *   PA_KV_FP8_E4M3  one-byte FP8 E4M3 codes (OCP format); fp16 query and
 *                   output; a K code c stands for e4m3(c) * k_scale, a V code
 *                   for e4m3(c) * v_scale (one scale per cache, host floats) */
enum {
    PA_KV_F16 = 0,
    PA_KV_BF16 = 1,
    PA_KV_FP8_E4M3 = 2
};

/* Static text for a status code (never NULL). */
PA_API const char *pa_status_string(int status);

/* Library ABI version, currently 1. */
PA_API int pa_version(void);

/* ------------------------------------------------------------- KV write */

/* Scatter the K/V rows of new tokens into their cache slots.
 *
 * The new token's K and V go into the free slot the allocator reserved for
 * it in the sequence's current block (deeplearn.tn page, "Un exemple concret
 * d'allocation", steps 2-4):
 *   k_cache[slot / block_size][h][slot % block_size][:] = key[t][h][:]
 *   v_cache[...same...]                                   = value[t][h][:]
 * for every token t with slot = slot_mapping[t] and every kv head h.
 *
 *   key, value     fp16 [num_tokens][num_kv_heads][head_dim]
 *   slot_mapping   int64 [num_tokens]; slot < 0 marks padding and is skipped;
 *                  slot >= num_blocks * block_size is skipped as well
 *                  (PA_DEBUG_VALIDATE reports it).  Two tokens with the same
 *                  slot in one call are a caller error (either row may win).
 *   k_cache, v_cache  fp16 caches in the layout above, num_blocks blocks.
 *   head_dim       a multiple of 8 (16-byte rows); block_size >= 1.
 * num_tokens = 0 is valid and launches nothing. */
PA_API int pa_kv_write(const uint16_t *key, const uint16_t *value, const int64_t *slot_mapping,
                uint16_t *k_cache, uint16_t *v_cache,
                int num_tokens, int num_kv_heads, int head_dim, int block_size,
                int64_t num_blocks, void *stream);

/* -------------------------------------------------------- block copy */

/* Copy whole blocks (all kv heads, all offsets, K and V): the copy half of
 * copy-on-write (deepsonar page section 2.3: a writer that finds a block
 * shared copies it first, then writes).
 *
 *   pairs      int64 [num_pairs][2] = (src_block, dst_block)
 * Destinations must be distinct and no destination may also be a source in
 * the same call; a source may repeat.  Pairs with an id outside
 * [0, num_blocks) are skipped (PA_DEBUG_VALIDATE reports them and any
 * conflict).  num_pairs = 0 is valid and launches nothing.
 * head_dim must be a multiple of 8. */
PA_API int pa_block_copy(uint16_t *k_cache, uint16_t *v_cache, const int64_t *pairs, int num_pairs,
                  int num_kv_heads, int head_dim, int block_size, int64_t num_blocks,
                  void *stream);

/* ------------------------------------------------------------ decode */

/* Bytes of device workspace pa_decode needs for these sizes (a host-side
 * bound; the same value for any context lengths up to max_context_len).
 * Returns 0 for invalid sizes. */
PA_API size_t pa_decode_workspace_size(int num_seqs, int num_heads, int num_kv_heads, int head_dim,
                                       int max_context_len);

/* Single-token decode attention over the paged cache.
 *
 * For each sequence i with L = context_lens[i] tokens (the token written this
 * step included) and each query head h, with G = num_heads / num_kv_heads and
 * kv head g = h / G (groups of G consecutive query heads share one kv head,
 * deepsonar page section 2.1):
 *   token t (t < L) is gathered from physical block block_tables[i][t / block_size]
 *   at offset t % block_size (deepsonar page section 2.2; deeplearn.tn page
 *   "La table de blocs en arriere-plan"),
 *   s_t = scale * <query[i][h], K_t[g]>,
 *   out[i][h] = sum_t softmax(s)_t * V_t[g].
 * The context is processed in partitions of PT tokens, PT the largest of
 * 1024, 512 and 256 for which num_seqs * num_kv_heads *
 * ceil(max_context_len / PT) >= 4096 * max(1, 8 / G), G = num_heads /
 * num_kv_heads (256 if none); a sequence longer than one partition is
 * finished by a log-sum-exp merge of its partitions.  PT depends on these
 * host-side sizes only.
 * Arithmetic: fp16 inputs, fp32 accumulation, fp16 output.
 *
 *   out            fp16 [num_seqs][num_heads][head_dim]
 *   query          fp16 [num_seqs][num_heads][head_dim]
 *   k_cache, v_cache  fp16 caches, layout above, num_blocks blocks; 16-byte aligned.
 *   block_tables   int32 [num_seqs][max_blocks_per_seq]
 *   context_lens   int32 [num_seqs]
 *   head_dim in {64, 128}; block_size in {8, 16, 32};
 *   num_heads % num_kv_heads == 0 and 1 <= G <= 16.
 *   max_context_len  host-side upper bound on every context_lens[i]; it sizes
 *                  the workspace and needs no device read.
 *   workspace      device buffer of at least pa_decode_workspace_size(...)
 *                  bytes, 256-byte aligned, used only for the duration of
 *                  the work on `stream`.
 * Device-side cases: L = 0 gives a zero output row.  L < 0,
 * L > max_context_len or L > max_blocks_per_seq * block_size gives a NaN
 * output row.  A block id outside [0, num_blocks) is never read; the
 * partition that met it writes NaN.  Results are deterministic: the same
 * inputs give the same bits, whatever the physical placement of the blocks
 * and whatever the block size.  scale must be positive and finite. */
PA_API int pa_decode(uint16_t *out, const uint16_t *query,
              const uint16_t *k_cache, const uint16_t *v_cache,
              const int32_t *block_tables, const int32_t *context_lens,
              int num_seqs, int num_heads, int num_kv_heads, int head_dim, int block_size,
              int64_t num_blocks, int max_blocks_per_seq, int max_context_len, float scale,
              void *workspace, size_t workspace_bytes, void *stream);

/* ------------------------------------------- decode with shared prefixes */

/* Workspace bytes pa_decode_shared_prefix needs (a host-side bound). */
PA_API size_t pa_decode_shared_prefix_workspace_size(int num_seqs, int num_heads, int num_kv_heads, int head_dim,
                                                     int max_context_len);

/* pa_decode for a batch in which groups of sequences share the physical
 * blocks of a common prefix (parallel sampling or beam search over one
 * prompt: deepsonar page section 2.3; a prompt shared by several requests:
 * deeplearn.tn page, "Les benefices concrets a l'usage").  A shared block is
 * then read from HBM and reduced once for several members together (up to
 * 16 query rows, i.e. 16 / G members, per pass) instead of once per member.
 * Same arguments as pa_decode, plus two device int32 arrays of num_seqs:
 *   group_leader[i]  the first sequence of i's group (i itself when it leads
 *                    a group or shares nothing).  A group is the run of
 *                    consecutive sequences, starting at its leader, that all
 *                    name that leader; a sequence outside its leader's run is
 *                    treated as sharing nothing.
 *   shared_len[i]    read at leaders only: tokens at the start of every
 *                    member's context that live in the same physical blocks
 *                    (the first shared_len / block_size table entries of all
 *                    members are equal).  Rounded down to whole blocks and
 *                    capped by the shortest member's context; 0 = no sharing.
 * The caller guarantees the equal table entries (PA_DEBUG_VALIDATE checks
 * them).  The result is the same attention as pa_decode's (the partitioning
 * differs, so the bits may differ within the fp32 rounding).  Workspace:
 * pa_decode_shared_prefix_workspace_size. */
PA_API int pa_decode_shared_prefix(uint16_t *out, const uint16_t *query, const uint16_t *k_cache,
                                   const uint16_t *v_cache, const int32_t *block_tables,
                                   const int32_t *context_lens, const int32_t *group_leader,
                                   const int32_t *shared_len, int num_seqs, int num_heads, int num_kv_heads,
                                   int head_dim, int block_size, int64_t num_blocks, int max_blocks_per_seq,
                                   int max_context_len, float scale, void *workspace, size_t workspace_bytes,
                                   void *stream);

/* --------------------------------- several new tokens per sequence (causal) */

/* Workspace bytes pa_attention_causal needs (a host-side bound). */
PA_API size_t pa_attention_causal_workspace_size(int num_seqs, int num_query_tokens, int num_heads,
                                                 int num_kv_heads, int head_dim, int max_context_len);

/* Attention for a step in which a sequence computes several new tokens at
 * once: a chunk of a long prompt (chunked prefill), the rest of a prompt after
 * a prefix-cache hit, or speculative candidate tokens (deepsonar page section
 * 2.5: the scheduler gives each request a token budget per step).  The new
 * tokens' K and V are already in the cache (pa_kv_write), so sequence i has
 * L = context_lens[i] positions, the last T = query_start[i + 1] -
 * query_start[i] of them new.  New token j (0 <= j < T) is query row
 * query_start[i] + j and attends causally to positions t <= L - T + j:
 *   s_t = scale * <query[row][h], K_t[g]>,  out[row][h] = sum_t softmax(s)_t V_t[g],
 * gather, GQA grouping, partitions, merge and arithmetic as in pa_decode.
 * One token per sequence (query_start = 0, 1, ..., num_seqs) is the decode.
 *
 *   out, query     fp16 [num_query_tokens][num_heads][head_dim]
 *   query_start    int32 [num_seqs + 1], device: 0 = query_start[0] <= ...
 *                  <= query_start[num_seqs] = num_query_tokens (T = 0 allowed)
 *   num_query_tokens  host-side row count of query and out
 *   other arguments as in pa_decode.
 * Two kinds of kernel share the work.  A sequence with more than 16 query
 * rows (T x G) -- a prompt chunk, or a few speculative tokens at a large G --
 * is computed on the 5th-generation tensor cores in tiles of 128 query rows
 * (128 / G new tokens x the G heads of a kv head), each K/V tile read once
 * per tile (head_dim 128, any cache type, G dividing 128; PA_PREFILL=0 in
 * the environment turns this off).  Other sequences take the decode
 * pipeline, which reduces up to 16 / G new tokens of a sequence together, so
 * a KV tile is read once for that many tokens' query rows.  In a call that
 * may send rows to the tensor cores (head_dim 128, G dividing 128, more than
 * 16 query rows in the call), the decode pipeline runs on a stream of the
 * library's own beside the tensor-core kernels (forked from `stream` and joined back into it with
 * events; the first such call on a device creates that stream and its events,
 * so make it before any stream capture; PA_PREFILL_SIDE=0 keeps all work on
 * `stream`).  Device-side cases: a
 * sequence with T > L or an invalid L (as in pa_decode) gets NaN rows; a
 * query_start that is not a non-decreasing cover of [0, num_query_tokens)
 * makes every row NaN.  num_query_tokens = 0 launches nothing.  Workspace:
 * pa_attention_causal_workspace_size, 256-byte aligned.  Deterministic. */
PA_API int pa_attention_causal(uint16_t *out, const uint16_t *query, const uint16_t *k_cache,
                               const uint16_t *v_cache, const int32_t *block_tables, const int32_t *context_lens,
                               const int32_t *query_start, int num_seqs, int num_query_tokens, int num_heads,
                               int num_kv_heads, int head_dim, int block_size, int64_t num_blocks,
                               int max_blocks_per_seq, int max_context_len, float scale, void *workspace,
                               size_t workspace_bytes, void *stream);

/* ----------------------------------------- bf16 and fp8 E4M3 caches (typed) */

/* Quantising KV write into caches of one-byte FP8 E4M3 codes
 * (uint8 [num_blocks][num_kv_heads][block_size][head_dim]).  Each fp16
 * element x of key[t] / value[t] is stored at slot slot_mapping[t] as the
 * code of fl32(x * fl32(1 / scale)) (scale = k_scale or v_scale, the
 * reciprocal taken once in float on the host), rounded to the nearest E4M3
 * value with ties to the even code and saturated at +-448 (NaN stays NaN).
 * Slots as in pa_kv_write.  head_dim a multiple of 8, scales positive and
 * finite.  (A bf16 cache takes bf16 rows through pa_kv_write, which copies
 * 16-bit elements whatever their type.) */
PA_API int pa_kv_write_fp8(const uint16_t *key, const uint16_t *value, const int64_t *slot_mapping,
                           uint8_t *k_cache, uint8_t *v_cache, int num_tokens, int num_kv_heads, int head_dim,
                           int block_size, int64_t num_blocks, float k_scale, float v_scale, void *stream);

/* pa_block_copy for a cache of element type kv_dtype (PA_KV_*); for fp8
 * head_dim must be a multiple of 16. */
PA_API int pa_block_copy_typed(void *k_cache, void *v_cache, const int64_t *pairs, int num_pairs,
                               int num_kv_heads, int head_dim, int block_size, int64_t num_blocks, int kv_dtype,
                               void *stream);

/* pa_decode over a cache of element type kv_dtype (PA_KV_*): out and query
 * are bf16 for PA_KV_BF16, fp16 otherwise.  For PA_KV_FP8_E4M3 a K code c
 * stands for e4m3(c) * k_scale and a V code for e4m3(c) * v_scale (both
 * positive and finite; head_dim 128); the scales are ignored for the 16-bit
 * types.  MMA operands are fp16 (fp8 codes are turned into their exact fp16
 * values) or bf16, accumulation fp32.  Workspace: pa_decode_workspace_size.
 * PA_ERR_UNSUPPORTED for an fp8 cache with head_dim 64. */
PA_API int pa_decode_typed(void *out, const void *query, const void *k_cache, const void *v_cache,
                           const int32_t *block_tables, const int32_t *context_lens, int num_seqs, int num_heads,
                           int num_kv_heads, int head_dim, int block_size, int64_t num_blocks,
                           int max_blocks_per_seq, int max_context_len, float scale, int kv_dtype, float k_scale,
                           float v_scale, void *workspace, size_t workspace_bytes, void *stream);

/* pa_attention_causal over a cache of element type kv_dtype, as
 * pa_decode_typed.  Workspace: pa_attention_causal_workspace_size. */
PA_API int pa_attention_causal_typed(void *out, const void *query, const void *k_cache, const void *v_cache,
                                     const int32_t *block_tables, const int32_t *context_lens,
                                     const int32_t *query_start, int num_seqs, int num_query_tokens, int num_heads,
                                     int num_kv_heads, int head_dim, int block_size, int64_t num_blocks,
                                     int max_blocks_per_seq, int max_context_len, float scale, int kv_dtype,
                                     float k_scale, float v_scale, void *workspace, size_t workspace_bytes,
                                     void *stream);

/* Read the error word a pa_decode call left in its workspace: PA_OK, or
 * PA_ERR_TIMEOUT if a kernel gave up waiting for its own copies into shared
 * memory (the affected outputs are NaN).  Synchronises `stream`. */
PA_API int pa_workspace_status(const void *workspace, int *status_out, void *stream);

/* -------------------------------------------- decode without allocation */

/* Largest scratch area pa_decode_static_ws can use: 64 MiB. */
#define PA_DECODE_STATIC_WS_BYTES (64u << 20)

/* pa_decode for callers that cannot allocate device memory at all.
 *
 * No counterpart in the pages: this is a packaging choice of this library.
 * Some callers may not call cudaMalloc -- for example a plugin that runs
 * inside a host framework which owns every byte of device memory through its
 * own pool (a raw cudaMalloc there goes around the pool, can fail once the
 * pool holds the memory, and may synchronise the device), or a serving loop
 * whose rule is that nothing is allocated after start-up.  Such a caller
 * cannot provide pa_decode's workspace.  This entry point takes the same
 * arguments as pa_decode minus the workspace and uses instead a scratch array
 * of PA_DECODE_STATIC_WS_BYTES that the library declares at file scope in
 * device memory; every GPU that loads the library holds that array until the
 * process exits.  It allocates nothing: no cudaMalloc, no cudaFree, no
 * allocating library routine.
 *
 *  - The first call on a device looks the array's device address up (with
 *    that device current) and keeps it; make that first call before any
 *    stream capture.
 *  - If pa_decode_workspace_size(num_seqs, num_heads, num_kv_heads,
 *    head_dim, max_context_len) exceeds PA_DECODE_STATIC_WS_BYTES the call returns
 *    PA_ERR_WORKSPACE and launches nothing.
 *  - All calls on a device share the one array and it keeps whatever the last
 *    call left there (each call re-initialises what it needs before use).
 *    Calls whose work overlaps on the GPU -- on different streams without
 *    ordering between them -- race on the array and give wrong results:
 *    order them, or use pa_decode with a workspace per stream.
 *  - Arguments are checked as pa_decode checks them, and the same status is
 *    returned; only then is the size checked against the array.
 * Results are identical, bit for bit, to pa_decode's for the same inputs. */
PA_API int pa_decode_static_ws(uint16_t *out, const uint16_t *query,
                               const uint16_t *k_cache, const uint16_t *v_cache,
                               const int32_t *block_tables, const int32_t *context_lens,
                               int num_seqs, int num_heads, int num_kv_heads, int head_dim,
                               int block_size, int64_t num_blocks, int max_blocks_per_seq,
                               int max_context_len, float scale, void *stream);

/* The error word the last pa_decode_static_ws call on the current device left
 * in the library's scratch array, for callers that never see that array's
 * address: PA_OK, or PA_ERR_TIMEOUT if a kernel gave up waiting for its own
 * copies into shared memory (the affected outputs are NaN).  The pages have no
 * counterpart (see pa_decode_static_ws).  Synchronises `stream`; call it on the
 * stream of the decode it asks about.  PA_ERR_CUDA if the array's address
 * cannot be looked up. */
PA_API int pa_decode_static_ws_status(int *status_out, void *stream);

/* Failure-detection self-test.  Every wait of the decode kernel's pipeline
 * is bounded: after about a second it records PA_ERR_TIMEOUT in the
 * workspace (see pa_workspace_status), lets its own copies land and returns,
 * so a stuck pipeline never hangs the GPU.  This call runs that same bounded
 * wait in a one-warp kernel on a barrier that nothing ever completes: after
 * limit_cycles (1 .. 2^31) it must give up and write PA_ERR_TIMEOUT to the
 * device int *status_device.  Asynchronous on `stream`.
 * (PA_WAIT_LIMIT_CYCLES in the environment, read once, replaces the decode
 * pipeline's one-second bound.) */
PA_API int pa_selftest_wait_timeout(long long limit_cycles, int *status_device, void *stream);

/* ------------------------------------------------------ block allocator */

/* Host-side block allocator with reference counts (no GPU involved).
 *
 * Blocks hold block_size tokens.  A sequence takes a new block only when the
 * token to write starts one (allocation on demand, left to right; deepsonar
 * page section 2.2 and section VII step 2), so it never holds more than
 * ceil(len / block_size) blocks.  The free queue hands out from its head and
 * takes released blocks back at its tail, in table order (deepsonar page
 * section 2.4 and section VII step 1).  fork() shares every block of the
 * parent (count + 1).  Writing into a block whose count is above one first
 * takes a fresh block, reports the (shared, fresh) pair for pa_block_copy and
 * drops the shared block's count (deepsonar page section 2.3).
 *
 * Every call returns a status; on any error the allocator is unchanged. */
typedef struct pa_allocator pa_allocator;

typedef struct {
    int64_t num_blocks;
    int64_t free_blocks;
    int64_t used_blocks;     /* count > 0 */
    int64_t shared_blocks;   /* count > 1 */
    int64_t num_seqs;
    int64_t logical_tokens;  /* sum of sequence lengths */
} pa_alloc_stats_t;

/* free_order: optional permutation of [0, num_blocks) giving the initial
 * order of the free queue (NULL = 0, 1, 2, ...). */
PA_API int pa_alloc_create(int64_t num_blocks, int block_size, const int32_t *free_order,
                    pa_allocator **out);
PA_API int pa_alloc_destroy(pa_allocator *a);
PA_API int pa_alloc_add_seq(pa_allocator *a, int64_t seq_id);

/* Reserve slots for the next counts[k] tokens of sequence seq_ids[k], k in
 * order.  slots_out receives sum(counts) slot numbers (sequence by sequence,
 * token by token); pairs_out receives up to pairs_capacity (src, dst) block
 * pairs (int64 [n][2]) that pa_block_copy must copy before the K/V of these
 * tokens are written, and *num_pairs_out their number (at most one per
 * sequence).  All or nothing: PA_ERR_OUT_OF_BLOCKS if the free queue cannot
 * cover the whole call; PA_ERR_INVALID_ARG for an unknown or repeated id, a
 * negative count, or pairs_capacity below the number of pairs needed. */
PA_API int pa_alloc_append(pa_allocator *a, int num_seqs, const int64_t *seq_ids, const int32_t *counts,
                    int64_t *slots_out, int64_t *pairs_out, int pairs_capacity,
                    int *num_pairs_out);
PA_API int pa_alloc_fork(pa_allocator *a, int64_t parent_id, int64_t child_id);
PA_API int pa_alloc_free_seq(pa_allocator *a, int64_t seq_id);
PA_API int pa_alloc_seq_len(const pa_allocator *a, int64_t seq_id, int64_t *len_out);

/* Block tables for num_seqs sequences as int32 [num_seqs][max_blocks] (unused
 * entries -1) and their lengths as int32 [num_seqs]; PA_ERR_INVALID_ARG if a
 * sequence holds more than max_blocks blocks. */
PA_API int pa_alloc_block_tables(const pa_allocator *a, int num_seqs, const int64_t *seq_ids,
                          int32_t *tables_out, int max_blocks, int32_t *lens_out);
/* The free queue, head first: *count_out blocks into blocks_out (int32,
 * capacity entries; PA_ERR_INVALID_ARG if capacity is too small, with
 * *count_out still set). */
PA_API int pa_alloc_free_queue(const pa_allocator *a, int32_t *blocks_out, int64_t capacity, int64_t *count_out);

/* ------------------------------------------------------- prefix caching */

/* Prefix caching of full blocks (deepsonar page section 2.4 and section VII
 * step 5).  Each full block of a sequence whose token ids are known gets the
 * chained hash SHA-256(parent hash || token ids || extra key), where the
 * parent hash is the previous block's (32 zero bytes for the first block),
 * token ids are little-endian int32 and the extra key a little-endian
 * uint64; the first block registered with a hash is the one the map keeps.
 * A released block stays in the map while it waits in the free queue; when
 * it is handed out again from the queue head, its entry is dropped (the
 * queue order is the eviction order). */

/* Turn prefix caching on; only before any sequence exists. */
PA_API int pa_alloc_enable_prefix_cache(pa_allocator *a);

/* Start a new sequence seq_id for a prompt of num_tokens token ids: walk the
 * prompt's full blocks that lie inside its first num_tokens - 1 tokens (the
 * last prompt token is always computed, so that its logits exist), hash each
 * in chain, and take every block found in the map, in order, until the first
 * miss (a hit still in the free queue leaves the queue; its count rises by
 * one).  *cached_tokens_out = tokens now covered (a multiple of block_size);
 * the caller appends the rest with pa_alloc_append_ids.  PA_ERR_INVALID_ARG
 * if prefix caching is off or seq_id exists. */
PA_API int pa_alloc_match_prefix(pa_allocator *a, int64_t seq_id, const int32_t *tokens, int num_tokens,
                                 uint64_t extra_key, int *cached_tokens_out);

/* pa_alloc_append with the token ids of the appended tokens (token_ids:
 * sum(counts) int32, sequence by sequence), so that the blocks they complete
 * are hashed and cached.  A sequence appended to once without ids is never
 * hashed again. */
PA_API int pa_alloc_append_ids(pa_allocator *a, int num_seqs, const int64_t *seq_ids, const int32_t *counts,
                               const int32_t *token_ids, int64_t *slots_out, int64_t *pairs_out,
                               int pairs_capacity, int *num_pairs_out);

/* The hash recorded for a block (32 bytes, zeros if none) and whether the
 * map currently points at this block (*cached_out = 1). */
PA_API int pa_alloc_block_hash(const pa_allocator *a, int64_t block, uint8_t *hash_out, int *cached_out);

/* Blocks in the hash map, block lookups made by pa_alloc_match_prefix, hits. */
PA_API int pa_alloc_prefix_stats(const pa_allocator *a, int64_t *cached_blocks, int64_t *queries, int64_t *hits);

/* SHA-256 (FIPS 180-4) of num_bytes bytes: the hash the prefix cache uses. */
PA_API int pa_sha256(const void *data, size_t num_bytes, uint8_t *digest_out);

/* Reference count of one block (0 if free). */
PA_API int pa_alloc_refcount(const pa_allocator *a, int64_t block, int32_t *count_out);
PA_API int pa_alloc_stats(const pa_allocator *a, pa_alloc_stats_t *out);

#ifdef __cplusplus
}
#endif

#endif /* PA_H */
