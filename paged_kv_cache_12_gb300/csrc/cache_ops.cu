// KV write (scatter of new K/V rows into their slots) and block copy (the
// copy half of copy-on-write) for the paged cache
// [num_blocks][num_kv_heads][block_size][head_dim] of 16-bit elements (fp16 or
// bf16), and the quantising write into a cache of one-byte FP8 E4M3 codes.
//
// Both are pure data movement: every thread moves 16-byte vectors, K and V in
// the same thread, and every index read from the device is range-checked
// before it is used as an address.
//
// Sources: the new token goes into the free slot of the sequence's current
// block ("PagedAttention : comment optimiser la memoire GPU lors de
// l'inference des LLM", deeplearn.tn, section "Un exemple concret
// d'allocation", steps 2-4); a writer that finds a shared block copies it
// first ("PagedAttention de vLLM : comment la gestion de la VRAM soutient
// l'inference des grands modeles", deepsonar.com.cn, section 2.3).

#include <algorithm>
#include <cmath>
#include <vector>

#include "common.cuh"

namespace pa {
namespace {

// Eight fp16 values -> eight E4M3 codes (first value in the lowest byte).
__device__ __forceinline__ uint2 quantise8(uint4 x, float inv) {
    const uint32_t w[4] = {x.x, x.y, x.z, x.w};
    uint32_t c[4];
#pragma unroll
    for (int k = 0; k < 4; ++k) {
        const float2 f = __half22float2(*reinterpret_cast<const __half2 *>(&w[k]));
        const float2 y = make_float2(__fmul_rn(f.x, inv), __fmul_rn(f.y, inv));
        c[k] = static_cast<uint32_t>(__nv_cvt_float2_to_fp8x2(y, __NV_SATFINITE, __NV_E4M3));
    }
    return make_uint2(c[0] | (c[1] << 16), c[2] | (c[3] << 16));
}

// One thread per (token, kv head, 16-byte column vector).
__global__ void kv_write_kernel(const uint4 *__restrict__ key, const uint4 *__restrict__ value,
                                const int64_t *__restrict__ slot_mapping, uint4 *__restrict__ k_cache,
                                uint4 *__restrict__ v_cache, int num_tokens, int num_kv_heads, int vecs_per_row,
                                int block_size, long long num_slots) {
    const long long total = (long long)num_tokens * num_kv_heads * vecs_per_row;
    for (long long i = blockIdx.x * (long long)blockDim.x + threadIdx.x; i < total;
         i += (long long)gridDim.x * blockDim.x) {
        const int v = (int)(i % vecs_per_row);
        const long long th = i / vecs_per_row;   // token * num_kv_heads + head
        const int h = (int)(th % num_kv_heads);
        const long long t = th / num_kv_heads;
        const long long slot = slot_mapping[t];
        if (slot < 0 || slot >= num_slots) continue;
        const long long blk = slot / block_size;
        const long long off = slot - blk * block_size;
        const long long dst = ((blk * num_kv_heads + h) * block_size + off) * vecs_per_row + v;
        k_cache[dst] = key[i];
        v_cache[dst] = value[i];
    }
}

// The same scatter into FP8 E4M3 caches: one thread per (token, kv head,
// 8 elements); each fp16 element x is stored as the code of fl32(x * inv),
// rounded to the nearest E4M3 value (ties to even) and saturated at +-448,
// inv = fl32(1 / scale) computed once on the host.
__global__ void kv_write_fp8_kernel(const uint4 *__restrict__ key, const uint4 *__restrict__ value,
                                    const int64_t *__restrict__ slot_mapping, uint2 *__restrict__ k_cache,
                                    uint2 *__restrict__ v_cache, int num_tokens, int num_kv_heads, int vecs_per_row,
                                    int block_size, long long num_slots, float kinv, float vinv) {
    const long long total = (long long)num_tokens * num_kv_heads * vecs_per_row;
    for (long long i = blockIdx.x * (long long)blockDim.x + threadIdx.x; i < total;
         i += (long long)gridDim.x * blockDim.x) {
        const int v = (int)(i % vecs_per_row);
        const long long th = i / vecs_per_row;
        const int h = (int)(th % num_kv_heads);
        const long long t = th / num_kv_heads;
        const long long slot = slot_mapping[t];
        if (slot < 0 || slot >= num_slots) continue;
        const long long blk = slot / block_size;
        const long long off = slot - blk * block_size;
        const long long dst = ((blk * num_kv_heads + h) * block_size + off) * vecs_per_row + v;
        k_cache[dst] = quantise8(key[i], kinv);
        v_cache[dst] = quantise8(value[i], vinv);
    }
}

// blockIdx.y = pair; the block's vectors are strided over blockIdx.x.
__global__ void block_copy_kernel(uint4 *__restrict__ k_cache, uint4 *__restrict__ v_cache,
                                  const int64_t *__restrict__ pairs, long long vecs_per_block,
                                  long long num_blocks) {
    const long long src = pairs[2 * (long long)blockIdx.y];
    const long long dst = pairs[2 * (long long)blockIdx.y + 1];
    if (src < 0 || src >= num_blocks || dst < 0 || dst >= num_blocks) return;
    const uint4 *ks = k_cache + src * vecs_per_block;
    const uint4 *vs = v_cache + src * vecs_per_block;
    uint4 *kd = k_cache + dst * vecs_per_block;
    uint4 *vd = v_cache + dst * vecs_per_block;
    for (long long i = blockIdx.x * (long long)blockDim.x + threadIdx.x; i < vecs_per_block;
         i += (long long)gridDim.x * blockDim.x) {
        const uint4 a = ks[i];
        const uint4 b = vs[i];
        kd[i] = a;
        vd[i] = b;
    }
}

// PA_DEBUG_VALIDATE: every slot below num_slots, no slot written twice.
int validate_slots(const int64_t *slot_mapping, int num_tokens, long long num_slots, cudaStream_t st) {
    std::vector<int64_t> h((size_t)num_tokens);
    if (cudaMemcpyAsync(h.data(), slot_mapping, sizeof(int64_t) * num_tokens, cudaMemcpyDeviceToHost, st) !=
            cudaSuccess ||
        cudaStreamSynchronize(st) != cudaSuccess)
        return PA_ERR_CUDA;
    std::vector<int64_t> seen;
    seen.reserve(h.size());
    for (int64_t s : h) {
        if (s >= num_slots) return PA_ERR_INVALID_ARG;
        if (s >= 0) seen.push_back(s);
    }
    std::sort(seen.begin(), seen.end());
    for (size_t i = 1; i < seen.size(); ++i)
        if (seen[i] == seen[i - 1]) return PA_ERR_INVALID_ARG;
    return 0;
}

// SM count of the current device, asked on every call (a cheap attribute
// query), so that each device sizes its own grid.  The kernels stride over
// their work, so the count only sets the grid cap.
int num_sms() {
    int dev = 0, n = 0;
    if (cudaGetDevice(&dev) != cudaSuccess || cudaDeviceGetAttribute(&n, cudaDevAttrMultiProcessorCount, dev) !=
                                                  cudaSuccess || n <= 0)
        return 148;
    return n;
}

}  // namespace
}  // namespace pa

using namespace pa;

extern "C" int pa_kv_write(const uint16_t *key, const uint16_t *value, const int64_t *slot_mapping,
                           uint16_t *k_cache, uint16_t *v_cache, int num_tokens, int num_kv_heads, int head_dim,
                           int block_size, int64_t num_blocks, void *stream) {
    if (num_tokens < 0 || num_kv_heads <= 0 || head_dim <= 0 || head_dim % 8 != 0 || block_size <= 0 ||
        num_blocks <= 0)
        return PA_ERR_INVALID_ARG;
    if (num_tokens == 0) return PA_OK;
    if (!key || !value || !slot_mapping || !k_cache || !v_cache) return PA_ERR_INVALID_ARG;
    if (!aligned16(key) || !aligned16(value) || !aligned16(k_cache) || !aligned16(v_cache))
        return PA_ERR_INVALID_ARG;
    cudaStream_t st = static_cast<cudaStream_t>(stream);
    const long long num_slots = (long long)num_blocks * block_size;
    if (debug_validate())
        if (const int e = validate_slots(slot_mapping, num_tokens, num_slots, st)) return e;
    const int vecs = head_dim / 8;
    const long long total = (long long)num_tokens * num_kv_heads * vecs;
    const int threads = 256;
    long long blocks = (total + threads - 1) / threads;
    const long long cap = (long long)num_sms() * 16;
    if (blocks > cap) blocks = cap;
    kv_write_kernel<<<(unsigned)blocks, threads, 0, st>>>(
        reinterpret_cast<const uint4 *>(key), reinterpret_cast<const uint4 *>(value), slot_mapping,
        reinterpret_cast<uint4 *>(k_cache), reinterpret_cast<uint4 *>(v_cache), num_tokens, num_kv_heads, vecs,
        block_size, num_slots);
    return cuda_status(cudaGetLastError());
}

extern "C" int pa_block_copy(uint16_t *k_cache, uint16_t *v_cache, const int64_t *pairs, int num_pairs,
                             int num_kv_heads, int head_dim, int block_size, int64_t num_blocks, void *stream) {
    if (num_pairs < 0 || num_kv_heads <= 0 || head_dim <= 0 || head_dim % 8 != 0 || block_size <= 0 ||
        num_blocks <= 0)
        return PA_ERR_INVALID_ARG;
    if (num_pairs == 0) return PA_OK;
    if (!k_cache || !v_cache || !pairs || !aligned16(k_cache) || !aligned16(v_cache)) return PA_ERR_INVALID_ARG;
    if (num_pairs > 65535) return PA_ERR_UNSUPPORTED;
    cudaStream_t st = static_cast<cudaStream_t>(stream);
    if (debug_validate()) {
        std::vector<int64_t> h((size_t)num_pairs * 2);
        if (cudaMemcpyAsync(h.data(), pairs, sizeof(int64_t) * h.size(), cudaMemcpyDeviceToHost, st) !=
                cudaSuccess ||
            cudaStreamSynchronize(st) != cudaSuccess)
            return PA_ERR_CUDA;
        std::vector<int64_t> srcs, dsts;
        for (int i = 0; i < num_pairs; ++i) {
            int64_t s = h[2 * i], d = h[2 * i + 1];
            if (s < 0 || s >= num_blocks || d < 0 || d >= num_blocks) return PA_ERR_INVALID_ARG;
            srcs.push_back(s);
            dsts.push_back(d);
        }
        std::sort(srcs.begin(), srcs.end());
        std::sort(dsts.begin(), dsts.end());
        for (size_t i = 1; i < dsts.size(); ++i)
            if (dsts[i] == dsts[i - 1]) return PA_ERR_INVALID_ARG;
        for (int64_t d : dsts)
            if (std::binary_search(srcs.begin(), srcs.end(), d)) return PA_ERR_INVALID_ARG;
    }
    const long long vecs_per_block = (long long)num_kv_heads * block_size * head_dim / 8;
    const int threads = 256;
    long long gx = (vecs_per_block + threads - 1) / threads;
    if (gx > 64) gx = 64;
    dim3 grid((unsigned)gx, (unsigned)num_pairs);
    block_copy_kernel<<<grid, threads, 0, st>>>(reinterpret_cast<uint4 *>(k_cache),
                                                reinterpret_cast<uint4 *>(v_cache), pairs, vecs_per_block,
                                                (long long)num_blocks);
    return cuda_status(cudaGetLastError());
}

extern "C" int pa_kv_write_fp8(const uint16_t *key, const uint16_t *value, const int64_t *slot_mapping,
                               uint8_t *k_cache, uint8_t *v_cache, int num_tokens, int num_kv_heads, int head_dim,
                               int block_size, int64_t num_blocks, float k_scale, float v_scale, void *stream) {
    if (num_tokens < 0 || num_kv_heads <= 0 || head_dim <= 0 || head_dim % 8 != 0 || block_size <= 0 ||
        num_blocks <= 0 || !std::isfinite(k_scale) || !(k_scale > 0.f) || !std::isfinite(v_scale) ||
        !(v_scale > 0.f))
        return PA_ERR_INVALID_ARG;
    if (num_tokens == 0) return PA_OK;
    if (!key || !value || !slot_mapping || !k_cache || !v_cache) return PA_ERR_INVALID_ARG;
    if (!aligned16(key) || !aligned16(value) || !aligned16(k_cache) || !aligned16(v_cache))
        return PA_ERR_INVALID_ARG;
    cudaStream_t st = static_cast<cudaStream_t>(stream);
    const long long num_slots = (long long)num_blocks * block_size;
    if (debug_validate())
        if (const int e = validate_slots(slot_mapping, num_tokens, num_slots, st)) return e;
    const int vecs = head_dim / 8;
    const long long total = (long long)num_tokens * num_kv_heads * vecs;
    const int threads = 256;
    long long blocks = (total + threads - 1) / threads;
    const long long cap = (long long)num_sms() * 16;
    if (blocks > cap) blocks = cap;
    const float kinv = 1.0f / k_scale, vinv = 1.0f / v_scale;   // IEEE float division, once
    kv_write_fp8_kernel<<<(unsigned)blocks, threads, 0, st>>>(
        reinterpret_cast<const uint4 *>(key), reinterpret_cast<const uint4 *>(value), slot_mapping,
        reinterpret_cast<uint2 *>(k_cache), reinterpret_cast<uint2 *>(v_cache), num_tokens, num_kv_heads, vecs,
        block_size, num_slots, kinv, vinv);
    return cuda_status(cudaGetLastError());
}

extern "C" int pa_block_copy_typed(void *k_cache, void *v_cache, const int64_t *pairs, int num_pairs,
                                   int num_kv_heads, int head_dim, int block_size, int64_t num_blocks, int kv_dtype,
                                   void *stream) {
    if (kv_dtype == PA_KV_FP8_E4M3) {   // one-byte elements: a block is half as many 16-bit words
        if (head_dim % 16 != 0) return PA_ERR_INVALID_ARG;
        return pa_block_copy(static_cast<uint16_t *>(k_cache), static_cast<uint16_t *>(v_cache), pairs, num_pairs,
                             num_kv_heads, head_dim / 2, block_size, num_blocks, stream);
    }
    if (kv_dtype != PA_KV_F16 && kv_dtype != PA_KV_BF16) return PA_ERR_INVALID_ARG;
    return pa_block_copy(static_cast<uint16_t *>(k_cache), static_cast<uint16_t *>(v_cache), pairs, num_pairs,
                         num_kv_heads, head_dim, block_size, num_blocks, stream);
}
