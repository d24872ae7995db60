// The paged attention kernels over a bf16 cache (bf16 query and output; MMA
// operands bf16, fp32 accumulation).  What is computed is described in
// decode.cu; this file only instantiates the kernels for this element type.

#include "decode_common.cuh"

namespace pa {

int launch_kv_bf16(int D, int NT, bool causal, const CUtensorMap &tmk, const CUtensorMap &tmv,
                   const DecodeArgs &args, long long max_items, cudaStream_t st) {
    return launch_kv<PA_KV_BF16>(D, NT, causal, tmk, tmv, args, max_items, st);
}

}  // namespace pa
