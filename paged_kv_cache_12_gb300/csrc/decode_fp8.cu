// The paged attention kernels over a cache of FP8 E4M3 codes (fp16 query and
// output).  A 16-token stage of K or V is half the bytes of the fp16 one; the
// consumer turns each pair of codes into an exact fp16 pair as it builds its
// MMA fragments, folds the K scale into the softmax scale and applies the V
// scale to the output.  What is computed is described in decode.cu; this file
// only instantiates the kernels for this element type (head_dim 128).

#include "decode_common.cuh"

namespace pa {

int launch_kv_fp8(int D, int NT, bool causal, const CUtensorMap &tmk, const CUtensorMap &tmv,
                  const DecodeArgs &args, long long max_items, cudaStream_t st) {
    return launch_kv<PA_KV_FP8_E4M3>(D, NT, causal, tmk, tmv, args, max_items, st);
}

}  // namespace pa
