// decode.cu — paged-KV decode attention: split-KV partitions and their
// log-sum-exp merge in one kernel launch (the kernel is in decode_kernel.cuh).
// Caches with blocks of 16, 32 or 64 tokens are read a page at a time by TMA;
// smaller blocks go to the gather instantiation in decode_gather.cu.
#include "decode_kernel.cuh"

namespace pkv {

pkv_status launch_decode(const DecodeParams& p, int head_dim, pkv_dtype q_dtype,
                         pkv_dtype kv_dtype, const CUtensorMap& tmK, const CUtensorMap& tmV,
                         cudaStream_t stream, bool programmatic) {
  if (p.bs_log2 < 4)
    return launch_decode_gather(p, head_dim, q_dtype, kv_dtype, stream, programmatic);
  return launch_decode_mode<false>(p, head_dim, q_dtype, kv_dtype, tmK, tmV, stream,
                                   programmatic);
}

}  // namespace pkv
