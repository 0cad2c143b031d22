// decode_gather.cu — the decode kernel for caches whose blocks hold fewer
// than 16 tokens (block size 1, "TokenAttention", up to 8): a 16-token page
// is gathered row by row with 16-byte cp.async copies into the same swizzled
// shared-memory layout the TMA path produces, so the page math is shared.
#include "decode_kernel.cuh"

namespace pkv {

pkv_status launch_decode_gather(const DecodeParams& p, int head_dim, pkv_dtype q_dtype,
                                pkv_dtype kv_dtype, cudaStream_t stream, bool programmatic) {
  CUtensorMap unused{};
  return launch_decode_mode<true>(p, head_dim, q_dtype, kv_dtype, unused, unused, stream,
                                  programmatic);
}

}  // namespace pkv
