// decode_full_first.cu — the decode kernel over a 1-D grid in full-first
// (longest-first) CTA order (decode_item_full_first in decode_kernel.cuh),
// for decode planned beside a prefill grid. A translation unit of its own so
// the other instantiations keep their code and registers.
#include "decode_kernel.cuh"

namespace pkv {

pkv_status launch_decode_full_first(const DecodeParams& p, int head_dim, pkv_dtype q_dtype,
                                    pkv_dtype kv_dtype, const CUtensorMap& tmK,
                                    const CUtensorMap& tmV, cudaStream_t stream,
                                    bool programmatic) {
  return launch_decode_mode<false, kDecodeWarps, true>(p, head_dim, q_dtype, kv_dtype, tmK, tmV,
                                                       stream, programmatic);
}

}  // namespace pkv
