// decode_wide.cu — the decode kernel in its whole-context shape: one CTA of
// kDecodeWideWarps warps per (sequence, KV head), the context one partition
// taken page by page round-robin over the warps, three ring stages per warp
// (an SM per CTA), the warps merged on chip and the output written directly.
// Chosen by the planner (wide_decode in plan.h) for grids of about one wave.
#include "decode_kernel.cuh"

namespace pkv {

pkv_status launch_decode_wide(const DecodeParams& p, int head_dim, pkv_dtype q_dtype,
                              pkv_dtype kv_dtype, const CUtensorMap& tmK, const CUtensorMap& tmV,
                              cudaStream_t stream, bool programmatic) {
  return launch_decode_mode<false, kDecodeWideWarps>(p, head_dim, q_dtype, kv_dtype, tmK, tmV,
                                                     stream, programmatic);
}

}  // namespace pkv
