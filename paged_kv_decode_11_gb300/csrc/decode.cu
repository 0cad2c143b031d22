// decode.cu — paged-KV decode attention: split-KV partitions and their
// log-sum-exp merge in one kernel launch, one CTA per (CTA partition, KV
// head, sequence) (decode_kernel.cuh; the hardware hands CTAs to SMs as they
// free up, which balances uneven SMs for free). Blocks of fewer than 16
// tokens go to the gather instantiation in decode_gather.cu, whole-context
// plans to the 8-warp instantiation in decode_wide.cu, full-first CTA order
// to decode_full_first.cu.
#include "decode_kernel.cuh"

namespace pkv {

pkv_status launch_decode(const DecodeParams& p, int head_dim, pkv_dtype q_dtype,
                         pkv_dtype kv_dtype, const CUtensorMap& tmK, const CUtensorMap& tmV,
                         cudaStream_t stream, bool programmatic) {
  if (p.bs_log2 < 4)
    return launch_decode_gather(p, head_dim, q_dtype, kv_dtype, stream, programmatic);
  if (p.wide)
    return launch_decode_wide(p, head_dim, q_dtype, kv_dtype, tmK, tmV, stream, programmatic);
  if (p.full_first)
    return launch_decode_full_first(p, head_dim, q_dtype, kv_dtype, tmK, tmV, stream,
                                    programmatic);
  return launch_decode_mode<false>(p, head_dim, q_dtype, kv_dtype, tmK, tmV, stream,
                                   programmatic);
}

}  // namespace pkv
