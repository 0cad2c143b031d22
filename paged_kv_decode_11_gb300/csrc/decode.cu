// decode.cu — paged-KV decode attention: split-KV partitions and their
// log-sum-exp merge in one kernel launch (the kernel is in decode_kernel.cuh).
// Caches with blocks of 16, 32 or 64 tokens are read a page at a time by TMA;
// smaller blocks go to the gather instantiation in decode_gather.cu.
#include "decode_kernel.cuh"

namespace pkv {

size_t decode_smem_bytes(int head_dim, pkv_dtype kv_dtype, int G) {
  constexpr int NW = PKV_DECODE_NW;
  const bool fp8 = kv_dtype == PKV_FP8_E4M3;
  const int nst = fp8 ? PKV_DECODE_NST_E4M3 : PKV_DECODE_NST_16;
  const int page = 16 * head_dim * (fp8 ? 1 : 2);
  const size_t ring = (size_t)NW * nst * 2 * page;
  const size_t obuf = (size_t)NW * 8 * (G > 8 ? 2 : 1) * head_dim * 4;
  return 1024 + (ring > obuf ? ring : obuf);
}

pkv_status launch_decode(const DecodeParams& p, int head_dim, pkv_dtype q_dtype,
                         pkv_dtype kv_dtype, const CUtensorMap& tmK, const CUtensorMap& tmV,
                         cudaStream_t stream, bool programmatic) {
  if (p.bs_log2 < 4)
    return launch_decode_gather(p, head_dim, q_dtype, kv_dtype, stream, programmatic);
  return launch_decode_mode<false>(p, head_dim, q_dtype, kv_dtype, tmK, tmV, stream,
                                   programmatic);
}

}  // namespace pkv
