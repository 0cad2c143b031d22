// kv_store.cuh — storing 8 consecutive elements of one (token, KV head) row
// into the paged cache, the step that reshape_and_cache and the fused rotary
// cache write share.
//
// A 16-bit cache takes the source bits as they are. An E4M3 cache takes
// E4M3(x / scale) per element: x widened exactly to fp32, one correctly
// rounded fp32 division, then the conversion rounding to nearest even and
// saturating at +-448 (the "FP8 KV Cache" of the Litellama page, Features,
// with one fp32 scale per KV head).
#pragma once
#include <cstdint>
#include "ptx.cuh"

namespace pkv {

// Element e (0..7) of eight 16-bit values packed in a uint4, widened to fp32.
template <bool SRC_BF16>
__device__ __forceinline__ float widen16(uint32_t bits16) {
  if constexpr (SRC_BF16) return __uint_as_float(bits16 << 16);
  else return __half2float(__ushort_as_half(static_cast<unsigned short>(bits16)));
}

__device__ __forceinline__ uint32_t elem16(const uint4& v, int e) {
  const uint32_t w = e < 2 ? v.x : e < 4 ? v.y : e < 6 ? v.z : v.w;
  return (e & 1) ? (w >> 16) : (w & 0xFFFFu);
}

// Eight 16-bit source values -> eight E4M3 codes (element 0 in the low byte).
template <bool SRC_BF16>
__device__ __forceinline__ uint2 encode_e4m3x8(const uint4& in, float scale) {
  const uint32_t w[4] = {in.x, in.y, in.z, in.w};
  uint32_t out[2];
#pragma unroll
  for (int j = 0; j < 2; ++j) {
    float f[4];
#pragma unroll
    for (int e = 0; e < 2; ++e) {
      const uint32_t word = w[2 * j + e];
      f[2 * e] = widen16<SRC_BF16>(word & 0xFFFFu);
      f[2 * e + 1] = widen16<SRC_BF16>(word >> 16);
    }
    const uint32_t lo = f32x2_to_e4m3x2(__fdiv_rn(f[0], scale), __fdiv_rn(f[1], scale));
    const uint32_t hi = f32x2_to_e4m3x2(__fdiv_rn(f[2], scale), __fdiv_rn(f[3], scale));
    out[j] = lo | (hi << 16);
  }
  return make_uint2(out[0], out[1]);
}

// Store eight elements at element index `idx` (a multiple of 8) of a cache.
template <bool SRC_BF16, bool TO_FP8>
__device__ __forceinline__ void store_row8(void* cache, int64_t idx, const uint4& vals,
                                           float scale) {
  if constexpr (TO_FP8)
    *reinterpret_cast<uint2*>(static_cast<uint8_t*>(cache) + idx) =
        encode_e4m3x8<SRC_BF16>(vals, scale);
  else
    *reinterpret_cast<uint4*>(static_cast<uint16_t*>(cache) + idx) = vals;
}

// Element index of (slot, KV head h, element d) in the cache
// [num_blocks, Hkv, BS, D] with BS = 2^bs_log2: block slot / BS, offset slot % BS.
__device__ __forceinline__ int64_t cache_elem(int64_t slot, int h, int Hkv, int D, int d,
                                              int bs_log2) {
  const int64_t bs = int64_t(1) << bs_log2;
  return (((slot >> bs_log2) * Hkv + h) * bs + (slot & (bs - 1))) * D + d;
}

}  // namespace pkv
