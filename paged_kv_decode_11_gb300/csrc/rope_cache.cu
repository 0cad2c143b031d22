// rope_cache.cu — rope_reshape_and_cache: the rotary position embedding of
// the new tokens' queries and keys, fused with the cache write of their keys
// and values ("RoPE + KV cache write -- fused, no intermediate alloc",
// rvLLM: High-performance LLM inference in Rust, Kernel Compiler Stack). The
// rotation is RoFormer's rotary embedding: pair (x1, x2) of a head turned by
// the angle of the token's position, taken from the caller's cos/sin table:
//   y1 = x1 c - x2 s,   y2 = x2 c + x1 s.
//
// Each result is defined as the product terms exact in double, one rounding
// of the sum to double, then one round-to-nearest-even to the 16-bit source
// dtype. Doubles are slow on this part, so a thread first works in fp32:
//   r = fma(xa, ca, +-fl(xb sb)),  |r - exact| <= (ulp(r) + ulp(fl(xb sb))) / 2,
// and rounds r - b and r + b to 16 bits with b = 2 max(ulp(r), ulp(xb sb)),
// both computed so that [r - b, r + b] contains the exact value. Rounding is
// monotone, so when both ends give the same 16-bit value that value is the
// rounding of the exact sum; and the exact sum then lies at least one fp32
// ulp from every 16-bit midpoint, so its rounding to double does not move
// it across one either: the value equals the defined result. Only when the
// ends differ (the exact sum sits near a midpoint, about 1 element in 2^12)
// does the thread redo that element in double.
//
// Work items, per token: for each query head and each key head, rot_dim/16
// rotation items of 16 elements (rotate-half: dims 8j..8j+7 with their
// partners 8j+rot/2..; interleaved: dims 16j..16j+15, eight adjacent pairs);
// for each key head, (D - rot_dim)/8 pass-through chunks of 8; for each value
// head, D/8 chunks of 8. One thread per item, 16-byte loads and stores.
// Query rows are rewritten in place: an item owns both halves of its pairs,
// so no other thread reads what it writes. Rotated keys go straight to the
// cache (bit copy or E4M3 encode, as reshape_and_cache), never to memory in
// between.
#include <cuda_fp16.h>
#include <cuda_bf16.h>
#include "common.cuh"
#include "kv_store.cuh"
#include "launch_cache.h"

namespace pkv {

template <bool BF16>
__device__ __forceinline__ uint16_t round16(float x) {
  unsigned short r;
  if constexpr (BF16) asm("cvt.rn.bf16.f32 %0, %1;" : "=h"(r) : "f"(x));
  else asm("cvt.rn.f16.f32 %0, %1;" : "=h"(r) : "f"(x));
  return r;
}

template <bool BF16>
__device__ __forceinline__ uint16_t round16(double x) {
  unsigned short r;
  if constexpr (BF16) asm("cvt.rn.bf16.f64 %0, %1;" : "=h"(r) : "d"(x));
  else asm("cvt.rn.f16.f64 %0, %1;" : "=h"(r) : "d"(x));
  return r;
}

// Unit in the last place of a binary32 value (2^-149 for zero and subnormals).
__device__ __forceinline__ float ulp32(float v) {
  const uint32_t e = (__float_as_uint(v) >> 23) & 0xFFu;
  return __uint_as_float(e > 23u ? (e - 23u) << 23 : 1u << (e > 0u ? e - 1u : 0u));
}

// fp32 estimate of xa*ca - xb*sb (MINUS) or xa*ca + xb*sb, rounded to 16
// bits; *ok is false when the error bound straddles a 16-bit midpoint.
template <bool BF16, bool MINUS>
__device__ __forceinline__ uint16_t rotate_fast(float xa, float ca, float xb, float sb, bool* ok) {
  const float pb = __fmul_rn(xb, sb);
  const float r = fmaf(xa, ca, MINUS ? -pb : pb);
  const float b = 2.f * fmaxf(ulp32(r), ulp32(pb));
  const uint16_t lo = round16<BF16>(__fsub_rn(r, b));
  const uint16_t hi = round16<BF16>(__fadd_rn(r, b));
  *ok = (lo == hi);
  return lo;
}

struct Pair8 {
  uint4 a, b;
};

__device__ __forceinline__ uint4 pack8(const uint16_t (&h)[8]) {
  return make_uint4(h[0] | ((uint32_t)h[1] << 16), h[2] | ((uint32_t)h[3] << 16),
                    h[4] | ((uint32_t)h[5] << 16), h[6] | ((uint32_t)h[7] << 16));
}

// Element index (0..7) within chunk a (pair e < 4 or rotate-half) or chunk b
// of the first / second member of pair e.
template <bool NEOX>
__device__ __forceinline__ int pair_slot(int e, bool second) {
  return NEOX ? e : (2 * e + (second ? 1 : 0)) & 7;
}
template <bool NEOX>
__device__ __forceinline__ bool pair_in_b(int e, bool second) {
  return NEOX ? second : e >= 4;
}

// The 16 inputs of rotation item j in pair order: x1[e], x2[e] for pair e
// (rotate-half: element e of both chunks; interleaved: elements 2e, 2e+1 of
// the 16-element run).
template <bool BF16, bool NEOX>
__device__ __forceinline__ void item_pairs(const uint4& in_a, const uint4& in_b, float (&x1)[8],
                                           float (&x2)[8]) {
#pragma unroll
  for (int e = 0; e < 8; ++e) {
    x1[e] = widen16<BF16>(elem16(pair_in_b<NEOX>(e, false) ? in_b : in_a, pair_slot<NEOX>(e, false)));
    x2[e] = widen16<BF16>(elem16(pair_in_b<NEOX>(e, true) ? in_b : in_a, pair_slot<NEOX>(e, true)));
  }
}

// Places y1[e], y2[e] where their inputs came from.
template <bool NEOX>
__device__ __forceinline__ Pair8 item_pack(const uint16_t (&y1)[8], const uint16_t (&y2)[8]) {
  uint16_t oa[8], ob[8];
#pragma unroll
  for (int e = 0; e < 8; ++e) {
    (pair_in_b<NEOX>(e, false) ? ob : oa)[pair_slot<NEOX>(e, false)] = y1[e];
    (pair_in_b<NEOX>(e, true) ? ob : oa)[pair_slot<NEOX>(e, true)] = y2[e];
  }
  return Pair8{pack8(oa), pack8(ob)};
}

// Redoes in double the outputs whose bit is set in `redo` (bit e: y1 of pair
// e, bit 8+e: y2), one at a time, so the double-precision work is only what
// is undecided. Kept out of line: only threads with an undecided output call
// it, so the common path carries none of it.
template <bool BF16, bool NEOX>
__device__ __noinline__ Pair8 rotate_item_exact(uint32_t redo, uint4 in_a, uint4 in_b, float4 c0,
                                                float4 c1, float4 s0, float4 s1, Pair8 fast) {
  float x1[8], x2[8];
  item_pairs<BF16, NEOX>(in_a, in_b, x1, x2);
  const float c[8] = {c0.x, c0.y, c0.z, c0.w, c1.x, c1.y, c1.z, c1.w};
  const float s[8] = {s0.x, s0.y, s0.z, s0.w, s1.x, s1.y, s1.z, s1.w};
  uint16_t y[16];                   // y1 of pair e at [e], y2 at [8 + e]
#pragma unroll
  for (int e = 0; e < 8; ++e) {
    y[e] = elem16(pair_in_b<NEOX>(e, false) ? fast.b : fast.a, pair_slot<NEOX>(e, false));
    y[8 + e] = elem16(pair_in_b<NEOX>(e, true) ? fast.b : fast.a, pair_slot<NEOX>(e, true));
  }
  while (redo != 0u) {
    const int k = __ffs(redo) - 1;
    redo &= redo - 1u;
    const int e = k & 7;
    const bool first = k < 8;       // y1 = x1 c - x2 s, else y2 = x2 c + x1 s
    const double da = __dmul_rn((double)(first ? x1[e] : x2[e]), (double)c[e]);
    const double db = __dmul_rn((double)(first ? x2[e] : x1[e]), (double)s[e]);
    y[k] = round16<BF16>(__dadd_rn(da, first ? -db : db));
  }
  uint16_t y1[8], y2[8];
#pragma unroll
  for (int e = 0; e < 8; ++e) {
    y1[e] = y[e];
    y2[e] = y[8 + e];
  }
  return item_pack<NEOX>(y1, y2);
}

// Rotates the 16 elements of rotation item j of one head row. The result's
// a / b are the 8 elements stored at offsets off_a / off_b of the row.
template <bool BF16, bool NEOX>
__device__ __forceinline__ Pair8 rotate_item(const uint16_t* row, const float* cs, int rot, int j,
                                             int& off_a, int& off_b) {
  const int half = rot / 2;
  off_a = NEOX ? 8 * j : 16 * j;
  off_b = NEOX ? 8 * j + half : 16 * j + 8;
  const uint4 in_a = *reinterpret_cast<const uint4*>(row + off_a);
  const uint4 in_b = *reinterpret_cast<const uint4*>(row + off_b);
  const float4 c0 = *reinterpret_cast<const float4*>(cs + 8 * j);
  const float4 c1 = *reinterpret_cast<const float4*>(cs + 8 * j + 4);
  const float4 s0 = *reinterpret_cast<const float4*>(cs + half + 8 * j);
  const float4 s1 = *reinterpret_cast<const float4*>(cs + half + 8 * j + 4);
  const float c[8] = {c0.x, c0.y, c0.z, c0.w, c1.x, c1.y, c1.z, c1.w};
  const float s[8] = {s0.x, s0.y, s0.z, s0.w, s1.x, s1.y, s1.z, s1.w};
  float x1[8], x2[8];
  item_pairs<BF16, NEOX>(in_a, in_b, x1, x2);
  uint16_t y1[8], y2[8];
  uint32_t redo = 0;
#pragma unroll
  for (int e = 0; e < 8; ++e) {
    bool ok1, ok2;
    y1[e] = rotate_fast<BF16, true>(x1[e], c[e], x2[e], s[e], &ok1);
    y2[e] = rotate_fast<BF16, false>(x2[e], c[e], x1[e], s[e], &ok2);
    redo |= (ok1 ? 0u : 1u << e) | (ok2 ? 0u : 1u << (8 + e));
  }
  const Pair8 fast = item_pack<NEOX>(y1, y2);
  if (redo != 0u) return rotate_item_exact<BF16, NEOX>(redo, in_a, in_b, c0, c1, s0, s1, fast);
  return fast;
}

template <bool BF16, bool TO_FP8, bool NEOX>
__global__ void __launch_bounds__(256) rope_cache_kernel(const RopeCacheParams p) {
  // a decode launched behind this kernel may become resident now; it waits
  // for this grid to finish before it reads anything
  if (threadIdx.x == 0) griddep_launch_dependents();
  const int R = p.rot / 16;                 // rotation items per head
  const int PT = (p.D - p.rot) / 8;         // pass-through chunks per key head
  const int C8 = p.D / 8;                   // chunks per value head
  const int nq = p.Hq * R, nk = p.Hkv * (R + PT), nv = p.Hkv * C8;
  const int per_tok = nq + nk + nv;
  const int64_t i = (int64_t)blockIdx.x * blockDim.x + threadIdx.x;
  if (i >= (int64_t)p.num_tokens * per_tok) return;
  const int64_t t = i / per_tok;
  int r = (int)(i - t * per_tok);
  const int64_t pos = p.positions[t];
  if (pos < 0 || pos >= p.max_position) {
    if (r == 0) atomicOr(p.err, PKV_DEVERR_POSITION);
    return;
  }
  const float* cs = p.cos_sin + pos * p.rot;
  if (r < nq) {                                           // query: rotate in place
    const int h = r / R, j = r - (r / R) * R;
    uint16_t* row = static_cast<uint16_t*>(p.query) + (t * p.Hq + h) * p.D;
    int oa, ob;
    const Pair8 y = rotate_item<BF16, NEOX>(row, cs, p.rot, j, oa, ob);
    *reinterpret_cast<uint4*>(row + oa) = y.a;
    *reinterpret_cast<uint4*>(row + ob) = y.b;
    return;
  }
  const int64_t slot = p.slots[t];
  if (slot < 0) return;
  if (slot >= ((int64_t)p.num_blocks << p.bs_log2)) {
    if (r == nq) atomicOr(p.err, PKV_DEVERR_SLOT);
    return;
  }
  r -= nq;
  if (r < nk) {                                           // key: rotate, then store
    const int per_head = R + PT;
    const int h = r / per_head, j = r - h * per_head;
    const uint16_t* row = static_cast<const uint16_t*>(p.key) + (t * p.Hkv + h) * p.D;
    const float ks = TO_FP8 ? p.k_scales[h] : 1.f;
    const int64_t base = cache_elem(slot, h, p.Hkv, p.D, 0, p.bs_log2);
    if (j < R) {
      int oa, ob;
      const Pair8 y = rotate_item<BF16, NEOX>(row, cs, p.rot, j, oa, ob);
      store_row8<BF16, TO_FP8>(p.k_cache, base + oa, y.a, ks);
      store_row8<BF16, TO_FP8>(p.k_cache, base + ob, y.b, ks);
    } else {
      const int off = p.rot + 8 * (j - R);
      store_row8<BF16, TO_FP8>(p.k_cache, base + off,
                               *reinterpret_cast<const uint4*>(row + off), ks);
    }
    return;
  }
  r -= nk;                                                // value: store
  const int h = r / C8, off = 8 * (r - h * C8);
  const uint16_t* row = static_cast<const uint16_t*>(p.value) + (t * p.Hkv + h) * p.D;
  const float vs = TO_FP8 ? p.v_scales[h] : 1.f;
  store_row8<BF16, TO_FP8>(p.v_cache, cache_elem(slot, h, p.Hkv, p.D, off, p.bs_log2),
                           *reinterpret_cast<const uint4*>(row + off), vs);
}

pkv_status launch_rope_cache(const RopeCacheParams& p, pkv_dtype src_dtype, pkv_dtype kv_dtype,
                             cudaStream_t stream) {
  const int64_t per_tok = (int64_t)p.Hq * (p.rot / 16) +
                          (int64_t)p.Hkv * (p.rot / 16 + (p.D - p.rot) / 8) +
                          (int64_t)p.Hkv * (p.D / 8);
  const int64_t total = (int64_t)p.num_tokens * per_tok;
  if (total == 0) return PKV_OK;
  const int threads = 256;
  const int64_t blocks = (total + threads - 1) / threads;
  if (blocks > 0x7FFFFFFF) return PKV_ERR_INVALID_ARG;
  const bool bf = (src_dtype == PKV_BF16);
  const bool fp8 = (kv_dtype == PKV_FP8_E4M3);
  const unsigned g = (unsigned)blocks;
#define PKV_ROPE_LAUNCH(B, F, N) rope_cache_kernel<B, F, N><<<g, threads, 0, stream>>>(p)
  if (p.neox) {
    if (bf && fp8) PKV_ROPE_LAUNCH(true, true, true);
    else if (bf) PKV_ROPE_LAUNCH(true, false, true);
    else if (fp8) PKV_ROPE_LAUNCH(false, true, true);
    else PKV_ROPE_LAUNCH(false, false, true);
  } else {
    if (bf && fp8) PKV_ROPE_LAUNCH(true, true, false);
    else if (bf) PKV_ROPE_LAUNCH(true, false, false);
    else if (fp8) PKV_ROPE_LAUNCH(false, true, false);
    else PKV_ROPE_LAUNCH(false, false, false);
  }
#undef PKV_ROPE_LAUNCH
  return cudaGetLastError() == cudaSuccess ? PKV_OK : PKV_ERR_CUDA;
}

}  // namespace pkv
