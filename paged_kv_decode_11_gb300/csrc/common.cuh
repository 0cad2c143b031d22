// common.cuh — page geometry in shared memory and the warp-level fragment
// routines that decode and prefill share.
//
// A KV page is the BS x D run of one KV head inside one physical block
// (cache layout [num_blocks, Hkv, BS, D]); BS = 16 tokens. It reaches shared
// memory through a 3-D TMA tensor map {D, BS, num_blocks * Hkv}, box
// {BOX_ELEMS, 16, 1}, with the 128-byte (or 64-byte) swizzle, so a page is
// NBOX boxes of 16 rows x BOX_ROW_BYTES bytes.
//
// QK^T and PV of one page are m16n8k16 tensor-core products with 16 query
// rows (the GQA group, padded) and fp32 accumulators:
//   S[16 x 16 tokens]  = Q[16 x D] . K_page^T        (2 n-tiles, D/16 k-steps)
//   O[16 x D]         += P[16 x 16 tokens] . V_page   (D/8 n-tiles, 1 k-step)
// 16-bit caches feed the B operands with ldmatrix (.trans for V). E4M3
// caches are converted in registers (cvt e4m3x2 -> f16x2, exact) and use f16
// MMAs; their operand layouts are chosen so every thread reads whole 16-byte
// chunks without bank conflicts:
//   * K: the contraction index d is permuted. Thread (g = lane/4, c = lane%4)
//     reads chunk 4u + c (bytes 16(4u+c) .. +15) of its token row; byte pair
//     (4i, 4i+1) feeds b0 and (4i+2, 4i+3) feeds b1 of k-step 4u + i. The Q
//     fragments use the same permutation, so the dot products are unchanged.
//   * tokens: B column n of a K n-tile is token pi(n) = n ^ ((n & 1) << 2);
//     with the 128-byte swizzle this keeps both the K reads and the V reads
//     of every 8-lane phase on distinct banks. S column n is token pi(n).
//   * V: output column n of n-tile t is d = (D/8) n + t, so thread g reads
//     the D/8 contiguous bytes starting at d = (D/8) g of two token rows and
//     interleaves them with byte permutes into (token, token') pairs.
#pragma once
#include <cstdint>
#include "ptx.cuh"

namespace pkv {

constexpr int kBS = 16;                 // tokens per block (page rows)
constexpr float kLog2e = 1.4426950408889634f;
constexpr float kLn2 = 0.6931471805599453f;

enum KvKind { KV_F16 = 0, KV_BF16 = 1, KV_E4M3 = 2 };

template <int D, int KV>
struct PageGeom {
  static constexpr int ELT = (KV == KV_E4M3) ? 1 : 2;
  static constexpr int ROW_BYTES = D * ELT;
  static constexpr int BOX_ROW_BYTES = ROW_BYTES > 128 ? 128 : ROW_BYTES;
  static constexpr int NBOX = ROW_BYTES / BOX_ROW_BYTES;
  static constexpr int BOX_ELEMS = BOX_ROW_BYTES / ELT;
  static constexpr int BOX_BYTES = BOX_ROW_BYTES * kBS;
  static constexpr int PAGE_BYTES = ROW_BYTES * kBS;
  static constexpr int SWZ_MASK = BOX_ROW_BYTES / 16 - 1;   // 7: 128B swizzle, 3: 64B
  static constexpr int KSTEPS = D / 16;
  static constexpr int NTILES = D / 8;
  static_assert(BOX_ROW_BYTES == 128 || BOX_ROW_BYTES == 64, "unsupported page row");

  // Byte offset inside a swizzled box of row `r`, byte `x` of the row.
  __device__ __forceinline__ static uint32_t swz(uint32_t r, uint32_t x) {
    uint32_t off = r * BOX_ROW_BYTES + x;
    return off ^ (((off >> 7) & SWZ_MASK) << 4);
  }
  // Byte offset inside a page of byte x of row r, for rows of any width (a
  // row wider than one box continues in the next box).
  __device__ __forceinline__ static uint32_t row_off(uint32_t r, uint32_t x) {
    return (x / BOX_ROW_BYTES) * BOX_BYTES + swz(r, x % BOX_ROW_BYTES);
  }
  // Byte offset inside a page of element (token r, dim d) (16-bit caches).
  __device__ __forceinline__ static uint32_t elem_off(uint32_t r, uint32_t d) {
    return (d / BOX_ELEMS) * BOX_BYTES + swz(r, (d % BOX_ELEMS) * ELT);
  }
};

// A thread's run of D/8 bytes of row r of an E4M3 page, starting at byte xo
// (a multiple of D/8), as D/32 words.
template <int D>
__device__ __forceinline__ void lds_run(uint32_t (&w)[D / 32], uint32_t page, int r,
                                        uint32_t xo) {
  using Geo = PageGeom<D, KV_E4M3>;
  constexpr int CH = D / 8;
  if constexpr (CH == 8) {
    const uint2 v = lds64(page + Geo::row_off(r, xo));
    w[0] = v.x;
    w[1] = v.y;
  } else {
#pragma unroll
    for (int j = 0; j < CH / 16; ++j) {
      const uint4 v = lds128(page + Geo::row_off(r, xo + 16 * j));
      w[4 * j] = v.x;
      w[4 * j + 1] = v.y;
      w[4 * j + 2] = v.z;
      w[4 * j + 3] = v.w;
    }
  }
}

// E4M3 caches run f16 MMAs, so a bf16 query is converted to f16 first. To keep
// that conversion from overflowing (bf16 reaches 2^128, f16 only 65504) or
// losing the bits of small values, the query is scaled by 2^-e, with e chosen
// so that the largest magnitude of the scaled rows lies in [2^14, 2^15), and
// the scores are scaled back by 2^e. Both scalings are by powers of two, so
// they are exact: every element within 2^-28 of the largest converts to f16
// exactly, and where the unscaled conversion was exact the scores come out
// bit for bit the same. `max_abs` holds the bf16 bits (sign cleared) of the
// largest magnitude.
__device__ __forceinline__ int q_f16_shift(uint32_t max_abs) {
  const int eb = (int)((max_abs >> 7) & 0xFFu);     // biased exponent; 0: zero or subnormal
  const int e = eb == 0 ? -64 : eb - 127 - 14;
  return min(max(e, -64), 126);
}

// 2^e as a float, for e in [-126, 127].
__device__ __forceinline__ float pow2f(int e) { return __int_as_float((127 + e) << 23); }

// Largest bf16 magnitude (bits, sign cleared) of the two halves of a word.
__device__ __forceinline__ uint32_t bf16x2_max_abs(uint32_t w) {
  return max(w & 0x7FFFu, (w >> 16) & 0x7FFFu);
}

// Two bf16 values times 2^-e (exact, a power of two), rounded to f16x2.
__device__ __forceinline__ uint32_t bf16x2_to_f16x2_scaled(uint32_t w, float inv_pow2) {
  const float2 f = __bfloat1622float2(*reinterpret_cast<const __nv_bfloat162*>(&w));
  return pack_f16x2(f.x * inv_pow2, f.y * inv_pow2);
}

// Token (0..15) of S accumulator element e (0, 1) of n-tile j for a thread
// with c = lane % 4.
template <int KV>
__device__ __forceinline__ int s_col_token(int j, int c, int e) {
  int n = 2 * c + e;
  if constexpr (KV == KV_E4M3) n ^= ((n & 1) << 2);
  return 8 * j + n;
}

// Head dimension of O accumulator element e (0, 1) of n-tile t.
template <int D, int KV>
__device__ __forceinline__ int o_col_dim(int t, int c, int e) {
  int n = 2 * c + e;
  if constexpr (KV == KV_E4M3) return (D / 8) * n + t;
  else return 8 * t + n;
}

// Q fragments (A operand, 16 rows x D) for the page products. rowg / rowg8
// point at the D values of query rows g and g + 8 (nullptr = padding row, 0).
// E4M3 caches use f16 MMAs: a bf16 q is scaled per row by 2^-sh (q_f16_shift;
// sh0 for row g, sh8 for row g + 8, 0 otherwise) and converted to f16, and the
// contraction index follows the permutation described at the top of this file.
template <int D, int KV, bool QBF16>
__device__ __forceinline__ void load_q_frags(uint32_t (&qf)[D / 16][4], const void* rowg,
                                             const void* rowg8, int lane, int& sh0, int& sh8) {
  const int c = lane & 3;
  auto ld2 = [&](const void* row, int d) -> uint32_t {
    if (row == nullptr) return 0u;
    return *reinterpret_cast<const uint32_t*>(static_cast<const uint16_t*>(row) + d);
  };
#pragma unroll
  for (int s = 0; s < D / 16; ++s) {
    int d0, d1;
    if constexpr (KV == KV_E4M3) {
      const int u = s >> 2, i = s & 3;
      d0 = 16 * (4 * u + c) + 4 * i;
      d1 = d0 + 2;
    } else {
      d0 = 16 * s + 2 * c;
      d1 = d0 + 8;
    }
    qf[s][0] = ld2(rowg, d0);
    qf[s][1] = ld2(rowg8, d0);
    qf[s][2] = ld2(rowg, d1);
    qf[s][3] = ld2(rowg8, d1);
  }
  sh0 = sh8 = 0;
  if constexpr (KV == KV_E4M3 && QBF16) {
    // the four lanes of a quad hold the whole of rows g and g + 8
    uint32_t m0 = 0u, m8 = 0u;
#pragma unroll
    for (int s = 0; s < D / 16; ++s) {
      m0 = max(m0, max(bf16x2_max_abs(qf[s][0]), bf16x2_max_abs(qf[s][2])));
      m8 = max(m8, max(bf16x2_max_abs(qf[s][1]), bf16x2_max_abs(qf[s][3])));
    }
#pragma unroll
    for (int o = 1; o <= 2; o <<= 1) {
      m0 = max(m0, __shfl_xor_sync(0xffffffffu, m0, o));
      m8 = max(m8, __shfl_xor_sync(0xffffffffu, m8, o));
    }
    sh0 = q_f16_shift(m0);
    sh8 = q_f16_shift(m8);
    const float f0 = pow2f(-sh0), f8 = pow2f(-sh8);
#pragma unroll
    for (int s = 0; s < D / 16; ++s) {
      qf[s][0] = bf16x2_to_f16x2_scaled(qf[s][0], f0);
      qf[s][1] = bf16x2_to_f16x2_scaled(qf[s][1], f8);
      qf[s][2] = bf16x2_to_f16x2_scaled(qf[s][2], f0);
      qf[s][3] = bf16x2_to_f16x2_scaled(qf[s][3], f8);
    }
  }
}

// acc[j0 + j][.] += Q . K_page^T for the two 8-token n-tiles j of the page
// at shared-memory byte address kpage (j0 is a compile-time offset after
// unrolling, so acc stays in registers).
template <int D, int KV, int NJ>
__device__ __forceinline__ void qk_page(float (&acc)[NJ][4], int j0,
                                        const uint32_t (&qf)[D / 16][4], uint32_t kpage,
                                        int lane) {
  using Geo = PageGeom<D, KV>;
  if constexpr (KV == KV_E4M3) {
    const int g = lane >> 2, c = lane & 3;
    const int tn = g ^ ((g & 1) << 2);
#pragma unroll
    for (int j = 0; j < 2; ++j) {
      const int tok = 8 * j + tn;
#pragma unroll
      for (int u = 0; u < D / 64; ++u) {
        uint4 w = lds128(kpage + Geo::row_off(tok, 16 * (4 * u + c)));
        const uint32_t ws[4] = {w.x, w.y, w.z, w.w};
#pragma unroll
        for (int i = 0; i < 4; ++i) {
          uint32_t b0 = e4m3x2_to_f16x2(ws[i] & 0xFFFFu);
          uint32_t b1 = e4m3x2_to_f16x2(ws[i] >> 16);
          mma_f16(acc[j0 + j], qf[4 * u + i], b0, b1);
        }
      }
    }
  } else {
    constexpr bool BF = (KV == KV_BF16);
#pragma unroll
    for (int j = 0; j < 2; ++j) {
      const int tok = 8 * j + (lane & 7);
#pragma unroll
      for (int s2 = 0; s2 < D / 32; ++s2) {
        uint32_t r[4];
        ldmatrix_x4(r, kpage + Geo::elem_off(tok, 32 * s2 + 8 * (lane >> 3)));
        mma16816<BF>(acc[j0 + j], qf[2 * s2], r[0], r[1]);
        mma16816<BF>(acc[j0 + j], qf[2 * s2 + 1], r[2], r[3]);
      }
    }
  }
}

// Zero mask of the 16-bit half of a packed pair holding token t, if t is not
// among the page's first `valid` tokens (low half = even token).
__device__ __forceinline__ uint32_t keep_pair(int t_even, int valid) {
  return (t_even < valid ? 0x0000FFFFu : 0u) | (t_even + 1 < valid ? 0xFFFF0000u : 0u);
}

// oacc[t][.] += P . V_page for the page at shared-memory byte address vpage;
// pa is the A fragment of P (16 rows x 16 tokens of this page). Only the first
// `valid` token rows of the page are real: the others get weight 0 in P, and
// their V values are zeroed here so whatever the cache holds there (even NaN)
// cannot reach the output.
template <int D, int KV>
__device__ __forceinline__ void pv_page(float (&oacc)[D / 8][4], const uint32_t (&pa)[4],
                                        uint32_t vpage, int lane, int valid = kBS) {
  using Geo = PageGeom<D, KV>;
  if constexpr (KV == KV_E4M3) {
    const int g = lane >> 2, c = lane & 3;
    const int t0 = 2 * c, t1 = (2 * c + 1) ^ 4;      // pi(2c), pi(2c+1)
    constexpr int CH = D / 8;                        // bytes per thread per row
    const uint32_t xo = CH * g;
    uint32_t wa[CH / 4], wb[CH / 4], wc[CH / 4], wd[CH / 4];
    lds_run<D>(wa, vpage, t0, xo);
    lds_run<D>(wb, vpage, t1, xo);
    lds_run<D>(wc, vpage, 8 + t0, xo);
    lds_run<D>(wd, vpage, 8 + t1, xo);
    if (valid < kBS) {
#pragma unroll
      for (int i = 0; i < CH / 4; ++i) {
        if (t0 >= valid) wa[i] = 0u;
        if (t1 >= valid) wb[i] = 0u;
        if (8 + t0 >= valid) wc[i] = 0u;
        if (8 + t1 >= valid) wd[i] = 0u;
      }
    }
#pragma unroll
    for (int i = 0; i < CH / 4; ++i) {
      const uint32_t lo01 = __byte_perm(wa[i], wb[i], 0x5140);
      const uint32_t lo23 = __byte_perm(wa[i], wb[i], 0x7362);
      const uint32_t hi01 = __byte_perm(wc[i], wd[i], 0x5140);
      const uint32_t hi23 = __byte_perm(wc[i], wd[i], 0x7362);
      mma_f16(oacc[4 * i + 0], pa, e4m3x2_to_f16x2(lo01 & 0xFFFFu), e4m3x2_to_f16x2(hi01 & 0xFFFFu));
      mma_f16(oacc[4 * i + 1], pa, e4m3x2_to_f16x2(lo01 >> 16), e4m3x2_to_f16x2(hi01 >> 16));
      mma_f16(oacc[4 * i + 2], pa, e4m3x2_to_f16x2(lo23 & 0xFFFFu), e4m3x2_to_f16x2(hi23 & 0xFFFFu));
      mma_f16(oacc[4 * i + 3], pa, e4m3x2_to_f16x2(lo23 >> 16), e4m3x2_to_f16x2(hi23 >> 16));
    }
  } else {
    constexpr bool BF = (KV == KV_BF16);
    const int tok = (lane & 7) + 8 * ((lane >> 3) & 1);
#pragma unroll
    for (int t2 = 0; t2 < D / 16; ++t2) {
      uint32_t r[4];
      ldmatrix_x4_trans(r, vpage + Geo::elem_off(tok, 16 * t2 + 8 * (lane >> 4)));
      if (valid < kBS) {
        // r[0], r[2]: tokens 2c, 2c+1; r[1], r[3]: tokens 8+2c, 9+2c
        const int c2 = 2 * (lane & 3);
        r[0] &= keep_pair(c2, valid);
        r[2] &= keep_pair(c2, valid);
        r[1] &= keep_pair(8 + c2, valid);
        r[3] &= keep_pair(8 + c2, valid);
      }
      mma16816<BF>(oacc[2 * t2], pa, r[0], r[1]);
      mma16816<BF>(oacc[2 * t2 + 1], pa, r[2], r[3]);
    }
  }
}

// P operand of the page product, packed from the S n-tiles j0 and j0 + 1. 16-bit
// caches use their own dtype for P; E4M3 caches use f16.
template <int KV, int NJ>
__device__ __forceinline__ void pack_p(uint32_t (&pa)[4], const float (&p)[NJ][4], int j0) {
  constexpr bool BF = (KV == KV_BF16);
  pa[0] = pack2<BF>(p[j0][0], p[j0][1]);
  pa[1] = pack2<BF>(p[j0][2], p[j0][3]);
  pa[2] = pack2<BF>(p[j0 + 1][0], p[j0 + 1][1]);
  pa[3] = pack2<BF>(p[j0 + 1][2], p[j0 + 1][3]);
}

__device__ __forceinline__ float quad_max(float v) {
  v = fmaxf(v, __shfl_xor_sync(0xffffffffu, v, 1));
  v = fmaxf(v, __shfl_xor_sync(0xffffffffu, v, 2));
  return v;
}

__device__ __forceinline__ float quad_sum(float v) {
  v += __shfl_xor_sync(0xffffffffu, v, 1);
  v += __shfl_xor_sync(0xffffffffu, v, 2);
  return v;
}

}  // namespace pkv
