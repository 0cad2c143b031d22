// decode_frags.cuh — page products of the decode kernel with the query heads
// in the MMA N dimension.
//
// With one query token per sequence, a GQA group has G <= 16 query rows; as
// the M dimension of m16n8k16 they would leave most of the tile empty. The
// decode products are therefore transposed, so the heads fill N (8 per
// n-tile, NT = 1 for G <= 8, 2 for G <= 16):
//   S^T[16 tokens x 8NT heads]  = K_page[16 x D] . Q^T[D x 8NT]   (D/16 k-steps)
//   O^T[D x 8NT]               += V_page^T[D x 16] . P^T[16 x 8NT] (D/16 m-tiles)
// P^T is built from the S^T accumulators with movmatrix (an in-register 8x8
// transpose), so no shared memory round trip is needed. Accumulator state
// per thread: O^T NT x D/16 x 4 fp32, Q^T NT x D/16 x 2 registers.
//
// E4M3 caches: the K operand is the A fragment. The contraction index d is
// permuted (thread with c = lane%4 takes chunk 4u + c of its token row;
// byte pair (4i, 4i+1) of that chunk feeds a0/a1 and (4i+2, 4i+3) feeds a2/a3
// of k-step 4u + i), and the Q^T fragments follow the same permutation.
// Tokens: accumulator row r (0..7) is token pi(r) = r ^ ((r & 1) << 2), and
// row r + 8 is token 8 + pi(r); with the 128-byte swizzle this keeps every
// 8-lane phase of the 16-byte K and V reads on distinct banks. The V^T
// operand takes thread g = lane/4's D/8 contiguous bytes of four token rows
// and interleaves token pairs with byte permutes; m-tile t, row g is dim
// (D/8) g + 2t and row g + 8 is dim (D/8) g + 2t + 1.
#pragma once
#include "common.cuh"

namespace pkv {

// Token (0..15) of S^T accumulator row g (r8 = 0) or g + 8 (r8 = 1).
template <int KV>
__device__ __forceinline__ int st_row_token(int g, int r8) {
  if constexpr (KV == KV_E4M3) return 8 * r8 + (g ^ ((g & 1) << 2));
  else return 8 * r8 + g;
}

// Head dimension of O^T accumulator row g (r8 = 0) or g + 8 (r8 = 1) of m-tile t.
template <int D, int KV>
__device__ __forceinline__ int ot_row_dim(int t, int g, int r8) {
  if constexpr (KV == KV_E4M3) return (D / 8) * g + 2 * t + r8;
  else return 16 * t + g + 8 * r8;
}

// Q^T fragments (B operand, D x 8NT) from the G query rows [G][D] of a GQA
// group; head columns >= G are zero. 16-bit q; for E4M3 caches a bf16 q is
// scaled by 2^-qshift (q_f16_shift over the whole group, so one factor
// serves every score of the CTA) and converted to f16. qshift is 0 otherwise.
template <int D, int KV, bool QBF16, int NT>
__device__ __forceinline__ void load_qT_frags(uint32_t (&qf)[NT][D / 16][2],
                                              const uint16_t* qs, int G, int lane, int& qshift) {
  const int g = lane >> 2, c = lane & 3;
#pragma unroll
  for (int nt = 0; nt < NT; ++nt) {
    const bool live = 8 * nt + g < G;
    const uint16_t* row = qs + (live ? (8 * nt + g) : 0) * D;
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
      const uint32_t r0 = *reinterpret_cast<const uint32_t*>(row + d0);
      const uint32_t r1 = *reinterpret_cast<const uint32_t*>(row + d1);
      qf[nt][s][0] = live ? r0 : 0u;
      qf[nt][s][1] = live ? r1 : 0u;
    }
  }
  qshift = 0;
  if constexpr (KV == KV_E4M3 && QBF16) {
    // the warp holds every element of the group: one shift for all of it
    uint32_t m = 0u;
#pragma unroll
    for (int nt = 0; nt < NT; ++nt)
#pragma unroll
      for (int s = 0; s < D / 16; ++s)
        m = max(m, max(bf16x2_max_abs(qf[nt][s][0]), bf16x2_max_abs(qf[nt][s][1])));
    m = __reduce_max_sync(0xffffffffu, m);
    qshift = q_f16_shift(m);
    const float f = pow2f(-qshift);
#pragma unroll
    for (int nt = 0; nt < NT; ++nt)
#pragma unroll
      for (int s = 0; s < D / 16; ++s) {
        qf[nt][s][0] = bf16x2_to_f16x2_scaled(qf[nt][s][0], f);
        qf[nt][s][1] = bf16x2_to_f16x2_scaled(qf[nt][s][1], f);
      }
  }
}

// Byte offset of (token r, dim d) in a page whose TMA boxes (64-element
// column blocks of 16-bit caches) sit BSTRIDE bytes apart.
template <int D, int KV, int BSTRIDE>
__device__ __forceinline__ uint32_t page_off(uint32_t r, uint32_t d) {
  using Geo = PageGeom<D, KV>;
  return (d / Geo::BOX_ELEMS) * BSTRIDE + Geo::swz(r, (d % Geo::BOX_ELEMS) * Geo::ELT);
}

// E4M3 pages staged in registers: a thread's share of the K page (rows
// pi(g) and 8 + pi(g), chunk 4u + c) and of the V page (rows pi(2c), pi(2c+1),
// 8 + pi(2c), 8 + pi(2c+1), bytes (D/8) g ..). Reading them out of shared
// memory first lets the warp refill the ring stage before the math runs.
template <int D>
struct E4M3PageRegs {
  uint4 k[2][D / 64];
  uint32_t v[4][D / 32];
};

template <int D>
__device__ __forceinline__ void load_e4m3_page(E4M3PageRegs<D>& r, uint32_t kpage, uint32_t vpage,
                                               int lane) {
  using Geo = PageGeom<D, KV_E4M3>;
  const int g = lane >> 2, c = lane & 3;
  const int t0 = g ^ ((g & 1) << 2);
#pragma unroll
  for (int u = 0; u < D / 64; ++u) {
    r.k[0][u] = lds128(kpage + Geo::row_off(t0, 16 * (4 * u + c)));
    r.k[1][u] = lds128(kpage + Geo::row_off(8 + t0, 16 * (4 * u + c)));
  }
  const int ta = 2 * c, tb = (2 * c + 1) ^ 4;
  constexpr int CH = D / 8;
  const uint32_t xo = CH * g;
  const int rows[4] = {ta, tb, 8 + ta, 8 + tb};
#pragma unroll
  for (int q = 0; q < 4; ++q) {
    lds_run<D>(r.v[q], vpage, rows[q], xo);
  }
}

// acc += K . Q^T from E4M3 K words (raw[row][u]); two accumulator chains.
template <int D, int NT>
__device__ __forceinline__ void kq_regs(float (&acc)[NT][4], const uint32_t (&qf)[NT][D / 16][2],
                                        const uint4 (&raw)[2][D / 64]) {
  float acc2[NT][4];
#pragma unroll
  for (int nt = 0; nt < NT; ++nt) acc2[nt][0] = acc2[nt][1] = acc2[nt][2] = acc2[nt][3] = 0.f;
#pragma unroll
  for (int u = 0; u < D / 64; ++u) {
    const uint32_t lo[4] = {raw[0][u].x, raw[0][u].y, raw[0][u].z, raw[0][u].w};
    const uint32_t hi[4] = {raw[1][u].x, raw[1][u].y, raw[1][u].z, raw[1][u].w};
#pragma unroll
    for (int i = 0; i < 4; ++i) {
      uint32_t a[4];
      a[0] = e4m3x2_to_f16x2(lo[i] & 0xFFFFu);
      a[1] = e4m3x2_to_f16x2(hi[i] & 0xFFFFu);
      a[2] = e4m3x2_to_f16x2(lo[i] >> 16);
      a[3] = e4m3x2_to_f16x2(hi[i] >> 16);
#pragma unroll
      for (int nt = 0; nt < NT; ++nt)
        mma_f16((i & 1) ? acc2[nt] : acc[nt], a, qf[nt][4 * u + i][0], qf[nt][4 * u + i][1]);
    }
  }
#pragma unroll
  for (int nt = 0; nt < NT; ++nt)
#pragma unroll
    for (int i = 0; i < 4; ++i) acc[nt][i] += acc2[nt][i];
}

// oacc += V^T . P^T from E4M3 V words (rows pi(2c), pi(2c+1), 8+.., 8+..).
template <int D, int NT>
__device__ __forceinline__ void vp_regs(float (&oacc)[NT][D / 16][4], const uint32_t (&pb)[NT][2],
                                        const uint32_t (&v)[4][D / 32]) {
#pragma unroll
  for (int i = 0; i < D / 32; ++i) {
    // dims (D/8) g + 4i + {0,1} -> m-tile 2i, {2,3} -> m-tile 2i+1
    const uint32_t lo01 = __byte_perm(v[0][i], v[1][i], 0x5140);
    const uint32_t lo23 = __byte_perm(v[0][i], v[1][i], 0x7362);
    const uint32_t hi01 = __byte_perm(v[2][i], v[3][i], 0x5140);
    const uint32_t hi23 = __byte_perm(v[2][i], v[3][i], 0x7362);
    uint32_t a0[4], a1[4];
    a0[0] = e4m3x2_to_f16x2(lo01 & 0xFFFFu);
    a0[1] = e4m3x2_to_f16x2(lo01 >> 16);
    a0[2] = e4m3x2_to_f16x2(hi01 & 0xFFFFu);
    a0[3] = e4m3x2_to_f16x2(hi01 >> 16);
    a1[0] = e4m3x2_to_f16x2(lo23 & 0xFFFFu);
    a1[1] = e4m3x2_to_f16x2(lo23 >> 16);
    a1[2] = e4m3x2_to_f16x2(hi23 & 0xFFFFu);
    a1[3] = e4m3x2_to_f16x2(hi23 >> 16);
#pragma unroll
    for (int nt = 0; nt < NT; ++nt) {
      mma_f16(oacc[nt][2 * i], a0, pb[nt][0], pb[nt][1]);
      mma_f16(oacc[nt][2 * i + 1], a1, pb[nt][0], pb[nt][1]);
    }
  }
}

// acc[nt][.] += K_page . Q^T for the page at shared-memory byte address kpage
// (box stride BSTRIDE: several heads' pages may share each box).
template <int D, int KV, int NT, int BSTRIDE = PageGeom<D, KV>::BOX_BYTES>
__device__ __forceinline__ void kq_page(float (&acc)[NT][4], const uint32_t (&qf)[NT][D / 16][2],
                                        uint32_t kpage, int lane) {
  using Geo = PageGeom<D, KV>;
  if constexpr (KV == KV_E4M3) {
    const int g = lane >> 2, c = lane & 3;
    const int t0 = g ^ ((g & 1) << 2);
    uint4 raw[2][D / 64];
#pragma unroll
    for (int u = 0; u < D / 64; ++u) {
      raw[0][u] = lds128(kpage + Geo::row_off(t0, 16 * (4 * u + c)));
      raw[1][u] = lds128(kpage + Geo::row_off(8 + t0, 16 * (4 * u + c)));
    }
    kq_regs<D, NT>(acc, qf, raw);
  } else {
    constexpr bool BF = (KV == KV_BF16);
    const int mi = lane >> 3, r = lane & 7;
    const int tok = r + 8 * (mi & 1);
    // two independent accumulator chains (even / odd k-steps) halve the
    // dependent MMA latency of the contraction
    float acc2[NT][4];
#pragma unroll
    for (int nt = 0; nt < NT; ++nt) acc2[nt][0] = acc2[nt][1] = acc2[nt][2] = acc2[nt][3] = 0.f;
#pragma unroll
    for (int s = 0; s < D / 16; ++s) {
      uint32_t a[4];
      ldmatrix_x4(a, kpage + page_off<D, KV, BSTRIDE>(tok, 16 * s + 8 * (mi >> 1)));
#pragma unroll
      for (int nt = 0; nt < NT; ++nt)
        mma16816<BF>((s & 1) ? acc2[nt] : acc[nt], a, qf[nt][s][0], qf[nt][s][1]);
    }
#pragma unroll
    for (int nt = 0; nt < NT; ++nt)
#pragma unroll
      for (int i = 0; i < 4; ++i) acc[nt][i] += acc2[nt][i];
  }
}

// P^T B fragments from the probabilities held in S^T accumulator layout:
// p[nt][0..1] = tokens of row g, heads 2c, 2c+1; p[nt][2..3] = row g + 8.
template <int KV, int NT>
__device__ __forceinline__ void pT_frags(uint32_t (&pb)[NT][2], const float (&p)[NT][4]) {
  constexpr bool BF = (KV == KV_BF16);
#pragma unroll
  for (int nt = 0; nt < NT; ++nt) {
    pb[nt][0] = movmatrix_trans(pack2<BF>(p[nt][0], p[nt][1]));
    pb[nt][1] = movmatrix_trans(pack2<BF>(p[nt][2], p[nt][3]));
  }
}

// oacc[nt][t][.] += V_page^T . P^T for the page at shared-memory byte address vpage.
template <int D, int KV, int NT, int BSTRIDE = PageGeom<D, KV>::BOX_BYTES>
__device__ __forceinline__ void vp_page(float (&oacc)[NT][D / 16][4], const uint32_t (&pb)[NT][2],
                                        uint32_t vpage, int lane) {
  using Geo = PageGeom<D, KV>;
  if constexpr (KV == KV_E4M3) {
    const int g = lane >> 2, c = lane & 3;
    const int ta = 2 * c, tb = (2 * c + 1) ^ 4;     // pi(2c), pi(2c+1)
    constexpr int CH = D / 8;                      // bytes per token row for this thread
    const uint32_t xo = CH * g;
    uint32_t wa[CH / 4], wb[CH / 4], wc[CH / 4], wd[CH / 4];
    lds_run<D>(wa, vpage, ta, xo);
    lds_run<D>(wb, vpage, tb, xo);
    lds_run<D>(wc, vpage, 8 + ta, xo);
    lds_run<D>(wd, vpage, 8 + tb, xo);
#pragma unroll
    for (int i = 0; i < CH / 4; ++i) {
      // dims (D/8) g + 4i + {0,1} -> m-tile 2i, {2,3} -> m-tile 2i+1
      const uint32_t lo01 = __byte_perm(wa[i], wb[i], 0x5140);
      const uint32_t lo23 = __byte_perm(wa[i], wb[i], 0x7362);
      const uint32_t hi01 = __byte_perm(wc[i], wd[i], 0x5140);
      const uint32_t hi23 = __byte_perm(wc[i], wd[i], 0x7362);
      uint32_t a0[4], a1[4];
      a0[0] = e4m3x2_to_f16x2(lo01 & 0xFFFFu);
      a0[1] = e4m3x2_to_f16x2(lo01 >> 16);
      a0[2] = e4m3x2_to_f16x2(hi01 & 0xFFFFu);
      a0[3] = e4m3x2_to_f16x2(hi01 >> 16);
      a1[0] = e4m3x2_to_f16x2(lo23 & 0xFFFFu);
      a1[1] = e4m3x2_to_f16x2(lo23 >> 16);
      a1[2] = e4m3x2_to_f16x2(hi23 & 0xFFFFu);
      a1[3] = e4m3x2_to_f16x2(hi23 >> 16);
#pragma unroll
      for (int nt = 0; nt < NT; ++nt) {
        mma_f16(oacc[nt][2 * i], a0, pb[nt][0], pb[nt][1]);
        mma_f16(oacc[nt][2 * i + 1], a1, pb[nt][0], pb[nt][1]);
      }
    }
  } else {
    constexpr bool BF = (KV == KV_BF16);
    const int mi = lane >> 3, r = lane & 7;
    const int tok = r + 8 * (mi >> 1);
#pragma unroll
    for (int t = 0; t < D / 16; ++t) {
      uint32_t a[4];
      ldmatrix_x4_trans(a, vpage + page_off<D, KV, BSTRIDE>(tok, 16 * t + 8 * (mi & 1)));
#pragma unroll
      for (int nt = 0; nt < NT; ++nt) mma16816<BF>(oacc[nt][t], a, pb[nt][0], pb[nt][1]);
    }
  }
}

// Zeroes rows [valid, 16) of a page in shared memory (all its boxes). The
// swizzle only permutes 16-byte chunks inside a row, so a row's bytes are
// the row's whole 128-byte (or 64-byte) stripe of each box.
template <int D, int KV>
__device__ __forceinline__ void zero_page_rows(uint8_t* page, int valid, int lane) {
  using Geo = PageGeom<D, KV>;
  constexpr int CPR = Geo::ROW_BYTES / 16;
  for (int i = lane; i < (kBS - valid) * CPR; i += 32) {
    const int r = valid + i / CPR, x = (i % CPR) * 16;
    *reinterpret_cast<uint4*>(page + (x / Geo::BOX_ROW_BYTES) * Geo::BOX_BYTES +
                              r * Geo::BOX_ROW_BYTES + x % Geo::BOX_ROW_BYTES) =
        make_uint4(0u, 0u, 0u, 0u);
  }
}

// The decode kernels' softmax keeps, per column, a reference max that moves
// only when a page's max exceeds it by more than this (log2 units), so the
// accumulators are rescaled rarely; the probabilities stay below 2^8.
constexpr float kRefSlackLog2 = 8.f;

// Max / sum over the 8 lanes that share c = lane % 4 (the 8 token rows g).
__device__ __forceinline__ float col_max8(float v) {
  v = fmaxf(v, __shfl_xor_sync(0xffffffffu, v, 4));
  v = fmaxf(v, __shfl_xor_sync(0xffffffffu, v, 8));
  v = fmaxf(v, __shfl_xor_sync(0xffffffffu, v, 16));
  return v;
}

__device__ __forceinline__ float col_sum8(float v) {
  v += __shfl_xor_sync(0xffffffffu, v, 4);
  v += __shfl_xor_sync(0xffffffffu, v, 8);
  v += __shfl_xor_sync(0xffffffffu, v, 16);
  return v;
}

}  // namespace pkv
