// prefill_tc.cu — causal chunked-prefill attention on the fifth-generation
// tensor cores (tcgen05), for 16-bit caches at head_dim 64 and 128.
//
// Follows "Chunked Prefill" (Litellama, Features: a long prompt enters the
// batch as chunks of new query tokens attending their cached context) with
// the causal alignment of the library: query row i of a chunk of L tokens on
// P cached ones sees keys 0 .. P + i. Same result as prefill.cu (online
// softmax over key tiles, fp32 accumulation); the contraction runs on the
// tensor cores with its accumulators in tensor memory:
//
//   CTA = (query tile, KV head, chunk). Tile rows are (query token, head of
//   the GQA group) pairs, 128 of them: the MMA M. Warp 4 streams K and V
//   tiles of 4 pages (64 keys) through a TMA ring. Warp 5 issues
//     S[128 x 64]  = Q[128 x D] . K_tile^T   (K-major A and B, fp32 in TMEM)
//   and, once the softmax has written P,
//     O[128 x D]  += P[128 x 64] . V_tile     (V read MN-major)
//   Warps 0-3 own 32 TMEM lanes each: thread r holds row r of S, so the row
//   max and sum need no shuffles. O and the row sum are kept relative to a
//   reference max that moves only when the row max grows by more than 2^8,
//   so O in TMEM is rescaled rarely; the result is the same softmax.
//
// Shared memory: Q [D/64][128 rows][128 B], then NST stages of
// K [D/64][4 pages][16 rows][128 B] and V (same), then two P buffers
// [128 rows][128 B] (S has two TMEM buffers likewise, so the S product of
// the next tile runs while this one's softmax does),
// all in the 128-byte swizzled layout (tc.cuh). Placing the four pages of a
// 64-byte column block back to back gives every operand a uniform 1 KB
// stride between 8-row groups.
#include <cuda.h>
#include "common.cuh"
#include "launch.h"
#include "tc.cuh"

namespace pkv {

constexpr int kTcRows = 128;                  // query rows per CTA (MMA M)
constexpr int kTcKeys = 64;                   // keys per tile (S MMA N)
constexpr int kTcPages = kTcKeys / kBS;
constexpr float kRescaleLog2 = 8.f;           // reference-max slack (log2 units)

template <int D, int NST>
struct PrefillTcCfg {
  static constexpr int NBOX = D / 64;                        // 128-byte column blocks per row
  static constexpr int Q_BOX = kTcRows * 128;                // one column block of Q
  static constexpr int Q_BYTES = NBOX * Q_BOX;
  static constexpr int KV_BOX = kTcPages * kBS * 128;        // one column block of a K/V tile
  static constexpr int KV_BYTES = NBOX * KV_BOX;
  static constexpr int STAGE_BYTES = 2 * KV_BYTES;
  static constexpr int P_BYTES = kTcRows * 128;              // one P buffer (two are kept)
  static constexpr int SMEM_BYTES = 1024 + Q_BYTES + NST * STAGE_BYTES + 2 * P_BYTES;
  static constexpr uint32_t TMEM_COLS = 256;                  // S0, S1, O
};

__device__ __forceinline__ uint32_t swz128(uint32_t r, uint32_t chunk) {
  return r * 128u + ((chunk ^ (r & 7u)) << 4);
}

template <bool BF16>
__device__ __forceinline__ uint32_t pack16x2(float lo, float hi) {
  return pack2<BF16>(lo, hi);
}

// 2^x by the SFU's approximation (flushes subnormal results to 0; 2^-inf = 0).
// Softmax weights here lie in [0, 2^8] and are rounded to 16 bits next.
__device__ __forceinline__ float ex2_approx(float x) {
  float y;
  asm("ex2.approx.ftz.f32 %0, %1;" : "=f"(y) : "f"(x));
  return y;
}

// ---- thread-block cluster helpers (the key range of a query tile split over
// the CTAs of a cluster, merged in the leader's shared memory) ----------------
__device__ __forceinline__ uint32_t cluster_rank() {
  uint32_t r;
  asm volatile("mov.u32 %0, %%cluster_ctarank;" : "=r"(r));
  return r;
}
// Address of the same shared-memory location in CTA `rank` of the cluster.
__device__ __forceinline__ uint32_t cluster_map(uint32_t saddr, uint32_t rank) {
  uint32_t r;
  asm volatile("mapa.shared::cluster.u32 %0, %1, %2;" : "=r"(r) : "r"(saddr), "r"(rank));
  return r;
}
__device__ __forceinline__ void cluster_sync_all() {
  asm volatile("barrier.cluster.arrive.release.aligned;\n\tbarrier.cluster.wait.acquire.aligned;"
               ::: "memory");
}
__device__ __forceinline__ void st_cluster_v4(uint32_t addr, float a, float b, float c, float d) {
  asm volatile("st.shared::cluster.v4.f32 [%0], {%1, %2, %3, %4};" ::"r"(addr), "f"(a), "f"(b),
               "f"(c), "f"(d)
               : "memory");
}
__device__ __forceinline__ void st_cluster_v2(uint32_t addr, float a, float b) {
  asm volatile("st.shared::cluster.v2.f32 [%0], {%1, %2};" ::"r"(addr), "f"(a), "f"(b)
               : "memory");
}
// One arrival on an mbarrier of another CTA of the cluster, ordered after
// this thread's earlier shared-memory writes (cluster scope).
__device__ __forceinline__ void mbar_arrive_remote(uint32_t cluster_addr) {
  asm volatile("mbarrier.arrive.release.cluster.shared::cluster.b64 _, [%0];" ::"r"(cluster_addr)
               : "memory");
}
// Bounded wait on a local mbarrier whose arrivals come from other CTAs.
__device__ __forceinline__ bool mbar_wait_cluster(uint64_t* bar, uint32_t parity) {
  for (uint32_t i = 0; i < (1u << 22); ++i) {
    uint32_t ok;
    asm volatile(
        "{\n\t.reg .pred p;\n\tmbarrier.try_wait.parity.acquire.cluster.shared::cta.b64 p, [%1], "
        "%2;\n\tselp.u32 %0, 1, 0, p;\n\t}"
        : "=r"(ok)
        : "r"(smem_u32(bar)), "r"(parity)
        : "memory");
    if (ok) return true;
  }
  return false;
}

template <int D, bool BF16, int NST, int SPLIT>
__global__ void __launch_bounds__(192, 1)
    prefill_tc_kernel(const __grid_constant__ CUtensorMap tmK,
                      const __grid_constant__ CUtensorMap tmV, const PrefillParams p) {
  using Cfg = PrefillTcCfg<D, NST>;
  extern __shared__ uint8_t smem_raw[];
  __shared__ uint64_t full_bar[NST];
  __shared__ uint64_t empty_bar[NST];
  __shared__ uint64_t s_bar[2], o_bar[2], p_bar[2];
  __shared__ uint64_t ready_bar, recv_bar;              // cluster hand-off (SPLIT == 2)
  __shared__ uint32_t tmem_base;

  // a decode launched behind this kernel as a programmatic dependent may take
  // the SM room this grid leaves as soon as all of its CTAs are running
  if (threadIdx.x == 0) griddep_launch_dependents();
  const int tid = threadIdx.x, lane = tid & 31, warp = tid >> 5;
  const int qt = blockIdx.x / SPLIT, h = blockIdx.y, n = blockIdx.z;
  const int split = SPLIT > 1 ? (int)cluster_rank() : 0;  // the leader is split 0
  const int G = p.G;
  const int q0 = p.cu_q_lens[n];
  const int L = p.cu_q_lens[n + 1] - q0;
  const int ctx = p.seq_lens[n];
  if (L < 0 || L > ctx || ctx > ((p.max_blocks * kBS) << p.ppb_shift)) {
    if (tid == 0 && qt == 0 && h == 0) atomicOr(p.err, PKV_DEVERR_QLEN);
    return;
  }
  const int P0 = ctx - L;
  const int i0 = qt * p.q_tile;
  if (i0 >= L) return;
  const int i1 = min(L, i0 + p.q_tile);
  const int key_end = P0 + i1;                          // keys any row of the tile sees: < key_end
  const int n_pages = (key_end + kBS - 1) / kBS;
  const int n_tiles_all = (key_end + kTcKeys - 1) / kTcKeys;
  // this CTA's share of the key tiles: [t_begin, t_begin + n_tiles)
  const int per_split = (n_tiles_all + SPLIT - 1) / SPLIT;
  const int t_begin = split * per_split;
  const int n_tiles = max(0, min(n_tiles_all, t_begin + per_split) - t_begin);
  const int loaded_end = min(ctx, n_pages * kBS);       // keys with real data in the ring

  const uint32_t raw = smem_u32(smem_raw);
  const uint32_t base = (raw + 1023u) & ~1023u;
  uint8_t* basep = smem_raw + (base - raw);
  const uint32_t sQ = base;
  const uint32_t sKV = base + Cfg::Q_BYTES;
  const uint32_t sP = sKV + NST * Cfg::STAGE_BYTES;
  uint8_t* pQ = basep;
  uint8_t* pKV = basep + Cfg::Q_BYTES;
  uint8_t* pP = pKV + NST * Cfg::STAGE_BYTES;

  if (tid == 0) {
    prefetch_tensormap(&tmK);
    prefetch_tensormap(&tmV);
    for (int s = 0; s < NST; ++s) {
      mbar_init(&full_bar[s], 1);
      mbar_init(&empty_bar[s], 1);
    }
    for (int s = 0; s < 2; ++s) {
      mbar_init(&s_bar[s], 1);
      mbar_init(&o_bar[s], 1);
      mbar_init(&p_bar[s], kTcRows);                    // every softmax thread
    }
    mbar_init(&ready_bar, 1);
    mbar_init(&recv_bar, kTcRows);
    fence_barrier_init();
  }
  if (warp == 0) tc::alloc(&tmem_base, Cfg::TMEM_COLS);

  // ---- query tile into shared memory; rows past the chunk are zero ------------
  const int rows_used = p.q_tile * G;
  const int r = tid;                                    // this thread's tile row (tid < 128)
  const bool rvalid = tid < kTcRows && r < rows_used && i0 + r / G < i1;
  const int qi = i0 + r / G;                            // query token within the chunk
  const int hq = h * G + r % G;                         // query head
  if (tid < kTcRows) {
    const uint16_t* src =
        static_cast<const uint16_t*>(p.q) + ((int64_t)(q0 + (rvalid ? qi : 0)) * p.Hq +
                                             (rvalid ? hq : 0)) * D;
#pragma unroll
    for (int c = 0; c < D / 8; ++c) {
      const uint4 v = rvalid ? *reinterpret_cast<const uint4*>(src + 8 * c)
                             : make_uint4(0u, 0u, 0u, 0u);
      *reinterpret_cast<uint4*>(pQ + (c / 8) * Cfg::Q_BOX + swz128(r, c % 8)) = v;
    }
  }
  fence_proxy_async_smem();                             // the tensor cores read these stores
  tc::fence_before();
  __syncthreads();
  // every CTA of the cluster has its barriers initialised before any remote
  // arrival (the exits above are the same for the whole cluster)
  if constexpr (SPLIT > 1) cluster_sync_all();
  tc::fence_after();
  const uint32_t tm = tmem_base;
  const uint32_t tS = tm;                               // columns [0, 128): S of two tiles
  const uint32_t tO = tm + 2 * kTcKeys;                 // columns [128, 128 + D): O

  if (warp == 4) {
    // ---- producer: K and V tiles through the TMA ring -------------------------------
    if (lane == 0) {
      for (int u = 0; u < n_tiles; ++u) {
        const int t = t_begin + u, st = u % NST;
        if (u >= NST && !mbar_wait_bounded(&empty_bar[st], ((u / NST) - 1) & 1))
          atomicOr(p.err, PKV_DEVERR_TIMEOUT);          // keep going: the consumers time out too
        const int pg0 = t * kTcPages;
        const int npg = min(kTcPages, n_pages - pg0);
        mbar_arrive_expect_tx(&full_bar[st], npg * 2 * kBS * D * 2);
        uint8_t* dst = pKV + st * Cfg::STAGE_BYTES;
        for (int pg = 0; pg < npg; ++pg) {
          const int lp = pg0 + pg;
          int id = p.block_tables[(int64_t)n * p.max_blocks + (lp >> p.ppb_shift)];
          if (id < 0 || id >= p.num_blocks) {
            atomicOr(p.err, PKV_DEVERR_BLOCK_ID);
            id = 0;
          }
          const int z = ((id * p.Hkv + h) << p.ppb_shift) + (lp & ((1 << p.ppb_shift) - 1));
#pragma unroll
          for (int bx = 0; bx < Cfg::NBOX; ++bx) {
            uint8_t* kd = dst + bx * Cfg::KV_BOX + pg * (kBS * 128);
            tma_load_3d(kd, &tmK, &full_bar[st], bx * 64, 0, z);
            tma_load_3d(kd + Cfg::KV_BYTES, &tmV, &full_bar[st], bx * 64, 0, z);
          }
        }
      }
    }
    return;
  }

  constexpr uint32_t ID_S = tc::idesc_f16(kTcRows, kTcKeys, BF16, false);
  constexpr uint32_t ID_O = tc::idesc_f16(kTcRows, D, BF16, true);

  // S of tile t goes to TMEM buffer t % 2 and P of tile t to shared buffer
  // t % 2. s_bar[b] (S ready), p_bar[b] (P written) and o_bar[b] (P.V done)
  // complete once per use of buffer b, so every phase is waited on in order.
  if (warp == 5) {
    // ---- MMA warp: S of tile t as soon as its K lands and its S buffer is
    // free; P.V of tile t - 1 as soon as the softmax has written its P ----------------
    if (lane == 0) {
      // u counts this CTA's tiles; buffers and phases follow u
      auto pv = [&](int u) {
        if (!mbar_wait_bounded(&p_bar[u & 1], (u >> 1) & 1)) atomicOr(p.err, PKV_DEVERR_TIMEOUT);
        tc::fence_after();
        const uint32_t vst = sKV + (u % NST) * Cfg::STAGE_BYTES + Cfg::KV_BYTES;
#pragma unroll
        for (int k = 0; k < kTcKeys / 16; ++k) {
          const uint64_t a = tc::sdesc(sP + (u & 1) * Cfg::P_BYTES + k * 32, 16, 1024);
          const uint64_t b = tc::sdesc(vst + k * 2 * 1024, Cfg::KV_BOX, 1024);
          tc::mma(tO, a, b, ID_O, (u > 0 || k > 0) ? 1u : 0u);
        }
        tc::commit(&o_bar[u & 1]);
        tc::commit(&empty_bar[u % NST]);                // the stage is free once these are done
      };
      for (int u = 0; u < n_tiles; ++u) {
        const int st = u % NST;
        if (!mbar_wait_bounded(&full_bar[st], (u / NST) & 1)) atomicOr(p.err, PKV_DEVERR_TIMEOUT);
        tc::fence_after();
        // buffer u % 2 was last read by the softmax of tile u - 2, whose P the
        // P.V of tile u - 2 (issued below, in order) already waited for
        const uint32_t kst = sKV + st * Cfg::STAGE_BYTES;
#pragma unroll
        for (int k = 0; k < D / 16; ++k) {
          const uint32_t ko = (k % 4) * 32u;
          const uint64_t a = tc::sdesc(sQ + (k / 4) * Cfg::Q_BOX + ko, 16, 1024);
          const uint64_t b = tc::sdesc(kst + (k / 4) * Cfg::KV_BOX + ko, 16, 1024);
          tc::mma(tS + (u & 1) * kTcKeys, a, b, ID_S, k > 0 ? 1u : 0u);
        }
        tc::commit(&s_bar[u & 1]);
        if (u > 0) pv(u - 1);
      }
      if (n_tiles > 0) pv(n_tiles - 1);
    }
    return;
  }

  // ---- warps 0-3: the softmax, one row per thread --------------------------------
  const uint32_t lane_base = (uint32_t)(warp * 32) << 16;
  const int lim = rvalid ? P0 + qi : -1;                // last key this row sees
  const float sl2 = p.qk_scale_log2;
  float m_ref = -INFINITY, l = 0.f;

  for (int u = 0; u < n_tiles; ++u) {
    const int t = t_begin + u;                          // key tile
    const int st = u % NST;
    const int pb = u & 1;
    if (!mbar_wait_bounded(&s_bar[pb], (u >> 1) & 1)) atomicOr(p.err, PKV_DEVERR_TIMEOUT);
    tc::fence_after();
    uint32_t sv[2][32];
    tc::ld32(tS + pb * kTcKeys + lane_base, sv[0]);
    tc::ld32(tS + pb * kTcKeys + lane_base + 32, sv[1]);
    tc::wait_ld();
    // raw scores; keys past this row's causal limit become -inf (only the
    // tiles that cross the limit need the test)
    float x[kTcKeys];
#pragma unroll
    for (int j = 0; j < kTcKeys; ++j) x[j] = __uint_as_float(sv[j / 32][j % 32]);
    if (t * kTcKeys + kTcKeys - 1 > lim) {
#pragma unroll
      for (int j = 0; j < kTcKeys; ++j)
        if (t * kTcKeys + j > lim) x[j] = -INFINITY;
    }
    float mr = -INFINITY;
#pragma unroll
    for (int j = 0; j < kTcKeys; ++j) mr = fmaxf(mr, x[j]);
    const float mx = mr * sl2;                          // the scale is positive: max commutes
    // move the reference max only when the row max outgrows it by 2^8
    const bool move = mx > m_ref + kRescaleLog2;
    const float alpha = move ? (m_ref == -INFINITY ? 0.f : ex2_approx(m_ref - mx)) : 1.f;
    if (move) m_ref = mx;
    if (u > 0 && __any_sync(0xffffffffu, move)) {
      // O must hold every earlier tile before it is scaled
      if (!mbar_wait_bounded(&o_bar[(u - 1) & 1], ((u - 1) >> 1) & 1))
        atomicOr(p.err, PKV_DEVERR_TIMEOUT);
      tc::fence_after();
#pragma unroll
      for (int c0 = 0; c0 < D; c0 += 32) {
        uint32_t ov[32];
        tc::ld32(tO + lane_base + c0, ov);
        tc::wait_ld();
#pragma unroll
        for (int j = 0; j < 32; ++j) ov[j] = __float_as_uint(__uint_as_float(ov[j]) * alpha);
        tc::st32(tO + lane_base + c0, ov);
      }
      tc::wait_st();
    }
    if (u >= 2) {
      // P buffer pb was read by the P.V of tile u - 2
      if (!mbar_wait_bounded(&o_bar[pb], ((u - 2) >> 1) & 1)) atomicOr(p.err, PKV_DEVERR_TIMEOUT);
    }
    const float ms = m_ref == -INFINITY ? 0.f : m_ref;
    uint8_t* pPb = pP + pb * Cfg::P_BYTES;
    float rs = 0.f;
#pragma unroll
    for (int c = 0; c < kTcKeys / 8; ++c) {
      float e[8];
#pragma unroll
      for (int j = 0; j < 8; ++j) {
        e[j] = ex2_approx(fmaf(x[8 * c + j], sl2, -ms));
        rs += e[j];
      }
      const uint4 w = make_uint4(pack16x2<BF16>(e[0], e[1]), pack16x2<BF16>(e[2], e[3]),
                                 pack16x2<BF16>(e[4], e[5]), pack16x2<BF16>(e[6], e[7]));
      *reinterpret_cast<uint4*>(pPb + swz128(r, c)) = w;
    }
    l = l * alpha + rs;
    // V rows with no data for this tile (past the context, or pages not
    // loaded) meet weight 0 in P: zero them so their contents cannot make NaN.
    // Each warp zeroes a quarter; the P.V waits for every softmax thread.
    const int vz = loaded_end - t * kTcKeys;
    if (vz < kTcKeys) {
      uint8_t* vtile = pKV + st * Cfg::STAGE_BYTES + Cfg::KV_BYTES;
      for (int i = tid; i < (kTcKeys - vz) * Cfg::NBOX * 8; i += kTcRows) {
        const int row = vz + i / (Cfg::NBOX * 8), rest = i % (Cfg::NBOX * 8);
        const int bx = rest / 8, chunk = rest % 8;
        *reinterpret_cast<uint4*>(vtile + bx * Cfg::KV_BOX + row * 128 + chunk * 16) =
            make_uint4(0u, 0u, 0u, 0u);
      }
    }
    fence_proxy_async_smem();                           // P and the zeros, for the tensor cores
    tc::fence_before();
    mbar_arrive(&p_bar[pb]);
  }

  // ---- epilogue: O / l to the output rows ------------------------------------------
  if (n_tiles > 0) {
    // MMAs complete in issue order: the last P.V done means all are
    const int ul = n_tiles - 1;
    if (!mbar_wait_bounded(&o_bar[ul & 1], (ul >> 1) & 1)) atomicOr(p.err, PKV_DEVERR_TIMEOUT);
    tc::fence_after();
  }
  // SPLIT == 2: the follower hands its O row, reference max and sum to the
  // leader, in the leader's K/V ring (free once the leader's tiles are done):
  //   O as [D / 4][128 rows] float4 (a warp's rows side by side, no bank
  //   conflicts), then (m, l) as [128 rows][2] fp32.
  float m_other = -INFINITY, l_other = 0.f;
  const uint32_t recv_rows = sKV;
  const uint32_t recv_ml = sKV + kTcRows * D * 4;
  if constexpr (SPLIT > 1) {
    if (split == 0) {
      if (tid == 0) mbar_arrive_remote(cluster_map(smem_u32(&ready_bar), 1));
      if (!mbar_wait_cluster(&recv_bar, 0)) atomicOr(p.err, PKV_DEVERR_TIMEOUT);
      const float2 ml = *reinterpret_cast<const float2*>(basep + (recv_ml - base) + r * 8);
      m_other = ml.x;
      l_other = ml.y;
    } else {
      if (!mbar_wait_cluster(&ready_bar, 0)) atomicOr(p.err, PKV_DEVERR_TIMEOUT);
      const uint32_t dst = cluster_map(recv_rows, 0) + r * 16;
#pragma unroll
      for (int c0 = 0; c0 < D; c0 += 32) {
        uint32_t ov[32];
        tc::ld32(tO + lane_base + c0, ov);
        tc::wait_ld();
#pragma unroll
        for (int j = 0; j < 32; j += 4) {
          const bool has = n_tiles > 0;                  // no tile: nothing accumulated
          st_cluster_v4(dst + ((c0 + j) / 4) * (kTcRows * 16), has ? __uint_as_float(ov[j]) : 0.f,
                        has ? __uint_as_float(ov[j + 1]) : 0.f,
                        has ? __uint_as_float(ov[j + 2]) : 0.f,
                        has ? __uint_as_float(ov[j + 3]) : 0.f);
        }
      }
      st_cluster_v2(cluster_map(recv_ml, 0) + r * 8, m_ref, l);
      mbar_arrive_remote(cluster_map(smem_u32(&recv_bar), 0));
    }
  }
  if (split == 0) {
    // merge the two shares: M = max(m, m'), O = O 2^(m-M) + O' 2^(m'-M)
    const float M = fmaxf(m_ref, m_other);
    const float w0 = m_ref == -INFINITY ? 0.f : SPLIT == 1 ? 1.f : ex2_approx(m_ref - M);
    const float w1 = m_other == -INFINITY ? 0.f : ex2_approx(m_other - M);
    const float L = l * w0 + l_other * w1;
    const float inv = L > 0.f ? 1.f / L : 0.f;
    const float a0 = w0 * inv, a1 = w1 * inv;
    const float4* orecv = reinterpret_cast<const float4*>(basep + (recv_rows - base)) + r;
    uint16_t* orow = static_cast<uint16_t*>(p.out) + ((int64_t)(q0 + (rvalid ? qi : 0)) * p.Hq +
                                                      (rvalid ? hq : 0)) * D;
#pragma unroll
    for (int c0 = 0; c0 < D; c0 += 32) {
      uint32_t ov[32];
      tc::ld32(tO + lane_base + c0, ov);
      tc::wait_ld();
      if (rvalid) {
        float f[32];
#pragma unroll
        for (int j = 0; j < 32; j += 4) {
          float4 o1 = make_float4(0.f, 0.f, 0.f, 0.f);
          if constexpr (SPLIT > 1) o1 = orecv[((c0 + j) / 4) * kTcRows];
          f[j] = __uint_as_float(ov[j]) * a0 + o1.x * a1;
          f[j + 1] = __uint_as_float(ov[j + 1]) * a0 + o1.y * a1;
          f[j + 2] = __uint_as_float(ov[j + 2]) * a0 + o1.z * a1;
          f[j + 3] = __uint_as_float(ov[j + 3]) * a0 + o1.w * a1;
        }
#pragma unroll
        for (int c = 0; c < 4; ++c) {
          const uint4 w = make_uint4(
              pack16x2<BF16>(f[8 * c + 0], f[8 * c + 1]), pack16x2<BF16>(f[8 * c + 2], f[8 * c + 3]),
              pack16x2<BF16>(f[8 * c + 4], f[8 * c + 5]), pack16x2<BF16>(f[8 * c + 6], f[8 * c + 7]));
          *reinterpret_cast<uint4*>(orow + c0 + 8 * c) = w;
        }
      }
    }
    if (rvalid && p.out_lse != nullptr)
      p.out_lse[(int64_t)(q0 + qi) * p.Hq + hq] = L > 0.f ? (M + log2f(L)) * kLn2 : -INFINITY;
  }
  tc::fence_before();
  named_barrier(1, kTcRows);
  if (warp == 0) tc::dealloc(tm, Cfg::TMEM_COLS);
}

template <int D, bool BF16, int SPLIT>
static pkv_status launch_prefill_tc_s(const PrefillParams& q, const CUtensorMap& tmK,
                                      const CUtensorMap& tmV, cudaStream_t stream, int dev) {
  constexpr int NST = 3;
  using Cfg = PrefillTcCfg<D, NST>;
  static_assert(kTcRows * D * 4 + kTcRows * 8 <= NST * Cfg::STAGE_BYTES,
                "the follower's rows must fit in the leader's ring");
  auto kern = prefill_tc_kernel<D, BF16, NST, SPLIT>;
  static bool attr_set[64] = {};
  if (!attr_set[dev]) {
    if (cudaFuncSetAttribute(kern, cudaFuncAttributeMaxDynamicSharedMemorySize,
                             Cfg::SMEM_BYTES) != cudaSuccess)
      return PKV_ERR_CUDA;
    attr_set[dev] = true;
  }
  const int tiles = (q.max_q_len + q.q_tile - 1) / q.q_tile;
  cudaLaunchAttribute attr[1];
  attr[0].id = cudaLaunchAttributeClusterDimension;
  attr[0].val.clusterDim.x = SPLIT;
  attr[0].val.clusterDim.y = 1;
  attr[0].val.clusterDim.z = 1;
  cudaLaunchConfig_t cfg = {};
  cfg.gridDim = dim3(tiles * SPLIT, q.Hkv, q.num_seqs);
  cfg.blockDim = dim3(192);
  cfg.dynamicSmemBytes = Cfg::SMEM_BYTES;
  cfg.stream = stream;
  cfg.attrs = attr;
  cfg.numAttrs = 1;
  return cudaLaunchKernelEx(&cfg, kern, tmK, tmV, q) == cudaSuccess ? PKV_OK : PKV_ERR_CUDA;
}

// One CTA per query tile when that fills at least half of the GPU (or other
// work shares it); otherwise a cluster of two per tile, each taking half of
// the key tiles.
template <int D, bool BF16>
static pkv_status launch_prefill_tc_t(const PrefillParams& p, const CUtensorMap& tmK,
                                      const CUtensorMap& tmV, cudaStream_t stream,
                                      bool may_split) {
  int dev = 0;
  if (cudaGetDevice(&dev) != cudaSuccess || dev < 0 || dev >= 64) return PKV_ERR_CUDA;
  static int sms[64] = {};
  if (sms[dev] == 0 &&
      cudaDeviceGetAttribute(&sms[dev], cudaDevAttrMultiProcessorCount, dev) != cudaSuccess)
    return PKV_ERR_CUDA;
  PrefillParams q = p;
  q.q_tile = kTcRows / p.G;
  const int64_t ctas = (int64_t)((q.max_q_len + q.q_tile - 1) / q.q_tile) * q.Hkv * q.num_seqs;
  if (may_split && 2 * ctas <= sms[dev]) return launch_prefill_tc_s<D, BF16, 2>(q, tmK, tmV, stream, dev);
  return launch_prefill_tc_s<D, BF16, 1>(q, tmK, tmV, stream, dev);
}

bool prefill_tc_supported(int head_dim, pkv_dtype kv_dtype) {
  return (head_dim == 64 || head_dim == 128) && kv_dtype != PKV_FP8_E4M3;
}

pkv_status launch_prefill_tc(const PrefillParams& p, int head_dim, pkv_dtype kv_dtype,
                             const CUtensorMap& tmK, const CUtensorMap& tmV,
                             cudaStream_t stream, bool may_split) {
  const bool bf = kv_dtype == PKV_BF16;
  if (head_dim == 128)
    return bf ? launch_prefill_tc_t<128, true>(p, tmK, tmV, stream, may_split)
              : launch_prefill_tc_t<128, false>(p, tmK, tmV, stream, may_split);
  return bf ? launch_prefill_tc_t<64, true>(p, tmK, tmV, stream, may_split)
            : launch_prefill_tc_t<64, false>(p, tmK, tmV, stream, may_split);
}

}  // namespace pkv
