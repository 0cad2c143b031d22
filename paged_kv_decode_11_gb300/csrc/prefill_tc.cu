// prefill_tc.cu — causal chunked-prefill attention on the fifth-generation
// tensor cores (tcgen05): 16-bit caches at head_dim 64, 128 and 256, E4M3
// caches at 64 and 128.
//
// Follows "Chunked Prefill" (Litellama, Features: a long prompt enters the
// batch as chunks of new query tokens attending their cached context) with
// the causal alignment of the library: query row i of a chunk of L tokens on
// P cached ones sees keys 0 .. P + i. Same result as prefill.cu (online
// softmax over key tiles, fp32 accumulation); the contraction runs on the
// tensor cores with its accumulators in tensor memory:
//
//   CTA = (query tile, KV head, chunk). Tile rows are (query token, head of
//   the GQA group) pairs, 128 of them: the MMA M. Two producer warps stream
//   the K and the V tiles of 4 pages (64 keys) through two TMA rings (for an
//   E4M3 cache through a staging ring, converting each tile to f16). One
//   MMA warp issues, whichever is ready first,
//     S[128 x 64]  = Q[128 x D] . K_tile^T   (K-major A and B, fp32 in TMEM)
//   and, once the softmax has written P,
//     O_g[128 x D] += P[128 x 64] . V_tile   (V read MN-major)
//   Softmax groups of four warps take the key tiles in turn (two groups up to
//   D = 128: group g the tiles u with u % 2 == g; one at D = 256), each with
//   its own S buffers, P buffers and O accumulator, so one group's softmax
//   runs while the other waits on the tensor cores. In a group, warp w owns
//   TMEM lanes 32 (w % 4) ..: thread r holds row r of S, so the row max and
//   sum need no shuffles. O_g and the row sum are kept relative to a
//   reference max that moves only when the row max grows by more than 2^8,
//   so O in TMEM is rescaled rarely. At the end the groups' (O, max, sum)
//   are merged by log-sum-exp, the same softmax. When a small grid leaves
//   SMs idle, a cluster of two CTAs splits each tile's keys and the two
//   merge the same way through distributed shared memory.
//
// Shared memory: Q [D/64][128 rows][128 B], then NST stages of
// K [D/64][4 pages][16 rows][128 B], NST stages of V (same), then two P
// buffers [128 rows][128 B] per group (S has two TMEM buffers per group
// likewise, so the S product of a group's next tile runs while its softmax
// does), all in the 128-byte swizzled layout (tc.cuh), then (E4M3) the K and
// V staging rings. Placing the four pages of a 64-byte column block back to
// back gives every operand a uniform 1 KB stride between 8-row groups.
#include <cuda.h>
#include "common.cuh"
#include "launch_prefill.h"
#include "tc.cuh"

namespace pkv {

constexpr int kTcRows = kPrefillTcRows;       // query rows per CTA (MMA M)
constexpr float kRescaleLog2 = 8.f;           // reference-max slack (log2 units)

// NG softmax groups of four warps (two up to D = 128; one at D = 256, whose O
// takes 256 TMEM columns), then PK K producer warps, the MMA warp and PV V
// producer warps. One warp's TMA loads complete at about 16 GB/s for
// page-sized (2 KB) boxes on GB300, whatever the ring depth, and the rate
// grows with the number of issuing warps: with 128-key tiles a 16-bit cache
// has 4 K and 3 V producers, which take the boxes of a tile in turn, and the
// producer warpgroups hand registers to the softmax ones (REALLOC). KV8: an
// E4M3 cache. Its tiles land by TMA in an NSS-deep staging ring and one
// producer warp per operand converts them to f16 (exact: E4M3 is a subset
// of f16) into the rings the MMAs read.
// ALONE: nothing else runs on the GPU beside this grid (a chunk call of its
// own, not the prefill half of a varlen step).
template <int D, int NST, bool KV8 = false, bool ALONE = true>
struct PrefillTcCfg {
  // 128-key tiles (WIDE): one softmax group over two S buffers in tensor
  // memory, P written over its own S; otherwise two groups up to D = 128
  static constexpr bool WIDE = ALONE && !KV8 && D <= 128;
  static constexpr int NG = WIDE ? 1 : (D <= 128 ? 2 : 1);
  // keys per tile (the S MMA's N): 128 for 16-bit caches at D <= 128 running
  // alone, with one S buffer (TMEM) and one P buffer (shared) per group; 64
  // otherwise, with two. Beside a decode grid the 64-key kernel, whose loads
  // press less on L2, made the varlen step faster (102.7 against 104.4 us on
  // the mixed step), while alone the 128-key one is faster at every size.
  static constexpr int KEYS = WIDE ? 128 : 64;
  static constexpr int PAGES = KEYS / kBS;                   // 16-token pages per tile
  // S (and P) buffers per group: three for the one group of 128-key tiles
  // (3 x 128 S columns and 128 of O fill the 512), so an S product waits for
  // the P.V two tiles back, not the one before
  static constexpr int NSB = WIDE ? 3 : 2;
  // P in tensor memory (128-key tiles): the softmax writes P over its own S
  // columns (two 16-bit values per 32-bit column) and the P.V MMAs read it
  // there, which frees the shared P buffers for deeper K and V rings
  static constexpr bool PTM = WIDE;
  static constexpr int PK = WIDE ? 4 : 1;
  static constexpr int PV = WIDE ? 3 : 1;
  static constexpr int WARPS = 4 * NG + PK + 1 + PV;
  static constexpr int THREADS = WARPS * 32;
  static constexpr int W_K = 4 * NG, W_MMA = 4 * NG + PK, W_V = 4 * NG + PK + 1;
  // 16 warps (4 per SM sub-partition) launch at 128 registers a thread: the
  // softmax warpgroups rise to REG_SOFTMAX, the K producers (warpgroup 2) and
  // the MMA warp with the V producers (warpgroup 3) fall to REG_K / REG_MV
  static constexpr bool REALLOC = WARPS == 16;
  static constexpr int REG_SOFTMAX = 184, REG_K = 48, REG_MV = 56;
  static_assert(!REALLOC || (NG == 2 && W_MMA == 12), "warpgroups: 2 softmax, K, MMA + V");
  // registers the warpgroups hold after the moves; the launcher checks that
  // the kernel was built to launch with at least this many (512 threads)
  static constexpr int REG_TOTAL = 256 * REG_SOFTMAX + 128 * (REG_K + REG_MV);
  static_assert(!REALLOC || REG_TOTAL <= 512 * 128, "more than 16 warps can hold");
  static constexpr int NBOX = D / 64;                        // 128-byte column blocks per row
  static constexpr int Q_BOX = kTcRows * 128;                // one column block of Q
  static constexpr int Q_BYTES = NBOX * Q_BOX;
  static constexpr int KV_BOX = PAGES * kBS * 128;           // one column block of a K/V tile
  static constexpr int KV_BYTES = NBOX * KV_BOX;            // one K (or V) tile
  static constexpr int RING_BYTES = NST * KV_BYTES;          // one ring (K, then V)
  static constexpr int P_CB = kTcRows * 128;                 // 64 keys of a P buffer
  static constexpr int P_BYTES = (KEYS / 64) * P_CB;         // one P buffer (NSB per group)
  static constexpr int NSS = KV8 ? 4 : 0;                    // staging stages per operand
  static constexpr int STG_PAGE = kBS * D;                   // one E4M3 page
  static constexpr int STG_BYTES = PAGES * STG_PAGE;         // one staged E4M3 tile
  static constexpr int SMEM_BYTES =
      1024 + Q_BYTES + 2 * RING_BYTES + (PTM ? 0 : NSB * NG * P_BYTES) + 2 * NSS * STG_BYTES;
  static constexpr uint32_t TMEM_COLS = 512;                  // 2 S buffers and O per group
  static_assert(NG * (NSB * KEYS + D) <= (int)TMEM_COLS, "tensor memory");
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
// Split cluster barrier: every thread arrives once after the CTA's barriers
// are initialised and waits once before its first access to another CTA.
__device__ __forceinline__ void cluster_arrive() {
  asm volatile("barrier.cluster.arrive.release.aligned;" ::: "memory");
}
__device__ __forceinline__ void cluster_wait() {
  asm volatile("barrier.cluster.wait.acquire.aligned;" ::: "memory");
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

// n consecutive fp32 TMEM columns (n = 16 or 32) of this thread's lane.
template <int N>
__device__ __forceinline__ void tmem_ld(uint32_t taddr, uint32_t (&v)[N]) {
  static_assert(N == 16 || N == 32, "16 or 32 columns");
  if constexpr (N == 32) tc::ld32(taddr, v);
  else tc::ld16(taddr, v);
}

// KV: the cache type; the MMAs take bf16 operands for a bf16 cache and f16
// ones otherwise (an E4M3 cache is converted to f16, and bf16 queries with
// it). QBF16: the query and output type.
template <int D, int KV, bool QBF16, int NST, int SPLIT, bool ALONE>
__global__ void __launch_bounds__(PrefillTcCfg<D, NST, KV == KV_E4M3, ALONE>::THREADS, 1)
    prefill_tc_kernel(const __grid_constant__ CUtensorMap tmQ,
                      const __grid_constant__ CUtensorMap tmK,
                      const __grid_constant__ CUtensorMap tmV, const PrefillParams p) {
  constexpr bool KV8 = KV == KV_E4M3;
  constexpr bool BF16 = KV == KV_BF16;                  // MMA operand type
  using Cfg = PrefillTcCfg<D, NST, KV8, ALONE>;
  constexpr int NG = Cfg::NG;
  constexpr int NSS = Cfg::NSS > 0 ? Cfg::NSS : 1;
  constexpr int kTcKeys = Cfg::KEYS, kTcPages = Cfg::PAGES, NSB = Cfg::NSB;
  extern __shared__ uint8_t smem_raw[];
  // per ring stage: K (or V) tile ready, K (or V) tile read
  __shared__ uint64_t full_k[NST], empty_k[NST], full_v[NST], empty_v[NST];
  __shared__ uint64_t stg_k[NSS], stg_v[NSS];           // KV8: staged E4M3 tile landed
  // per softmax group g and buffer b: S ready, P written, P.V done
  __shared__ uint64_t s_bar[NG][NSB], o_bar[NG][NSB], p_bar[NG][NSB];
  __shared__ uint64_t ready_bar, recv_bar;              // cluster hand-off (SPLIT == 2)
  __shared__ uint64_t done_bar;                         // PTM: every MMA of the CTA is done
  __shared__ uint64_t q_bar;                            // 16-bit cache: the query tile landed
  __shared__ uint32_t tmem_base;
  __shared__ float s_qpow[KV8 ? kTcRows : 1];           // KV8, bf16 q: 2^shift of each row

  // a decode launched behind this kernel as a programmatic dependent may take
  // the SM room this grid leaves as soon as all of its CTAs are running
  if (threadIdx.x == 0) griddep_launch_dependents();
  const int tid = threadIdx.x, lane = tid & 31, warp = tid >> 5;
  const int qt = blockIdx.x / SPLIT, h = blockIdx.y, n = blockIdx.z;
  const int split = SPLIT > 1 ? (int)cluster_rank() : 0;
  const int G = p.G;
  const int q0 = p.cu_q_lens[n];
  const int L = p.cu_q_lens[n + 1] - q0;
  const int ctx = p.seq_lens[n];
  // a chunk longer than its context, or whose rows are not rows of q and out
  if (L < 0 || L > ctx || q0 < 0 || q0 > p.q_rows - L ||
      ctx > ((p.max_blocks * kBS) << p.ppb_shift)) {
    if (tid == 0 && qt == 0 && h == 0) atomicOr(p.err, PKV_DEVERR_QLEN);
    return;
  }
  const int P0 = ctx - L;
  const int i0 = qt * p.q_tile;
  if (i0 >= L) return;
  const int i1 = min(L, i0 + p.q_tile);
  const int rows_used = p.q_tile * G;                   // tile rows holding (token, head) pairs
  const int key_end = P0 + i1;                          // keys any row of the tile sees: < key_end
  const int n_pages = (key_end + kBS - 1) / kBS;
  const int n_tiles_all = (key_end + kTcKeys - 1) / kTcKeys;
  // this CTA's share of the key tiles: [t_begin, t_begin + n_tiles); its
  // local tile u goes to softmax group u % NG
  const int per_split = (n_tiles_all + SPLIT - 1) / SPLIT;
  const int t_begin = split * per_split;
  const int n_tiles = max(0, min(n_tiles_all, t_begin + per_split) - t_begin);
  const int loaded_end = min(ctx, n_pages * kBS);       // keys with real data in the ring

  const uint32_t raw = smem_u32(smem_raw);
  const uint32_t base = (raw + 1023u) & ~1023u;
  uint8_t* basep = smem_raw + (base - raw);
  const uint32_t sQ = base;
  const uint32_t sKV = base + Cfg::Q_BYTES;
  const uint32_t sV = sKV + Cfg::RING_BYTES;           // V ring after the K ring
  const uint32_t sP = sV + Cfg::RING_BYTES;            // [group][buffer] P tiles
  uint8_t* pQ = basep;
  uint8_t* pKV = basep + Cfg::Q_BYTES;
  uint8_t* pV = pKV + Cfg::RING_BYTES;
  uint8_t* pP = pV + Cfg::RING_BYTES;
  uint8_t* pStg = pP + (Cfg::PTM ? 0 : NSB * NG * Cfg::P_BYTES);   // KV8: K, then V staging

  bool failed = false;                                  // a wait ran out: stop waiting
  auto wait = [&](uint64_t* bar, uint32_t parity) {
    if (failed) return;
    if (!mbar_wait_bounded(bar, parity)) {
      failed = true;
      atomicOr(p.err, PKV_DEVERR_TIMEOUT);
    }
  };

  // ---- producers: warps W_K .. W_K + PK - 1 stream the K tiles and warps
  // W_V .. W_V + PV - 1 the V tiles, each operand through its own TMA ring, so
  // a K stage is refilled as soon as its S product is done and V stages wait
  // only on the P.V products; of the np producers of an operand, producer pw
  // loads boxes (16 rows x 128 B) pw, pw + np, .. of each tile. A producer's
  // lanes look up the page rows 32 pages at a time, one chunk ahead, so no
  // block-table read waits in front of a TMA issue; lane 0 issues the loads.
  const int pg_begin = t_begin * kTcPages;
  const int pg_end = min(n_pages, (t_begin + n_tiles) * kTcPages);
  auto page_row = [&](int lp) -> int {
    if (lp >= pg_end) return 0;
    int id = p.block_tables[(int64_t)n * p.max_blocks + (lp >> p.ppb_shift)];
    if (id < 0 || id >= p.num_blocks) {
      atomicOr(p.err, PKV_DEVERR_BLOCK_ID);
      id = 0;
    }
    return ((id * p.Hkv + h) << p.ppb_shift) + (lp & ((1 << p.ppb_shift) - 1));
  };
  static_assert(32 % kTcPages == 0, "a tile's pages lie in one chunk");
  const bool k_warp = warp >= Cfg::W_K && warp < Cfg::W_K + Cfg::PK;
  const bool v_warp = warp >= Cfg::W_V && warp < Cfg::W_V + Cfg::PV;
  const bool producer = k_warp || v_warp;
  const int np = k_warp ? Cfg::PK : Cfg::PV;              // producers of this operand
  const int pw = k_warp ? warp - Cfg::W_K : warp - Cfg::W_V;   // boxes pw, pw + np, ..
  const CUtensorMap* tmap = k_warp ? &tmK : &tmV;
  uint64_t* full_x = k_warp ? full_k : full_v;
  uint64_t* empty_x = k_warp ? empty_k : empty_v;
  uint64_t* stg_x = k_warp ? stg_k : stg_v;
  uint8_t* ring_x = k_warp ? pKV : pV;
  uint8_t* stage_x = pStg + (k_warp ? 0 : NSS * Cfg::STG_BYTES);
  int z_cur = 0, z_next = 0, chunk = 0;
  // TMA loads of tile u: into ring stage u % NST, or (KV8) into staging
  // stage u % NSS, one box per E4M3 page
  auto issue = [&](int u) {
    const int t = t_begin + u;
    if ((u * kTcPages) / 32 != chunk) {
      z_cur = z_next;
      ++chunk;
      z_next = page_row(pg_begin + 32 * (chunk + 1) + lane);
    }
    const int pg0 = t * kTcPages;
    const int npg = min(kTcPages, n_pages - pg0);
    if constexpr (KV8) {
      uint64_t* bar = &stg_x[u % NSS];
      if (lane == 0) mbar_arrive_expect_tx(bar, npg * Cfg::STG_PAGE);
      uint8_t* dst = stage_x + (u % NSS) * Cfg::STG_BYTES;
      for (int pg = 0; pg < npg; ++pg) {
        const int z = __shfl_sync(0xffffffffu, z_cur, (u * kTcPages + pg) % 32);
        if (lane == 0) tma_load_3d(dst + pg * Cfg::STG_PAGE, tmap, bar, 0, 0, z);
      }
    } else {
      const int st = u % NST;
      const int nbx = npg * Cfg::NBOX;                   // boxes (16 rows x 128 B) of the tile
      const int mine = pw < nbx ? (nbx - pw + np - 1) / np : 0;
      if (lane == 0) mbar_arrive_expect_tx(&full_x[st], mine * kBS * 128);
      uint8_t* dst = ring_x + st * Cfg::KV_BYTES;
      for (int b = pw; b < nbx; b += np) {
        const int pg = b / Cfg::NBOX, bx = b % Cfg::NBOX;
        const int z = __shfl_sync(0xffffffffu, z_cur, (u * kTcPages + pg) % 32);
        if (lane == 0)
          tma_load_3d(dst + bx * Cfg::KV_BOX + pg * (kBS * 128), tmap, &full_x[st], bx * 64, 0, z);
      }
    }
  };
  // KV8: the warp turns staged tile u into f16 in ring stage u % NST (rows
  // past the loaded keys become zeros), then refills the staging stage
  auto convert = [&](int u) {
    using Geo8 = PageGeom<D, KV_E4M3>;
    constexpr int CPR = D / 16;                          // 16-element chunks per row
    const int t = t_begin + u, st = u % NST;
    wait(&stg_x[u % NSS], (u / NSS) & 1);
    if (u >= NST) wait(&empty_x[st], ((u / NST) - 1) & 1);
    const uint8_t* src = stage_x + (u % NSS) * Cfg::STG_BYTES;
    const int valid = loaded_end - t * kTcKeys;          // rows of this tile holding keys
    // lane = (row in a group of RPI rows, 16-element chunk x of the row): x is
    // fixed per lane, so the chunk's column block and swizzle slot are too
    constexpr int RPI = 32 / CPR;
    const int x = lane % CPR, rsub = lane / CPR;
    uint8_t* dcol = ring_x + st * Cfg::KV_BYTES + (x / 4) * Cfg::KV_BOX;
    const int c16 = 2 * (x % 4);
#pragma unroll
    for (int k = 0; k < kTcKeys / RPI; ++k) {
      const int row = k * RPI + rsub;
      // rows of pages not loaded hold stale bytes: read anyway, zero below
      const uint4 e = *reinterpret_cast<const uint4*>(src + (row / kBS) * Cfg::STG_PAGE +
                                                      Geo8::row_off(row % kBS, 16 * x));
      const bool keep = row < valid;
      const uint4 lo = keep ? make_uint4(e4m3x2_to_f16x2(e.x & 0xFFFFu), e4m3x2_to_f16x2(e.x >> 16),
                                         e4m3x2_to_f16x2(e.y & 0xFFFFu), e4m3x2_to_f16x2(e.y >> 16))
                            : make_uint4(0u, 0u, 0u, 0u);
      const uint4 hi = keep ? make_uint4(e4m3x2_to_f16x2(e.z & 0xFFFFu), e4m3x2_to_f16x2(e.z >> 16),
                                         e4m3x2_to_f16x2(e.w & 0xFFFFu), e4m3x2_to_f16x2(e.w >> 16))
                            : make_uint4(0u, 0u, 0u, 0u);
      // elements 16 x .. 16 x + 15: 16-byte chunks c16 and c16 + 1 of the row
      *reinterpret_cast<uint4*>(dcol + swz128(row, c16)) = lo;
      *reinterpret_cast<uint4*>(dcol + swz128(row, c16 + 1)) = hi;
    }
    fence_proxy_async_smem();                            // the tensor cores read these stores
    mbar_arrive(&full_x[st]);                            // one arrival per lane
    __syncwarp();
    fence_proxy_async_smem();                            // before the staging stage is refilled
    if (u + NSS < n_tiles) issue(u + NSS);
  };
  if (warp == Cfg::W_K) {
    // the first K producer sets up the barriers and starts the query tile's
    // load; the K producers then start K tile 0 (below), while the other warps
    // allocate tensor memory
    if (lane == 0) {
      prefetch_tensormap(&tmK);
      prefetch_tensormap(&tmV);
      for (int s = 0; s < NST; ++s) {
        mbar_init(&full_k[s], KV8 ? 32 : Cfg::PK);      // KV8: the converting warp's lanes
        mbar_init(&empty_k[s], 1);
        mbar_init(&full_v[s], KV8 ? 32 : Cfg::PV);
        mbar_init(&empty_v[s], 1);
      }
      for (int s = 0; s < NSS; ++s) {
        mbar_init(&stg_k[s], 1);
        mbar_init(&stg_v[s], 1);
      }
      for (int g = 0; g < NG; ++g)
        for (int b = 0; b < NSB; ++b) {
          mbar_init(&s_bar[g][b], 1);
          mbar_init(&o_bar[g][b], 1);
          mbar_init(&p_bar[g][b], kTcRows);             // every thread of the group
        }
      mbar_init(&ready_bar, 1);
      mbar_init(&recv_bar, NG * kTcRows);
      mbar_init(&done_bar, 1);
      mbar_init(&q_bar, 1);
      fence_barrier_init();
      if constexpr (!KV8) {
        // the query tile by TMA ahead of every K and V tile: rows 0 ..
        // rows_used - 1 of each 64-column block, tokens past the queries as zeros
        mbar_arrive_expect_tx(&q_bar, Cfg::NBOX * rows_used * 128);
        for (int c = 0; c < Cfg::NBOX; ++c)
          tma_load_3d(pQ + c * Cfg::Q_BOX, &tmQ, &q_bar, c * 64, h * G, q0 + i0);
      }
    }
    __syncwarp();
  }
  if (producer) {
    z_cur = page_row(pg_begin + lane);
    z_next = page_row(pg_begin + 32 + lane);
  }
  if constexpr (KV8) {
    if (warp == Cfg::W_K)
      for (int u = 0; u < Cfg::NSS && u < n_tiles; ++u) issue(u);
  } else if (producer) {
    // the first S product needs only the query tile and K tile 0: the K
    // producers load their shares of K tile 0 right behind the query tile, as
    // soon as the barriers are set up (a barrier of the producer warps alone),
    // ahead of the grid-wide burst of the other first stages, which start
    // after the CTA barrier. (Holding that burst back until the query tile had
    // landed made the 512-on-1500 chunk 0.6 us slower.)
    named_barrier(2, (Cfg::PK + Cfg::PV) * 32);
    if (k_warp && n_tiles > 0) issue(0);
  }
  if (warp == 0) tc::alloc(&tmem_base, Cfg::TMEM_COLS);

  // ---- query tile into shared memory. 16-bit cache: by TMA (issued above), the
  // last softmax group zeroing the rows no pair uses; rows of tokens past the
  // chunk hold the next tokens' queries (their results are never stored). E4M3
  // cache: loaded (and scaled to f16) by the last softmax group, rows past the
  // chunk zero ----------------------------------------------------------------------
  const int grp = warp >> 2;                            // softmax group (warps 0 .. 4 NG - 1)
  const int r = tid & (kTcRows - 1);                    // this thread's tile row
  const int qi = i0 + r / G;                            // query token within the chunk
  const int hq = h * G + r % G;                         // query head
  const bool rvalid = r < rows_used && qi < i1;
  if (!KV8 && grp == NG - 1 && r >= rows_used) {
    // rows no (token, head) pair uses (G not dividing the tile): zeros
#pragma unroll
    for (int c = 0; c < D / 8; ++c)
      *reinterpret_cast<uint4*>(pQ + (c / 8) * Cfg::Q_BOX + swz128(r, c % 8)) =
          make_uint4(0u, 0u, 0u, 0u);
  }
  if (KV8 && grp == NG - 1) {
    const uint16_t* src =
        static_cast<const uint16_t*>(p.q) + ((int64_t)(q0 + (rvalid ? qi : 0)) * p.Hq +
                                             (rvalid ? hq : 0)) * D;
    // the MMAs run in f16 against an E4M3 cache: a bf16 query row is scaled by
    // 2^-shift (q_f16_shift of the row) and rounded to f16; its scores are
    // scaled back by 2^shift in the softmax
    float qinv = 1.f;
    if constexpr (KV8 && QBF16) {
      uint32_t mx = 0u;
      if (rvalid) {
#pragma unroll 4
        for (int c = 0; c < D / 8; ++c) {
          const uint4 v = *reinterpret_cast<const uint4*>(src + 8 * c);
          mx = max(mx, max(max(bf16x2_max_abs(v.x), bf16x2_max_abs(v.y)),
                           max(bf16x2_max_abs(v.z), bf16x2_max_abs(v.w))));
        }
      }
      const int sh = rvalid ? q_f16_shift(mx) : 0;
      qinv = pow2f(-sh);
      s_qpow[r] = pow2f(sh);
    }
#pragma unroll
    for (int c = 0; c < D / 8; ++c) {
      uint4 v = rvalid ? *reinterpret_cast<const uint4*>(src + 8 * c)
                       : make_uint4(0u, 0u, 0u, 0u);
      if constexpr (KV8 && QBF16) {
        v = make_uint4(bf16x2_to_f16x2_scaled(v.x, qinv), bf16x2_to_f16x2_scaled(v.y, qinv),
                       bf16x2_to_f16x2_scaled(v.z, qinv), bf16x2_to_f16x2_scaled(v.w, qinv));
      }
      *reinterpret_cast<uint4*>(pQ + (c / 8) * Cfg::Q_BOX + swz128(r, c % 8)) = v;
    }
  }
  fence_proxy_async_smem();                             // the tensor cores read these stores
  tc::fence_before();
  __syncthreads();
  // the barriers of every CTA of the cluster are initialised once all have
  // arrived; each thread waits for that before its first remote access
  if constexpr (SPLIT > 1) cluster_arrive();
  tc::fence_after();
  const uint32_t tm = tmem_base;
  // TMEM columns: S of group g, buffer b at KEYS (NSB g + b); O of group g after them
  const uint32_t tS = tm;
  const uint32_t tO = tm + NSB * NG * kTcKeys;

  // ---- producer and MMA warps (warpgroups 2 and 3 when registers move) ----------------
  if (warp >= Cfg::W_K) {
    if constexpr (Cfg::REALLOC) {
      if (warp >= Cfg::W_MMA) tc::reg_lower<Cfg::REG_MV>();
      else tc::reg_lower<Cfg::REG_K>();
    }
    if (producer) {
      // KV8: the V producer starts once the barriers are set up (after the CTA barrier)
      if constexpr (KV8) {
        if (!k_warp)
          for (int u = 0; u < Cfg::NSS && u < n_tiles; ++u) issue(u);
        for (int u = 0; u < n_tiles; ++u) convert(u);
      } else {
        for (int u = k_warp ? 1 : 0; u < n_tiles; ++u) {
          if (u >= NST) wait(&empty_x[u % NST], ((u / NST) - 1) & 1);
          issue(u);
        }
      }
      __syncwarp();
      if constexpr (SPLIT > 1) cluster_wait();
      return;
    }

    constexpr uint32_t ID_S = tc::idesc_f16(kTcRows, kTcKeys, BF16, false);
    constexpr uint32_t ID_O = tc::idesc_f16(kTcRows, D, BF16, true);

    // Tile u belongs to group g = u % NG as its j-th tile (j = u / NG): S goes to
    // TMEM buffer (g, j % NSB), P to shared buffer (g, j % NSB), P.V accumulates
    // into O of group g. Each barrier (g, b) completes once per use of its
    // buffer (use j / NSB), so every phase is waited on in order.
    if (warp == Cfg::W_MMA) {
      // ---- MMA warp: issues whatever is ready, S products first. S of tile u
      // needs its K tile landed and its TMEM buffer free: the buffer's previous
      // tile is u - NSB NG, whose softmax finished reading it before writing the
      // P that the P.V of u - NSB NG waited for, so S may run up to NSB NG tiles
      // ahead of the P.V products. P.V of tile u (in order) needs the group's P.
      if (lane == 0) {
        int us = 0, up = 0;                               // next S, next P.V
        uint32_t idle = 0;
        if constexpr (!KV8) wait(&q_bar, 0);             // the query tile (TMA)
        // PTM: the P.V that read P from this S buffer (its previous tile)
        // must be complete, not just issued, before S overwrites it
        auto s_ready = [&]() {
          return us < n_tiles && us < up + NSB * NG &&
                 mbar_test_wait(&full_k[us % NST], (us / NST) & 1) &&
                 (!Cfg::PTM || us < NSB * NG ||
                  mbar_test_wait(&o_bar[us % NG][(us / NG) % NSB], (((us / NG) - NSB) / NSB) & 1));
        };
        auto s_issue = [&]() {
          const int g = us % NG, j = us / NG;
          tc::fence_after();
          const uint32_t kst = sKV + (us % NST) * Cfg::KV_BYTES;
  #pragma unroll
          for (int k = 0; k < D / 16; ++k) {
            const uint32_t ko = (k % 4) * 32u;
            const uint64_t a = tc::sdesc(sQ + (k / 4) * Cfg::Q_BOX + ko, 16, 1024);
            const uint64_t bd = tc::sdesc(kst + (k / 4) * Cfg::KV_BOX + ko, 16, 1024);
            tc::mma(tS + (NSB * g + j % NSB) * kTcKeys, a, bd, ID_S, k > 0 ? 1u : 0u);
          }
          tc::commit(&s_bar[g][j % NSB]);
          tc::commit(&empty_k[us % NST]);                 // the K stage is free once S is done
          ++us;
        };
        auto pv_ready = [&]() {
          return up < us && mbar_test_wait(&p_bar[up % NG][(up / NG) % NSB], ((up / NG) / NSB) & 1) &&
                 mbar_test_wait(&full_v[up % NST], (up / NST) & 1);
        };
        auto pv_issue = [&]() {
          const int g = up % NG, j = up / NG, b = j % NSB;
          tc::fence_after();
          const uint32_t vst = sV + (up % NST) * Cfg::KV_BYTES;
  #pragma unroll
          for (int k = 0; k < kTcKeys / 16; ++k) {
            const uint64_t bd = tc::sdesc(vst + k * 2 * 1024, Cfg::KV_BOX, 1024);
            if constexpr (Cfg::PTM) {
              // 16 keys of P: 8 columns of the group's S buffer, each
              // 64-key half of P at the start of that half's S columns
              tc::mma_ts(tO + g * D, tS + (NSB * g + b) * kTcKeys + 64 * (k / 4) + 8 * (k % 4),
                         bd, ID_O, (j > 0 || k > 0) ? 1u : 0u);
            } else {
              const uint64_t a = tc::sdesc(
                  sP + (NSB * g + b) * Cfg::P_BYTES + (k / 4) * Cfg::P_CB + (k % 4) * 32, 16,
                  1024);
              tc::mma(tO + g * D, a, bd, ID_O, (j > 0 || k > 0) ? 1u : 0u);
            }
          }
          tc::commit(&o_bar[g][b]);
          tc::commit(&empty_v[up % NST]);                 // the V stage is free once P.V is done
          ++up;
        };
        while (up < n_tiles && !failed) {
          // S products first: the softmax waits on them
          bool did = true;
          if (s_ready()) s_issue();
          else if (pv_ready()) pv_issue();
          else did = false;
          if (did) {
            idle = 0;
          } else if (++idle > (1u << 26)) {
            failed = true;                                // nothing became ready: give up
            atomicOr(p.err, PKV_DEVERR_TIMEOUT);
          }
        }
        if constexpr (Cfg::PTM) tc::commit(&done_bar);  // once every MMA above is complete
      }
      __syncwarp();
      if constexpr (SPLIT > 1) cluster_wait();
      return;
    }
  }
  if constexpr (Cfg::REALLOC) tc::reg_raise<Cfg::REG_SOFTMAX>();

  // ---- warps 0 .. 4 NG - 1: the softmax groups, one row per thread each ------------
  const uint32_t lane_base = (uint32_t)((warp & 3) * 32) << 16;
  // last key this row sees. A row no (token, head) pair of the chunk uses (G
  // not dividing the tile, or tokens past the chunk) sees the keys of the
  // tile's last token: its output is never stored, and rows do not mix in the
  // MMAs, so it only has to stay finite and cheap. (With no key at all it
  // took the masking pass on every tile, which held its warp and with it every
  // P.V back: 1.5 us a tile at G = 7 against 1.1 at G = 4.)
  const int lim = P0 + (rvalid ? qi : i1 - 1);
  const float sl2 = p.qk_scale_log2 * (KV8 ? p.k_scales[h] : 1.f) *
                   ((KV8 && QBF16) ? s_qpow[r] : 1.f);     // undoes the row's q scaling
  const uint32_t tOg = tO + grp * D;
  const int n_mine = (n_tiles - grp + NG - 1) / NG;     // this group's tiles
  float m_ref = -INFINITY, l = 0.f;

  for (int j = 0; j < n_mine; ++j) {
    const int u = NG * j + grp;                         // local tile
    const int t = t_begin + u;                          // key tile
    const int st = u % NST;
    const int b = j % NSB;
    wait(&s_bar[grp][b], (j / NSB) & 1);
    tc::fence_after();
    const uint32_t sbuf = tS + (NSB * grp + b) * kTcKeys + lane_base;
    // raw scores, 64 keys at a time; keys past this row's causal limit become
    // -inf (only the halves that cross the limit need the test). A 128-key
    // tile is read from TMEM twice, for the max and then for P, which keeps
    // 64 scores in registers
    constexpr int HALVES = kTcKeys / 64;
    float x[64];
    auto load_half = [&](int hh) {
      uint32_t sv[2][32];
      tc::ld32(sbuf + hh * 64, sv[0]);
      tc::ld32(sbuf + hh * 64 + 32, sv[1]);
      tc::wait_ld();
#pragma unroll
      for (int c = 0; c < 64; ++c) x[c] = __uint_as_float(sv[c / 32][c % 32]);
      const int k0 = t * kTcKeys + hh * 64;
      if (k0 + 63 > lim) {
#pragma unroll
        for (int c = 0; c < 64; ++c)
          if (k0 + c > lim) x[c] = -INFINITY;
      }
    };
    // row max over 8 independent chains, then a tree
    float m8[8];
#pragma unroll
    for (int k = 0; k < 8; ++k) m8[k] = -INFINITY;
#pragma unroll
    for (int hh = 0; hh < HALVES; ++hh) {
      load_half(hh);
#pragma unroll
      for (int c = 0; c < 64; ++c) m8[c % 8] = fmaxf(m8[c % 8], x[c]);
    }
#pragma unroll
    for (int w = 4; w > 0; w >>= 1)
#pragma unroll
      for (int k = 0; k < w; ++k) m8[k] = fmaxf(m8[k], m8[k + w]);
    const float mx = m8[0] * sl2;                       // the scale is positive: max commutes
    // move the reference max only when the row max outgrows it by 2^8
    const bool move = mx > m_ref + kRescaleLog2;
    const float alpha = move ? (m_ref == -INFINITY ? 0.f : ex2_approx(m_ref - mx)) : 1.f;
    if (move) m_ref = mx;
    if (j > 0 && __any_sync(0xffffffffu, move)) {
      // O must hold every earlier tile of this group before it is scaled
      wait(&o_bar[grp][(j - 1) % NSB], ((j - 1) / NSB) & 1);
      tc::fence_after();
#pragma unroll
      for (int c0 = 0; c0 < D; c0 += 32) {
        uint32_t ov[32];
        tc::ld32(tOg + lane_base + c0, ov);
        tc::wait_ld();
#pragma unroll
        for (int c = 0; c < 32; ++c) ov[c] = __float_as_uint(__uint_as_float(ov[c]) * alpha);
        tc::st32(tOg + lane_base + c0, ov);
      }
      tc::wait_st();
    }
    // P buffer b was read by the P.V of this group's tile j - NSB
    if (j >= NSB) wait(&o_bar[grp][b], ((j - NSB) / NSB) & 1);
    const float ms = m_ref == -INFINITY ? 0.f : m_ref;
    uint8_t* pPb = pP + (NSB * grp + b) * Cfg::P_BYTES;
    float rs8[8];
#pragma unroll
    for (int k = 0; k < 8; ++k) rs8[k] = 0.f;
#pragma unroll
    for (int it = 0; it < HALVES; ++it) {
      // PTM: the last half first, from the registers the max pass left it in,
      // then the others reloaded; P of keys 64 hh .. 64 hh + 63 goes to
      // columns 64 hh .. 64 hh + 31, the first half of that half's own scores
      // (already in x), so no score is overwritten before it is read
      const int hh = Cfg::PTM ? HALVES - 1 - it : it;
      if (HALVES > 1 && (!Cfg::PTM || it > 0)) load_half(hh);   // (else x holds it)
      uint32_t pv[32];
#pragma unroll
      for (int c = 0; c < 8; ++c) {
        float e[8];
#pragma unroll
        for (int k = 0; k < 8; ++k) {
          e[k] = ex2_approx(fmaf(x[8 * c + k], sl2, -ms));
          rs8[k] += e[k];
        }
        const uint4 w = make_uint4(pack16x2<BF16>(e[0], e[1]), pack16x2<BF16>(e[2], e[3]),
                                   pack16x2<BF16>(e[4], e[5]), pack16x2<BF16>(e[6], e[7]));
        if constexpr (Cfg::PTM) {
          pv[4 * c] = w.x;
          pv[4 * c + 1] = w.y;
          pv[4 * c + 2] = w.z;
          pv[4 * c + 3] = w.w;
        } else {
          *reinterpret_cast<uint4*>(pPb + hh * Cfg::P_CB + swz128(r, c)) = w;
        }
      }
      if constexpr (Cfg::PTM) tc::st32(sbuf + hh * 64, pv);
    }
    if constexpr (Cfg::PTM) tc::wait_st();
#pragma unroll
    for (int w = 4; w > 0; w >>= 1)
#pragma unroll
      for (int k = 0; k < w; ++k) rs8[k] += rs8[k + w];
    l = l * alpha + rs8[0];
    // V rows with no data for this tile (past the context, or pages not
    // loaded) meet weight 0 in P: zero them so their contents cannot make NaN.
    // The group's threads share the rows; the P.V waits for all of them.
    const int vz = loaded_end - t * kTcKeys;
    if (!KV8 && vz < kTcKeys) {                         // (KV8: zeroed by the conversion)
      // the V tile has its own barrier: zero its rows only once it has landed
      wait(&full_v[st], (u / NST) & 1);
      uint8_t* vtile = pV + st * Cfg::KV_BYTES;
      for (int i = r; i < (kTcKeys - vz) * Cfg::NBOX * 8; i += kTcRows) {
        const int row = vz + i / (Cfg::NBOX * 8), rest = i % (Cfg::NBOX * 8);
        const int bx = rest / 8, chk = rest % 8;
        *reinterpret_cast<uint4*>(vtile + bx * Cfg::KV_BOX + row * 128 + chk * 16) =
            make_uint4(0u, 0u, 0u, 0u);
      }
    }
    // P (shared memory) and the zeros, for the tensor cores; with P in tensor
    // memory only the zeros need it
    if (!Cfg::PTM || (!KV8 && vz < kTcKeys)) fence_proxy_async_smem();
    tc::fence_before();
    mbar_arrive(&p_bar[grp][b]);
  }

  // ---- epilogue ------------------------------------------------------------------------
  if (n_mine > 0) {
    // MMAs complete in issue order: this group's last P.V done means all of its are
    const int jl = n_mine - 1;
    wait(&o_bar[grp][jl % NSB], (jl / NSB) & 1);
    tc::fence_after();
  }
  // The groups' shares of row r: O_g relative to 2^m_g with sum l_g.
  // Combined: M = max(m_0, m_1), O = O_0 w_0 + O_1 w_1 with w_g = 2^(m_g - M),
  // and the same for the sum. (reference max, sum) of each row go through the
  // group's first P buffer, which its last P.V has finished reading.
  // (PTM: through the query tile's space, once every MMA, the S products
  // that read it included, is complete)
  if constexpr (Cfg::PTM) {
    wait(&done_bar, 0);
    tc::fence_after();
  }
  float2* ml_g0 = Cfg::PTM ? reinterpret_cast<float2*>(pQ) : reinterpret_cast<float2*>(pP);
  float2* ml_g1 = Cfg::PTM ? reinterpret_cast<float2*>(pQ) + kTcRows
                           : reinterpret_cast<float2*>(pP + NSB * Cfg::P_BYTES);
  (grp == 0 ? ml_g0 : ml_g1)[r] = make_float2(m_ref, l);
  named_barrier(1, NG * kTcRows);
  const float2 ml0 = ml_g0[r];
  const float2 ml1 = NG > 1 ? ml_g1[r] : make_float2(-INFINITY, 0.f);
  // a group with no tile has no O
  const bool has0 = n_tiles > 0, has1 = NG > 1 && n_tiles > 1;
  const float M = fmaxf(ml0.x, ml1.x);
  const float w0 = has0 && ml0.x != -INFINITY ? ex2_approx(ml0.x - M) : 0.f;
  const float w1 = has1 && ml1.x != -INFINITY ? ex2_approx(ml1.x - M) : 0.f;
  const float Lc = ml0.y * w0 + ml1.y * w1;

  // CTA `split` of the cluster finishes columns [split CW, (split + 1) CW),
  // group g of it the part [g QW, (g + 1) QW) of those.
  constexpr int CW = D / SPLIT;
  constexpr int QW = CW / NG;
  constexpr int CH = QW < 32 ? QW : 32;                 // TMEM columns per load
  const int mycol = split * CW + grp * QW;
  // combined O of this CTA for columns [c, c + CH)
  auto combined = [&](int c, float (&f)[CH]) {
    uint32_t o0[CH], o1[CH];
    tmem_ld<CH>(tO + lane_base + c, o0);
    if constexpr (NG > 1) tmem_ld<CH>(tO + D + lane_base + c, o1);
    tc::wait_ld();
#pragma unroll
    for (int k = 0; k < CH; ++k) {
      f[k] = w0 != 0.f ? __uint_as_float(o0[k]) * w0 : 0.f;
      if constexpr (NG > 1) f[k] += w1 != 0.f ? __uint_as_float(o1[k]) * w1 : 0.f;
    }
  };

  // SPLIT == 2: each CTA hands the other the combined O of the other's
  // columns, with its M and sum, into the other's K ring (drained once that
  // CTA's last P.V, and so its last S, is done):
  //   O as [CW / 4][128 rows] float4 (a warp's rows side by side, no bank
  //   conflicts), then (M, sum) as [128 rows] float2.
  float M_o = -INFINITY, L_o = 0.f;
  const uint32_t recv_rows = sKV;
  const uint32_t recv_ml = sKV + kTcRows * CW * 4;
  if constexpr (SPLIT > 1) {
    const uint32_t other = (uint32_t)(split ^ 1);
    cluster_wait();                                     // the other CTA's barriers are set up
    if (tid == 0) mbar_arrive_remote(cluster_map(smem_u32(&ready_bar), other));
    if (!mbar_wait_cluster(&ready_bar, 0)) atomicOr(p.err, PKV_DEVERR_TIMEOUT);
    const uint32_t dst = cluster_map(recv_rows, other) + r * 16;
#pragma unroll
    for (int c0 = 0; c0 < QW; c0 += CH) {
      float f[CH];
      combined((int)other * CW + grp * QW + c0, f);
#pragma unroll
      for (int c = 0; c < CH; c += 4)
        st_cluster_v4(dst + ((grp * QW + c0 + c) / 4) * (kTcRows * 16), f[c], f[c + 1],
                      f[c + 2], f[c + 3]);
    }
    if (grp == 0) st_cluster_v2(cluster_map(recv_ml, other) + r * 8, M, Lc);
    mbar_arrive_remote(cluster_map(smem_u32(&recv_bar), other));
    if (!mbar_wait_cluster(&recv_bar, 0)) atomicOr(p.err, PKV_DEVERR_TIMEOUT);
    const float2 ml = *reinterpret_cast<const float2*>(basep + (recv_ml - base) + r * 8);
    M_o = ml.x;
    L_o = ml.y;
  }
  // with the other CTA's share: M2 = max(M, M_o), O = O 2^(M - M2) + O_o 2^(M_o - M2)
  const float M2 = fmaxf(M, M_o);
  const float a0 = M == -INFINITY ? 0.f : SPLIT == 1 ? 1.f : ex2_approx(M - M2);
  const float a1 = M_o == -INFINITY ? 0.f : ex2_approx(M_o - M2);
  const float L2 = Lc * a0 + L_o * a1;
  const float inv = L2 > 0.f ? (KV8 ? p.v_scales[h] : 1.f) / L2 : 0.f;
  const float4* orecv = reinterpret_cast<const float4*>(basep + (recv_rows - base)) + r;
  uint16_t* orow = static_cast<uint16_t*>(p.out) + ((int64_t)(q0 + (rvalid ? qi : 0)) * p.Hq +
                                                    (rvalid ? hq : 0)) * D;
#pragma unroll
  for (int c0 = 0; c0 < QW; c0 += CH) {
    float f[CH];
    combined(mycol + c0, f);
    if (rvalid) {
#pragma unroll
      for (int c = 0; c < CH; c += 4) {
        float4 of = make_float4(0.f, 0.f, 0.f, 0.f);
        if constexpr (SPLIT > 1) of = orecv[((grp * QW + c0 + c) / 4) * kTcRows];
        f[c] = (f[c] * a0 + of.x * a1) * inv;
        f[c + 1] = (f[c + 1] * a0 + of.y * a1) * inv;
        f[c + 2] = (f[c + 2] * a0 + of.z * a1) * inv;
        f[c + 3] = (f[c + 3] * a0 + of.w * a1) * inv;
      }
#pragma unroll
      for (int c = 0; c < CH / 8; ++c) {
        const uint4 w = make_uint4(
            pack16x2<QBF16>(f[8 * c + 0], f[8 * c + 1]), pack16x2<QBF16>(f[8 * c + 2], f[8 * c + 3]),
            pack16x2<QBF16>(f[8 * c + 4], f[8 * c + 5]), pack16x2<QBF16>(f[8 * c + 6], f[8 * c + 7]));
        *reinterpret_cast<uint4*>(orow + mycol + c0 + 8 * c) = w;
      }
    }
  }
  if (split == 0 && grp == 0 && rvalid && p.out_lse != nullptr)
    p.out_lse[(int64_t)(q0 + qi) * p.Hq + hq] = L2 > 0.f ? (M2 + log2f(L2)) * kLn2 : -INFINITY;
  tc::fence_before();
  named_barrier(1, NG * kTcRows);
  if (warp == 0) tc::dealloc(tm, Cfg::TMEM_COLS);
}

template <int D, int KV, bool QBF16, int SPLIT, bool ALONE>
static pkv_status launch_prefill_tc_s(const PrefillParams& q, const CUtensorMap& tmQ,
                                      const CUtensorMap& tmK, const CUtensorMap& tmV,
                                      cudaStream_t stream, int dev) {
  constexpr bool KV8 = KV == KV_E4M3;
  // ring stages: the 128-key tiles (P in tensor memory) take 3 of 32 KB at
  // D = 128 and 6 of 16 KB at D = 64; E4M3 and D = 256 take 2, the rest 4
  constexpr bool WIDE = PrefillTcCfg<D, 2, KV8, ALONE>::WIDE;
  constexpr int NST = WIDE ? (D == 128 ? 3 : 6) : ((D > 128 || KV8) ? 2 : 4);
  using Cfg = PrefillTcCfg<D, NST, KV8, ALONE>;
  static_assert(Cfg::SMEM_BYTES + 512 <= 227 * 1024, "shared memory (dynamic + static)");
  static_assert(SPLIT == 1 || kTcRows * (D / SPLIT) * 4 + kTcRows * 8 <= 2 * Cfg::RING_BYTES,
                "the other CTA's rows must fit in the ring");
  auto kern = prefill_tc_kernel<D, KV, QBF16, NST, SPLIT, ALONE>;
  static std::atomic<bool> attr_set[64];  // per device; the call is idempotent
  if (!attr_set[dev]) {
    if (cudaFuncSetAttribute(kern, cudaFuncAttributeMaxDynamicSharedMemorySize,
                             Cfg::SMEM_BYTES) != cudaSuccess)
      return PKV_ERR_CUDA;
    if constexpr (Cfg::REALLOC) {
      // a register raise waits for registers the CTA does not have unless
      // the launch allocation covers every warpgroup's count: never launch then
      cudaFuncAttributes fa{};
      if (cudaFuncGetAttributes(&fa, kern) != cudaSuccess) return PKV_ERR_CUDA;
      if ((int64_t)fa.numRegs * Cfg::THREADS < Cfg::REG_TOTAL) return PKV_ERR_UNSUPPORTED;
    }
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
  cfg.blockDim = dim3(Cfg::THREADS);
  cfg.dynamicSmemBytes = Cfg::SMEM_BYTES;
  cfg.stream = stream;
  cfg.attrs = attr;
  cfg.numAttrs = 1;
  return cudaLaunchKernelEx(&cfg, kern, tmQ, tmK, tmV, q) == cudaSuccess ? PKV_OK : PKV_ERR_CUDA;
}

// One CTA per query tile when that fills at least half of the GPU (or other
// work shares it); otherwise a cluster of two per tile, each taking half of
// the key tiles. Beside a decode grid (may_split false), the 64-key tiles.
template <int D, int KV, bool QBF16>
static pkv_status launch_prefill_tc_t(const PrefillParams& p, const CUtensorMap& tmQ,
                                      const CUtensorMap& tmK, const CUtensorMap& tmV,
                                      cudaStream_t stream,
                                      bool may_split) {
  int dev = 0;
  if (cudaGetDevice(&dev) != cudaSuccess || dev < 0 || dev >= 64) return PKV_ERR_CUDA;
  static std::atomic<int> sms[64];                      // per device SM count, read once
  int n_sms = sms[dev].load();
  if (n_sms == 0) {
    if (cudaDeviceGetAttribute(&n_sms, cudaDevAttrMultiProcessorCount, dev) != cudaSuccess)
      return PKV_ERR_CUDA;
    sms[dev].store(n_sms);
  }
  PrefillParams q = p;
  q.q_tile = kTcRows / p.G;
  const int64_t ctas = (int64_t)((q.max_q_len + q.q_tile - 1) / q.q_tile) * q.Hkv * q.num_seqs;
  if (!may_split) return launch_prefill_tc_s<D, KV, QBF16, 1, false>(q, tmQ, tmK, tmV, stream, dev);
  if (2 * ctas <= n_sms)
    return launch_prefill_tc_s<D, KV, QBF16, 2, true>(q, tmQ, tmK, tmV, stream, dev);
  return launch_prefill_tc_s<D, KV, QBF16, 1, true>(q, tmQ, tmK, tmV, stream, dev);
}

template <int D>
static pkv_status launch_prefill_tc_d(const PrefillParams& p, pkv_dtype q_dtype,
                                      pkv_dtype kv_dtype, const CUtensorMap& tmQ,
                                      const CUtensorMap& tmK, const CUtensorMap& tmV,
                                      cudaStream_t stream,
                                      bool may_split) {
  if (kv_dtype == PKV_BF16)
    return launch_prefill_tc_t<D, KV_BF16, true>(p, tmQ, tmK, tmV, stream, may_split);
  if (kv_dtype == PKV_F16)
    return launch_prefill_tc_t<D, KV_F16, false>(p, tmQ, tmK, tmV, stream, may_split);
  if constexpr (D <= 128) {
    return q_dtype == PKV_BF16
               ? launch_prefill_tc_t<D, KV_E4M3, true>(p, tmQ, tmK, tmV, stream, may_split)
               : launch_prefill_tc_t<D, KV_E4M3, false>(p, tmQ, tmK, tmV, stream, may_split);
  }
  return PKV_ERR_UNSUPPORTED;
}

bool prefill_tc_supported(int head_dim, pkv_dtype kv_dtype) {
  if (kv_dtype == PKV_FP8_E4M3) return head_dim == 64 || head_dim == 128;
  return head_dim == 64 || head_dim == 128 || head_dim == 256;
}

pkv_status launch_prefill_tc(const PrefillParams& p, int head_dim, pkv_dtype q_dtype,
                             pkv_dtype kv_dtype, const CUtensorMap& tmQ, const CUtensorMap& tmK,
                             const CUtensorMap& tmV, cudaStream_t stream, bool may_split) {
  if (head_dim == 256)
    return launch_prefill_tc_d<256>(p, q_dtype, kv_dtype, tmQ, tmK, tmV, stream, may_split);
  if (head_dim == 128)
    return launch_prefill_tc_d<128>(p, q_dtype, kv_dtype, tmQ, tmK, tmV, stream, may_split);
  return launch_prefill_tc_d<64>(p, q_dtype, kv_dtype, tmQ, tmK, tmV, stream, may_split);
}

}  // namespace pkv
