// prefill.cu — causal attention of a prefill chunk over the paged cache.
//
// Follows "Chunked Prefill ... long prompts split into 512-token chunks"
// (Litellama, Features) and the paged attention it runs over (Welcome to
// vLLM, feature list: PagedAttention, chunked prefill). Query row i of a
// chunk of length L on P cached tokens sits at absolute position P + i and
// attends keys 0 .. P + i.
//
// Work decomposition: one CTA per (query tile, KV head, sequence). The
// tile's 64 MMA rows are (query token, query head of the GQA group) pairs,
// so the K/V of a KV head is shared by every head of its group. A producer
// warp streams KT pages of K and V per stage through TMA into an NST-deep
// ring (full barriers count TMA bytes, empty barriers count the four
// consumer warps); each consumer warp owns 16 rows and runs an online
// softmax over 16*KT-key tiles with m16n8k16 tensor-core products.
#include <cuda.h>
#include "common.cuh"
#include "launch_prefill.h"

namespace pkv {

constexpr int kPrefillConsumers = 4;
constexpr int kPrefillRows = 16 * kPrefillConsumers;

int prefill_q_tile(int G) { return kPrefillRows / G; }

template <int D, int KV, int NST, int KT>
struct PrefillCfg {
  using Geo = PageGeom<D, KV>;
  static constexpr int STAGE_BYTES = 2 * KT * Geo::PAGE_BYTES;
  static constexpr int SMEM_BYTES = NST * STAGE_BYTES + 1024;
};

template <int D, int KV, bool QBF16, int NST, int KT>
__global__ void __launch_bounds__((kPrefillConsumers + 1) * 32)
    prefill_chunk_kernel(const __grid_constant__ CUtensorMap tmK,
                         const __grid_constant__ CUtensorMap tmV, const PrefillParams p) {
  using Geo = PageGeom<D, KV>;
  using Cfg = PrefillCfg<D, KV, NST, KT>;
  constexpr int STAGE = Cfg::STAGE_BYTES;
  constexpr int TILE = kBS * KT;
  extern __shared__ uint8_t smem_raw[];
  __shared__ uint64_t full_bar[NST];
  __shared__ uint64_t empty_bar[NST];

  // a decode launched behind this kernel as a programmatic dependent may take
  // the SM room this grid leaves as soon as all of its CTAs are running
  if (threadIdx.x == 0) griddep_launch_dependents();
  const int lane = threadIdx.x & 31, warp = threadIdx.x >> 5;
  const int qt = blockIdx.x, h = blockIdx.y, n = blockIdx.z;
  const int G = p.G;
  const int q0 = p.cu_q_lens[n];
  const int L = p.cu_q_lens[n + 1] - q0;
  const int ctx = p.seq_lens[n];
  // a chunk longer than its context, or whose rows are not rows of q and out
  if (L < 0 || L > ctx || q0 < 0 || q0 > p.q_rows - L ||
      ctx > ((p.max_blocks * kBS) << p.ppb_shift)) {
    if (threadIdx.x == 0 && qt == 0 && h == 0) atomicOr(p.err, PKV_DEVERR_QLEN);
    return;
  }
  const int P = ctx - L;
  const int i0 = qt * p.q_tile;
  if (i0 >= L) return;
  const int i1 = min(L, i0 + p.q_tile);
  const int key_end = P + i1;                          // exclusive
  const int n_pages = (key_end + kBS - 1) / kBS;
  const int n_tiles = (key_end + TILE - 1) / TILE;

  const uint32_t raw_base = smem_u32(smem_raw);
  const uint32_t base = (raw_base + 1023u) & ~1023u;
  uint8_t* basep = smem_raw + (base - raw_base);

  if (threadIdx.x == 0) {
    prefetch_tensormap(&tmK);
    prefetch_tensormap(&tmV);
    for (int s = 0; s < NST; ++s) {
      mbar_init(&full_bar[s], 1);
      mbar_init(&empty_bar[s], kPrefillConsumers);
    }
    fence_barrier_init();
  }
  __syncthreads();

  if (warp == kPrefillConsumers) {
    // ---- producer warp: its lanes look up the page rows 32 pages at a time,
    // one chunk ahead, so no block-table read waits in front of a TMA issue;
    // lane 0 issues the loads ---------------------------------------------------------
    static_assert(32 % KT == 0, "a tile's pages lie in one chunk");
    auto page_row = [&](int lp) -> int {
      if (lp >= n_pages) return 0;
      int id = p.block_tables[(int64_t)n * p.max_blocks + (lp >> p.ppb_shift)];
      if (id < 0 || id >= p.num_blocks) {
        atomicOr(p.err, PKV_DEVERR_BLOCK_ID);
        id = 0;
      }
      return ((id * p.Hkv + h) << p.ppb_shift) + (lp & ((1 << p.ppb_shift) - 1));
    };
    int z_cur = page_row(lane), z_next = page_row(32 + lane), chunk = 0;
    for (int t = 0; t < n_tiles; ++t) {
      const int st = t % NST;
      bool ok = t < NST || mbar_wait_bounded(&empty_bar[st], ((t / NST) - 1) & 1);
      ok = __all_sync(0xffffffffu, ok);
      if (!ok) {
        if (lane == 0) atomicOr(p.err, PKV_DEVERR_TIMEOUT);
        break;
      }
      if ((t * KT) / 32 != chunk) {
        z_cur = z_next;
        ++chunk;
        z_next = page_row(32 * (chunk + 1) + lane);
      }
      const int pg0 = t * KT;
      const int npg = min(KT, n_pages - pg0);
      if (lane == 0) mbar_arrive_expect_tx(&full_bar[st], npg * 2 * Geo::PAGE_BYTES);
      uint8_t* dst = basep + st * STAGE;
      for (int pg = 0; pg < npg; ++pg) {
        const int z = __shfl_sync(0xffffffffu, z_cur, (pg0 + pg) % 32);
        if (lane == 0) {
#pragma unroll
          for (int bx = 0; bx < Geo::NBOX; ++bx) {
            tma_load_3d(dst + pg * Geo::PAGE_BYTES + bx * Geo::BOX_BYTES, &tmK, &full_bar[st],
                        bx * Geo::BOX_ELEMS, 0, z);
            tma_load_3d(dst + (KT + pg) * Geo::PAGE_BYTES + bx * Geo::BOX_BYTES, &tmV,
                        &full_bar[st], bx * Geo::BOX_ELEMS, 0, z);
          }
        }
      }
    }
    return;
  }

  // ---- consumer warps: 16 rows each ---------------------------------------------
  const int g = lane >> 2, c = lane & 3;
  const int rows_used = p.q_tile * G;
  const int r0 = warp * 16 + g, r8 = r0 + 8;
  const bool v0 = r0 < rows_used && i0 + r0 / G < i1;
  const bool v8 = r8 < rows_used && i0 + r8 / G < i1;
  const int qi0 = i0 + r0 / G, qi8 = i0 + r8 / G;     // query index within the chunk
  const int hq0 = h * G + r0 % G, hq8 = h * G + r8 % G;
  const uint16_t* qbase = static_cast<const uint16_t*>(p.q);
  const void* rowg = v0 ? qbase + ((int64_t)(q0 + qi0) * p.Hq + hq0) * D : nullptr;
  const void* rowg8 = v8 ? qbase + ((int64_t)(q0 + qi8) * p.Hq + hq8) * D : nullptr;
  uint32_t qf[D / 16][4];
  int qsh0, qsh8;
  load_q_frags<D, KV, QBF16>(qf, rowg, rowg8, lane, qsh0, qsh8);
  // last key each row may see (-1: none)
  const int lim0 = v0 ? P + qi0 : -1;
  const int lim8 = v8 ? P + qi8 : -1;
  const int warp_lim = __reduce_max_sync(0xffffffffu, max(lim0, lim8));

  float oacc[D / 8][4];
#pragma unroll
  for (int t = 0; t < D / 8; ++t) oacc[t][0] = oacc[t][1] = oacc[t][2] = oacc[t][3] = 0.f;
  float m0 = -INFINITY, m8 = -INFINITY, l0 = 0.f, l8 = 0.f;
  // rows g and g + 8 of q were scaled by 2^-qsh for the f16 MMAs: scale their
  // scores back (exact)
  const float sl2 = p.qk_scale_log2 * (KV == KV_E4M3 ? p.k_scales[h] : 1.f);
  const float sl2_0 = sl2 * pow2f(qsh0), sl2_8 = sl2 * pow2f(qsh8);

  for (int t = 0; t < n_tiles; ++t) {
    const int st = t % NST;
    bool ok = mbar_wait_bounded(&full_bar[st], (t / NST) & 1);
    ok = __all_sync(0xffffffffu, ok);
    if (!ok) {
      if (lane == 0) atomicOr(p.err, PKV_DEVERR_TIMEOUT);
      break;
    }
    const int kbase = t * TILE;
    if (kbase <= warp_lim) {
      const uint32_t kst = base + st * STAGE;
      const uint32_t vst = kst + KT * Geo::PAGE_BYTES;
      const int npg = min(KT, n_pages - t * KT);
      float s[2 * KT][4];
#pragma unroll
      for (int j = 0; j < 2 * KT; ++j) s[j][0] = s[j][1] = s[j][2] = s[j][3] = 0.f;
#pragma unroll
      for (int pg = 0; pg < KT; ++pg) {
        if (pg < npg && kbase + pg * kBS <= warp_lim) {
          qk_page<D, KV>(s, 2 * pg, qf, kst + pg * Geo::PAGE_BYTES, lane);
        }
      }
      float mx0 = -INFINITY, mx8 = -INFINITY;
#pragma unroll
      for (int pg = 0; pg < KT; ++pg)
#pragma unroll
        for (int jj = 0; jj < 2; ++jj)
#pragma unroll
          for (int e = 0; e < 2; ++e) {
            const int j = 2 * pg + jj;
            const int key = kbase + pg * kBS + s_col_token<KV>(jj, c, e);
            s[j][e] = key <= lim0 ? s[j][e] * sl2_0 : -INFINITY;
            s[j][2 + e] = key <= lim8 ? s[j][2 + e] * sl2_8 : -INFINITY;
            mx0 = fmaxf(mx0, s[j][e]);
            mx8 = fmaxf(mx8, s[j][2 + e]);
          }
      mx0 = quad_max(mx0);
      mx8 = quad_max(mx8);
      const float mn0 = fmaxf(m0, mx0), mn8 = fmaxf(m8, mx8);
      const float ms0 = mn0 == -INFINITY ? 0.f : mn0;
      const float ms8 = mn8 == -INFINITY ? 0.f : mn8;
      const float a0 = exp2f(m0 - ms0), a8 = exp2f(m8 - ms8);
      m0 = mn0;
      m8 = mn8;
      float rs0 = 0.f, rs8 = 0.f;
#pragma unroll
      for (int j = 0; j < 2 * KT; ++j)
#pragma unroll
        for (int e = 0; e < 2; ++e) {
          s[j][e] = exp2f(s[j][e] - ms0);
          s[j][2 + e] = exp2f(s[j][2 + e] - ms8);
          rs0 += s[j][e];
          rs8 += s[j][2 + e];
        }
      l0 = l0 * a0 + rs0;
      l8 = l8 * a8 + rs8;
#pragma unroll
      for (int tt = 0; tt < D / 8; ++tt) {
        oacc[tt][0] *= a0;
        oacc[tt][1] *= a0;
        oacc[tt][2] *= a8;
        oacc[tt][3] *= a8;
      }
#pragma unroll
      for (int pg = 0; pg < KT; ++pg) {
        if (pg < npg && kbase + pg * kBS <= warp_lim) {
          uint32_t pa[4];
          pack_p<KV>(pa, s, 2 * pg);
          pv_page<D, KV>(oacc, pa, vst + pg * Geo::PAGE_BYTES, lane,
                         min(kBS, ctx - (kbase + pg * kBS)));
        }
      }
    }
    __syncwarp();
    if (lane == 0) mbar_arrive(&empty_bar[st]);
  }

  const float L0 = quad_sum(l0), L8 = quad_sum(l8);
  const float vscale = (KV == KV_E4M3) ? p.v_scales[h] : 1.f;
  const float inv0 = L0 > 0.f ? vscale / L0 : 0.f;
  const float inv8 = L8 > 0.f ? vscale / L8 : 0.f;
  uint16_t* out = static_cast<uint16_t*>(p.out);
#pragma unroll
  for (int tt = 0; tt < D / 8; ++tt)
#pragma unroll
    for (int e = 0; e < 2; ++e) {
      const int d = o_col_dim<D, KV>(tt, c, e);
      if (v0) {
        float v = oacc[tt][e] * inv0;
        __half hv = __float2half_rn(v);
        __nv_bfloat16 bv = __float2bfloat16_rn(v);
        out[((int64_t)(q0 + qi0) * p.Hq + hq0) * D + d] =
            QBF16 ? *reinterpret_cast<uint16_t*>(&bv) : *reinterpret_cast<uint16_t*>(&hv);
      }
      if (v8) {
        float v = oacc[tt][2 + e] * inv8;
        __half hv = __float2half_rn(v);
        __nv_bfloat16 bv = __float2bfloat16_rn(v);
        out[((int64_t)(q0 + qi8) * p.Hq + hq8) * D + d] =
            QBF16 ? *reinterpret_cast<uint16_t*>(&bv) : *reinterpret_cast<uint16_t*>(&hv);
      }
    }
  if (c == 0 && p.out_lse != nullptr) {
    if (v0) p.out_lse[(int64_t)(q0 + qi0) * p.Hq + hq0] = L0 > 0.f ? (m0 + log2f(L0)) * kLn2 : -INFINITY;
    if (v8) p.out_lse[(int64_t)(q0 + qi8) * p.Hq + hq8] = L8 > 0.f ? (m8 + log2f(L8)) * kLn2 : -INFINITY;
  }
}

template <int D, int KV, bool QBF16>
static pkv_status launch_prefill_t(const PrefillParams& p, const CUtensorMap& tmK,
                                   const CUtensorMap& tmV, cudaStream_t stream) {
  // D = 256: two pages per tile and two stages keep registers and shared memory in bounds
  constexpr int NST = D > 128 ? 2 : 3;
  constexpr int KT = D > 128 ? 2 : 4;
  using Cfg = PrefillCfg<D, KV, NST, KT>;
  auto kern = prefill_chunk_kernel<D, KV, QBF16, NST, KT>;
  int dev = 0;
  if (cudaGetDevice(&dev) != cudaSuccess || dev < 0 || dev >= 64) return PKV_ERR_CUDA;
  static std::atomic<bool> attr_set[64];  // per device; the call is idempotent
  if (!attr_set[dev]) {
    if (cudaFuncSetAttribute(kern, cudaFuncAttributeMaxDynamicSharedMemorySize,
                             Cfg::SMEM_BYTES) != cudaSuccess)
      return PKV_ERR_CUDA;
    attr_set[dev] = true;
  }
  dim3 grid((p.max_q_len + p.q_tile - 1) / p.q_tile, p.Hkv, p.num_seqs);
  kern<<<grid, (kPrefillConsumers + 1) * 32, Cfg::SMEM_BYTES, stream>>>(tmK, tmV, p);
  return cudaGetLastError() == cudaSuccess ? PKV_OK : PKV_ERR_CUDA;
}

template <int D>
static pkv_status launch_prefill_d(const PrefillParams& p, pkv_dtype q_dtype, pkv_dtype kv_dtype,
                                   const CUtensorMap& tmK, const CUtensorMap& tmV,
                                   cudaStream_t stream) {
  const bool qbf = (q_dtype == PKV_BF16);
  if (kv_dtype == PKV_FP8_E4M3)
    return qbf ? launch_prefill_t<D, KV_E4M3, true>(p, tmK, tmV, stream)
               : launch_prefill_t<D, KV_E4M3, false>(p, tmK, tmV, stream);
  if (kv_dtype == PKV_BF16) return launch_prefill_t<D, KV_BF16, true>(p, tmK, tmV, stream);
  return launch_prefill_t<D, KV_F16, false>(p, tmK, tmV, stream);
}

pkv_status launch_prefill(const PrefillParams& p, int head_dim, pkv_dtype q_dtype,
                          pkv_dtype kv_dtype, const CUtensorMap& tmK, const CUtensorMap& tmV,
                          cudaStream_t stream) {
  if (head_dim == 256) return launch_prefill_d<256>(p, q_dtype, kv_dtype, tmK, tmV, stream);
  if (head_dim == 128) return launch_prefill_d<128>(p, q_dtype, kv_dtype, tmK, tmV, stream);
  return launch_prefill_d<64>(p, q_dtype, kv_dtype, tmK, tmV, stream);
}

}  // namespace pkv
