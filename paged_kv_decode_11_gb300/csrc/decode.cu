// decode.cu — paged-KV decode attention with split-KV partitions and a
// log-sum-exp merge.
//
// Follows "flash attention decode (online softmax, paged KV, GQA)" and
// "Split-KV paged attention for long context" (rvLLM: High-performance LLM
// inference in Rust, Kernel Compiler Stack; Tier 2: Hand-written CUDA
// kernels; FA3 v3 Attention Kernel, "split-KV ... distributes KV tiles across
// thread blocks") and the log-sum-exp merge of partial attention (rapid_llm
// README, feature table, "Decode context parallelism").
//
// Work decomposition: one CTA per (partition, KV head, sequence). A
// partition is `part` consecutive tokens of one sequence's context. The CTA's
// NW warps take the partition's pages round-robin; each warp runs its own
// NST-deep ring of TMA loads (one K page + one V page per stage, completion on
// an mbarrier), so no warp ever waits for another until the end. All G query
// heads that share the KV head ride in the 16 MMA rows, so every K/V byte is
// read from HBM once per call. Each warp keeps an online softmax (running
// max m, running sum l, fp32 O accumulator) in the log2 domain; at the end the
// CTA merges its warps through shared memory and either writes the final
// output (single-partition sequences) or the normalised partition output and
// its log2-sum-exp to the workspace, which decode_merge_kernel combines.
#include <cuda.h>
#include <cfloat>
#include "common.cuh"
#include "launch.h"

namespace pkv {

template <int D, int KV, bool QBF16, int MROWS, int NW, int NST>
struct DecodeCfg {
  using Geo = PageGeom<D, KV>;
  static constexpr int STAGE_BYTES = 2 * Geo::PAGE_BYTES;
  static constexpr int PIPE_BYTES = NW * NST * STAGE_BYTES;
  static constexpr int OBUF_BYTES = NW * MROWS * D * 4;
  static constexpr int SMEM_BYTES = (PIPE_BYTES > OBUF_BYTES ? PIPE_BYTES : OBUF_BYTES) + 1024;
};

template <int D, int KV, bool QBF16, int MROWS, int NW, int NST>
__global__ void __launch_bounds__(NW * 32)
    decode_split_kernel(const __grid_constant__ CUtensorMap tmK,
                        const __grid_constant__ CUtensorMap tmV, const DecodeParams p) {
  using Geo = PageGeom<D, KV>;
  using Cfg = DecodeCfg<D, KV, QBF16, MROWS, NW, NST>;
  constexpr int STAGE = Cfg::STAGE_BYTES;
  constexpr int MAXP = kMaxPartitionTokens / kBS;
  extern __shared__ uint8_t smem_raw[];
  __shared__ uint64_t bars[NW][NST];
  __shared__ float red_m[NW][MROWS];
  __shared__ float red_l[NW][MROWS];
  __shared__ int s_ids[MAXP];

  const int lane = threadIdx.x & 31, warp = threadIdx.x >> 5;
  const int part_idx = blockIdx.x, h = blockIdx.y, b = blockIdx.z;
  const int G = p.G;

  int ctx = p.seq_lens[b];
  const int cap = min(p.max_seq_len, p.max_blocks * kBS);
  if (ctx < 0 || ctx > cap) {
    if (threadIdx.x == 0 && part_idx == 0 && h == 0) atomicOr(p.err, PKV_DEVERR_SEQ_LEN);
    ctx = ctx < 0 ? 0 : cap;
  }
  const int nparts = ctx > 0 ? (ctx + p.part - 1) / p.part : 1;
  if (part_idx >= nparts) return;
  const int tok0 = part_idx * p.part;
  const int tok1 = min(ctx, tok0 + p.part);
  const int npages = (tok1 - tok0 + kBS - 1) / kBS;
  const int page0 = tok0 / kBS;

  const uint32_t raw_base = smem_u32(smem_raw);
  const uint32_t base = (raw_base + 1023u) & ~1023u;
  uint8_t* basep = smem_raw + (base - raw_base);

  for (int i = threadIdx.x; i < npages; i += NW * 32) {
    int id = p.block_tables[(int64_t)b * p.max_blocks + page0 + i];
    if (id < 0 || id >= p.num_blocks) {
      atomicOr(p.err, PKV_DEVERR_BLOCK_ID);
      id = 0;
    }
    s_ids[i] = id;
  }
  if (threadIdx.x == 0) {
    prefetch_tensormap(&tmK);
    prefetch_tensormap(&tmV);
#pragma unroll
    for (int w = 0; w < NW; ++w)
#pragma unroll
      for (int s = 0; s < NST; ++s) mbar_init(&bars[w][s], 1);
    fence_barrier_init();
  }
  __syncthreads();

  // ---- per-warp TMA ring --------------------------------------------------
  const uint32_t wbase = base + warp * NST * STAGE;
  uint8_t* wbasep = basep + warp * NST * STAGE;
  const int nmine = warp < npages ? (npages - warp + NW - 1) / NW : 0;
  const int zh = h;
  auto issue = [&](int k) {
    const int st = k % NST;
    uint64_t* bar = &bars[warp][st];
    const int z = s_ids[warp + NW * k] * p.Hkv + zh;
    uint8_t* dst = wbasep + st * STAGE;
    mbar_arrive_expect_tx(bar, STAGE);
#pragma unroll
    for (int bx = 0; bx < Geo::NBOX; ++bx) {
      tma_load_3d(dst + bx * Geo::BOX_BYTES, &tmK, bar, bx * Geo::BOX_ELEMS, 0, z);
      tma_load_3d(dst + Geo::PAGE_BYTES + bx * Geo::BOX_BYTES, &tmV, bar, bx * Geo::BOX_ELEMS, 0,
                  z);
    }
  };
  int issued = 0;
  if (lane == 0) {
    for (int k = 0; k < NST && k < nmine; ++k) issue(k);
  }
  issued = min(NST, nmine);

  // ---- Q fragments: rows g and g + 8 of the GQA group --------------------------
  const int g = lane >> 2, c = lane & 3;
  const uint16_t* qb = static_cast<const uint16_t*>(p.q) + ((int64_t)b * p.Hq + h * G) * D;
  const void* rowg = g < G ? qb + g * D : nullptr;
  const void* rowg8 = (MROWS == 16 && g + 8 < G) ? qb + (g + 8) * D : nullptr;
  uint32_t qf[D / 16][4];
  load_q_frags<D, KV, QBF16>(qf, rowg, rowg8, lane);

  float oacc[D / 8][4];
#pragma unroll
  for (int t = 0; t < D / 8; ++t) oacc[t][0] = oacc[t][1] = oacc[t][2] = oacc[t][3] = 0.f;
  float m0 = -INFINITY, m8 = -INFINITY, l0 = 0.f, l8 = 0.f;
  const float sl2 = p.qk_scale_log2 * (KV == KV_E4M3 ? p.k_scales[h] : 1.f);
  bool aborted = false;

  for (int k = 0; k < nmine; ++k) {
    const int st = k % NST;
    bool ok = mbar_wait_bounded(&bars[warp][st], (k / NST) & 1);
    ok = __all_sync(0xffffffffu, ok);
    if (!ok) {
      aborted = true;
      if (lane == 0) atomicOr(p.err, PKV_DEVERR_TIMEOUT);
      // drain what this warp still has in flight (bounded), then stop
      for (int kk = k + 1; kk < issued; ++kk)
        mbar_wait_bounded(&bars[warp][kk % NST], (kk / NST) & 1, 1u << 16);
      break;
    }
    const uint32_t kpage = wbase + st * STAGE;
    const uint32_t vpage = kpage + Geo::PAGE_BYTES;

    float s[2][4];
#pragma unroll
    for (int j = 0; j < 2; ++j) s[j][0] = s[j][1] = s[j][2] = s[j][3] = 0.f;
    qk_page<D, KV>(s, 0, qf, kpage, lane);

    const int tbase = tok0 + (warp + NW * k) * kBS;
    float mx0 = -INFINITY, mx8 = -INFINITY;
#pragma unroll
    for (int j = 0; j < 2; ++j)
#pragma unroll
      for (int e = 0; e < 2; ++e) {
        const bool valid = tbase + s_col_token<KV>(j, c, e) < tok1;
        s[j][e] = valid ? s[j][e] * sl2 : -INFINITY;
        s[j][2 + e] = valid ? s[j][2 + e] * sl2 : -INFINITY;
        mx0 = fmaxf(mx0, s[j][e]);
        mx8 = fmaxf(mx8, s[j][2 + e]);
      }
    mx0 = quad_max(mx0);
    const float mn0 = fmaxf(m0, mx0);
    const float ms0 = (mn0 == -INFINITY) ? 0.f : mn0;
    const float a0 = exp2f(m0 - ms0);
    m0 = mn0;
    float pr[2][4];
    float rs0 = 0.f, rs8 = 0.f;
#pragma unroll
    for (int j = 0; j < 2; ++j)
#pragma unroll
      for (int e = 0; e < 2; ++e) {
        pr[j][e] = exp2f(s[j][e] - ms0);
        rs0 += pr[j][e];
      }
    l0 = l0 * a0 + rs0;
    float a8 = 1.f;
    if constexpr (MROWS == 16) {
      mx8 = quad_max(mx8);
      const float mn8 = fmaxf(m8, mx8);
      const float ms8 = (mn8 == -INFINITY) ? 0.f : mn8;
      a8 = exp2f(m8 - ms8);
      m8 = mn8;
#pragma unroll
      for (int j = 0; j < 2; ++j)
#pragma unroll
        for (int e = 0; e < 2; ++e) {
          pr[j][2 + e] = exp2f(s[j][2 + e] - ms8);
          rs8 += pr[j][2 + e];
        }
      l8 = l8 * a8 + rs8;
    } else {
#pragma unroll
      for (int j = 0; j < 2; ++j) pr[j][2] = pr[j][3] = 0.f;
    }
#pragma unroll
    for (int t = 0; t < D / 8; ++t) {
      oacc[t][0] *= a0;
      oacc[t][1] *= a0;
      if constexpr (MROWS == 16) {
        oacc[t][2] *= a8;
        oacc[t][3] *= a8;
      }
    }
    uint32_t pa[4];
    pack_p<KV>(pa, pr, 0);
    pv_page<D, KV>(oacc, pa, vpage, lane);

    __syncwarp();
    if (lane == 0 && k + NST < nmine) {
      fence_proxy_async_smem();
      issue(k + NST);
    }
    issued = min(k + 1 + NST, nmine);
  }
  (void)aborted;

  // ---- merge the warps of this CTA ----------------------------------------------
  const float ls0 = quad_sum(l0);
  const float ls8 = quad_sum(l8);
  if (c == 0) {
    red_m[warp][g] = m0;
    red_l[warp][g] = ls0;
    if constexpr (MROWS == 16) {
      red_m[warp][g + 8] = m8;
      red_l[warp][g + 8] = ls8;
    }
  }
  __syncthreads();  // every warp is done with its ring: the pipeline smem is free
  float M0 = -INFINITY, M8 = -INFINITY;
#pragma unroll
  for (int w = 0; w < NW; ++w) {
    M0 = fmaxf(M0, red_m[w][g]);
    if constexpr (MROWS == 16) M8 = fmaxf(M8, red_m[w][g + 8]);
  }
  const float f0 = (m0 == -INFINITY) ? 0.f : exp2f(m0 - M0);
  const float f8 = (MROWS == 16 && m8 != -INFINITY) ? exp2f(m8 - M8) : 0.f;
  float* obuf = reinterpret_cast<float*>(basep);
#pragma unroll
  for (int t = 0; t < D / 8; ++t)
#pragma unroll
    for (int e = 0; e < 2; ++e) {
      const int d = o_col_dim<D, KV>(t, c, e);
      if (g < G) obuf[(warp * MROWS + g) * D + d] = oacc[t][e] * f0;
      if (MROWS == 16 && g + 8 < G) obuf[(warp * MROWS + g + 8) * D + d] = oacc[t][2 + e] * f8;
    }
  __syncthreads();

  const float vscale = (KV == KV_E4M3) ? p.v_scales[h] : 1.f;
  const int64_t row0 = (int64_t)b * p.Hq + h * G;
  for (int idx = threadIdx.x; idx < G * (D / 2); idx += NW * 32) {
    const int r = idx / (D / 2), d = 2 * (idx % (D / 2));
    float M = -INFINITY;
#pragma unroll
    for (int w = 0; w < NW; ++w) M = fmaxf(M, red_m[w][r]);
    float L = 0.f, o0 = 0.f, o1 = 0.f;
#pragma unroll
    for (int w = 0; w < NW; ++w) {
      if (red_m[w][r] != -INFINITY) L += red_l[w][r] * exp2f(red_m[w][r] - M);
      o0 += obuf[(w * MROWS + r) * D + d];
      o1 += obuf[(w * MROWS + r) * D + d + 1];
    }
    const bool nonempty = L > 0.f;
    const float inv = nonempty ? 1.f / L : 0.f;
    if (nparts == 1) {
      const float v0 = o0 * inv * vscale, v1 = o1 * inv * vscale;
      uint32_t packed = pack2<QBF16>(v0, v1);
      *reinterpret_cast<uint32_t*>(static_cast<uint16_t*>(p.out) + (row0 + r) * D + d) = packed;
      if (d == 0 && p.out_lse != nullptr)
        p.out_lse[row0 + r] = nonempty ? (M + log2f(L)) * kLn2 : -INFINITY;
    } else {
      const int64_t wrow = (row0 + r) * p.max_parts + part_idx;
      *reinterpret_cast<float2*>(p.ws_o + wrow * D + d) = make_float2(o0 * inv, o1 * inv);
      if (d == 0) p.ws_lse[wrow] = nonempty ? M + log2f(L) : -INFINITY;
    }
  }
}

// Combines the partitions of every (sequence, query head) whose context
// spans more than one partition:
//   LSE = log2 sum_p 2^{lse_p},  out = v_scale * sum_p 2^{lse_p - LSE} o_p,
// empty partitions (lse_p = -inf) weigh 0. One CTA per (sequence, head).
template <int D, bool QBF16, bool FP8>
__global__ void __launch_bounds__(128) decode_merge_kernel(const DecodeParams p) {
  constexpr int NW = 4;
  constexpr int PER = D / 32;   // dims per lane
  __shared__ float red[NW];
  __shared__ float accs[NW][D];
  __shared__ float zs[NW];
  const int bh = blockIdx.x;
  const int b = bh / p.Hq, hq = bh % p.Hq;
  const int lane = threadIdx.x & 31, warp = threadIdx.x >> 5;
  int ctx = p.seq_lens[b];
  const int cap = min(p.max_seq_len, p.max_blocks * kBS);
  ctx = ctx < 0 ? 0 : (ctx > cap ? cap : ctx);
  const int nparts = ctx > 0 ? (ctx + p.part - 1) / p.part : 1;
  if (nparts <= 1) return;
  const int64_t wrow = ((int64_t)b * p.Hq + hq) * p.max_parts;
  const float* lse = p.ws_lse + wrow;

  float mx = -INFINITY;
  for (int i = threadIdx.x; i < nparts; i += 128) mx = fmaxf(mx, lse[i]);
#pragma unroll
  for (int o = 16; o > 0; o >>= 1) mx = fmaxf(mx, __shfl_xor_sync(0xffffffffu, mx, o));
  if (lane == 0) red[warp] = mx;
  __syncthreads();
  const float M = fmaxf(fmaxf(red[0], red[1]), fmaxf(red[2], red[3]));

  float acc[PER];
#pragma unroll
  for (int i = 0; i < PER; ++i) acc[i] = 0.f;
  float z = 0.f;
  if (M != -INFINITY) {
    for (int i = warp; i < nparts; i += NW) {
      const float l = lse[i];
      if (l == -INFINITY) continue;
      const float w = exp2f(l - M);
      z += w;
      const float* o = p.ws_o + (wrow + i) * D + lane * PER;
      if constexpr (PER == 4) {
        const float4 v = *reinterpret_cast<const float4*>(o);
        acc[0] += w * v.x; acc[1] += w * v.y; acc[2] += w * v.z; acc[3] += w * v.w;
      } else {
        const float2 v = *reinterpret_cast<const float2*>(o);
        acc[0] += w * v.x; acc[1] += w * v.y;
      }
    }
  }
#pragma unroll
  for (int i = 0; i < PER; ++i) accs[warp][lane * PER + i] = acc[i];
  if (lane == 0) zs[warp] = z;
  __syncthreads();
  const float Z = zs[0] + zs[1] + zs[2] + zs[3];
  const float vscale = FP8 ? p.v_scales[hq / p.G] : 1.f;
  const float inv = Z > 0.f ? vscale / Z : 0.f;
  const int64_t orow = (int64_t)b * p.Hq + hq;
  for (int d = 2 * threadIdx.x; d < D; d += 256) {
    const float v0 = (accs[0][d] + accs[1][d] + accs[2][d] + accs[3][d]) * inv;
    const float v1 = (accs[0][d + 1] + accs[1][d + 1] + accs[2][d + 1] + accs[3][d + 1]) * inv;
    *reinterpret_cast<uint32_t*>(static_cast<uint16_t*>(p.out) + orow * D + d) =
        pack2<QBF16>(v0, v1);
  }
  if (threadIdx.x == 0 && p.out_lse != nullptr)
    p.out_lse[orow] = Z > 0.f ? (M + log2f(Z)) * kLn2 : -INFINITY;
}

template <int D, int KV, bool QBF16, int MROWS>
static pkv_status launch_decode_t(const DecodeParams& p, const CUtensorMap& tmK,
                                  const CUtensorMap& tmV, cudaStream_t stream) {
  constexpr int NW = 4;
  constexpr int NST = (KV == KV_E4M3) ? 4 : 3;
  using Cfg = DecodeCfg<D, KV, QBF16, MROWS, NW, NST>;
  auto kern = decode_split_kernel<D, KV, QBF16, MROWS, NW, NST>;
  int dev = 0;
  cudaGetDevice(&dev);
  static bool attr_set[64] = {};
  if (dev < 0 || dev >= 64) return PKV_ERR_CUDA;
  if (!attr_set[dev]) {
    if (cudaFuncSetAttribute(kern, cudaFuncAttributeMaxDynamicSharedMemorySize,
                             Cfg::SMEM_BYTES) != cudaSuccess)
      return PKV_ERR_CUDA;
    attr_set[dev] = true;
  }
  dim3 grid(p.max_parts, p.Hkv, p.B);
  kern<<<grid, NW * 32, Cfg::SMEM_BYTES, stream>>>(tmK, tmV, p);
  if (cudaGetLastError() != cudaSuccess) return PKV_ERR_CUDA;
  if (p.max_parts > 1) {
    decode_merge_kernel<D, QBF16, KV == KV_E4M3><<<p.B * p.Hq, 128, 0, stream>>>(p);
    if (cudaGetLastError() != cudaSuccess) return PKV_ERR_CUDA;
  }
  return PKV_OK;
}

template <int D, int KV, bool QBF16>
static pkv_status launch_decode_rows(const DecodeParams& p, const CUtensorMap& tmK,
                                     const CUtensorMap& tmV, cudaStream_t stream) {
  if (p.G <= 8) return launch_decode_t<D, KV, QBF16, 8>(p, tmK, tmV, stream);
  return launch_decode_t<D, KV, QBF16, 16>(p, tmK, tmV, stream);
}

template <int D>
static pkv_status launch_decode_d(const DecodeParams& p, pkv_dtype q_dtype, pkv_dtype kv_dtype,
                                  const CUtensorMap& tmK, const CUtensorMap& tmV,
                                  cudaStream_t stream) {
  const bool qbf = (q_dtype == PKV_BF16);
  if (kv_dtype == PKV_FP8_E4M3)
    return qbf ? launch_decode_rows<D, KV_E4M3, true>(p, tmK, tmV, stream)
               : launch_decode_rows<D, KV_E4M3, false>(p, tmK, tmV, stream);
  if (kv_dtype == PKV_BF16) return launch_decode_rows<D, KV_BF16, true>(p, tmK, tmV, stream);
  return launch_decode_rows<D, KV_F16, false>(p, tmK, tmV, stream);
}

pkv_status launch_decode(const DecodeParams& p, int head_dim, pkv_dtype q_dtype,
                         pkv_dtype kv_dtype, const CUtensorMap& tmK, const CUtensorMap& tmV,
                         cudaStream_t stream) {
  if (head_dim == 128) return launch_decode_d<128>(p, q_dtype, kv_dtype, tmK, tmV, stream);
  return launch_decode_d<64>(p, q_dtype, kv_dtype, tmK, tmV, stream);
}

}  // namespace pkv
