// decode_kernel.cuh — the paged-KV decode kernel and its launch helpers,
// instantiated by decode.cu (TMA page loads, block sizes 16/32/64) and by
// decode_gather.cu (per-row cp.async gathers, block sizes 1/2/4/8).
//
// Follows "flash attention decode (online softmax, paged KV, GQA)" and
// "Split-KV paged attention for long context" (rvLLM: High-performance LLM
// inference in Rust, Kernel Compiler Stack; Tier 2: Hand-written CUDA
// kernels; FA3 v3 Attention Kernel, "split-KV ... distributes KV tiles across
// thread blocks") and the log-sum-exp merge of partial attention (rapid_llm
// README, feature table, "Decode context parallelism").
//
// Work decomposition: one CTA per (CTA partition, KV head, sequence); a CTA
// partition is `part` consecutive tokens of one context. With warp
// partitions (an explicit partition size, pages loaded by TMA) warp w takes
// the w-th run of `wpart` tokens of it, one split-KV partition with its own
// online softmax; otherwise the CTA's NW warps take the CTA partition's
// pages round-robin. Each warp runs its own NST-deep
// ring of TMA loads (one K page + one V page per stage, completion on an
// mbarrier), issued by the warp itself as soon as it has read a stage, so
// every warp keeps its own stream of requests in flight. The GQA group's
// query heads sit in the MMA N dimension (decode_frags.cuh), so each K/V byte
// is read from HBM once per call. Each warp runs an online softmax in the
// log2 domain; at the end the warps are merged through shared memory (the
// ring's space, then free) by log-sum-exp. A sequence with one CTA partition
// is written out directly. Otherwise the CTA partition's normalised output
// and its log2-sum-exp go to the workspace and a per-(sequence, KV head)
// counter is bumped; the CTA whose bump completes the count merges the CTA
// partitions:
//   LSE = log2 sum_p 2^{lse_p},  out = v_scale * sum_p 2^{lse_p - LSE} o_p.
// (With warp partitions the split-KV partitions are thus merged in two
// levels, the LSE merge being associative.)
#pragma once
#include <cuda.h>
#include "decode_frags.cuh"
#include "launch.h"

namespace pkv {


template <int D, int KV, int NT, int NW, int NST>
struct DecodeCfg {
  using Geo = PageGeom<D, KV>;
  static constexpr int STAGE_BYTES = 2 * Geo::PAGE_BYTES;
  static constexpr int RING_BYTES = NW * NST * STAGE_BYTES;
  static constexpr int OBUF_BYTES = NW * 8 * NT * D * 4;      // warp merge, aliases the ring
  static constexpr int SMEM_BYTES =
      1024 + (RING_BYTES > OBUF_BYTES ? RING_BYTES : OBUF_BYTES);
};

// Full-first CTA order (a 1-D grid of B * Hkv * grid_parts CTAs): CTA L
// takes the L-th work item of a list that holds every full CTA partition
// first (sequence by sequence, KV head, then partition), then each
// sequence's last, shorter partition (and the single empty one of a
// zero-length context) in order of decreasing length, ties by sequence. The
// hardware hands out CTAs in index order as SMs free up, so this is a
// longest-first schedule: the short partitions fill the final wave instead
// of full ones starting late. Every CTA derives the list from seq_lens
// (B <= kFullFirstMaxSeqs values, in the dynamic shared memory, free at this
// point).
// Returns false for CTAs past the list. Invalid seq_lens are clamped as in
// the grid order, and CTA 0 flags them.
template <int NW>
__device__ bool decode_item_full_first(const DecodeParams& p, int cap, int* s_tmp, int& part_idx,
                                       int& h, int& b, int& ctx) {
  constexpr int NTH = NW * 32;
  __shared__ int s_wsum[NW];
  __shared__ int s_item[3];
  const int tid = threadIdx.x, lane = tid & 31, warp = tid >> 5;
  const int B = p.B, Hkv = p.Hkv, part = p.part;
  const int L = blockIdx.x;
  int* s_ctx = s_tmp;          // [B] clamped context lengths
  int* s_last = s_tmp + B;     // [B] length of the last partial partition, -1 if none
  bool bad = false;
  for (int i = tid; i < B; i += NTH) {
    int v = p.seq_lens[i];
    if (v < 0 || v > cap) {
      bad = true;
      v = v < 0 ? 0 : cap;
    }
    s_ctx[i] = v;
    s_last[i] = (v == 0) ? 0 : ((v % part) ? v % part : -1);
  }
  if (tid == 0) s_item[0] = -1;
  if (__syncthreads_or(bad) && L == 0 && tid == 0) atomicOr(p.err, PKV_DEVERR_SEQ_LEN);
  // exclusive scan of the full partitions over sequences (consecutive
  // sequences per thread)
  const int per = (B + NTH - 1) / NTH;
  const int b_lo = min(B, tid * per), b_hi = min(B, b_lo + per);
  int mine = 0;
  for (int i = b_lo; i < b_hi; ++i) mine += s_ctx[i] / part;
  int incl = mine;
#pragma unroll
  for (int o = 1; o < 32; o <<= 1) {
    const int v = __shfl_up_sync(0xffffffffu, incl, o);
    if (lane >= o) incl += v;
  }
  if (lane == 31) s_wsum[warp] = incl;
  __syncthreads();
  int before = 0, nfull = 0;
#pragma unroll
  for (int w = 0; w < NW; ++w) {
    before += (w < warp) ? s_wsum[w] : 0;
    nfull += s_wsum[w];
  }
  const int64_t full_items = (int64_t)Hkv * nfull;
  if (L < full_items) {
    int f = before + incl - mine;
    for (int i = b_lo; i < b_hi; ++i) {
      const int nf = s_ctx[i] / part;
      const int64_t lo = (int64_t)Hkv * f;
      if (L >= lo && L < lo + (int64_t)Hkv * nf) {
        const int loc = (int)(L - lo);
        s_item[0] = i;
        s_item[1] = loc / nf;
        s_item[2] = loc % nf;
      }
      f += nf;
    }
  } else {
    const int64_t j = L - full_items;
    const int r = (int)(j / Hkv), hh = (int)(j % Hkv);
    if (r < B) {
      for (int i = tid; i < B; i += NTH) {
        const int li = s_last[i];
        if (li < 0) continue;
        int rank = 0;
        for (int k = 0; k < B; ++k) {
          const int lk = s_last[k];
          rank += (lk > li) || (lk == li && k < i);
        }
        if (rank == r) {
          s_item[0] = i;
          s_item[1] = hh;
          s_item[2] = s_ctx[i] / part;
        }
      }
    }
  }
  __syncthreads();
  b = s_item[0];
  if (b < 0) return false;
  h = s_item[1];
  part_idx = s_item[2];
  ctx = s_ctx[b];
  __syncthreads();   // the ring's space is reused from here on
  return true;
}

template <int D, int KV, bool QBF16, int NT, int NW, int NST, bool GATHER, bool FF>
__global__ void __launch_bounds__(NW * 32)
    decode_kernel(const __grid_constant__ CUtensorMap tmK, const __grid_constant__ CUtensorMap tmV,
                  const DecodeParams p) {
  using Geo = PageGeom<D, KV>;
  using Cfg = DecodeCfg<D, KV, NT, NW, NST>;
  constexpr int STAGE = Cfg::STAGE_BYTES;
  constexpr int NH = 8 * NT;                       // head columns of the N dimension
  // TMA mode keeps one page row per 16-token page, gather mode one cache row per token
  constexpr int NIDS = GATHER ? kGatherMaxPartitionTokens : kMaxPartitionTokens / kBS;
  extern __shared__ uint8_t smem_raw[];
  __shared__ uint64_t bars[NW][NST];
  __shared__ float red_m[NW][NH];
  __shared__ float red_l[NW][NH];
  __shared__ int s_ids[NIDS];
  __shared__ int s_last;
  __shared__ int s_stuck;         // a warp's copies may still land in the ring
  __shared__ uint64_t s_mbar;     // the merge's bulk copies of the partials

  const int tid = threadIdx.x, lane = tid & 31, warp = tid >> 5;
  const int g = lane >> 2, c = lane & 3;
  const int G = p.G;
  // launched as a programmatic dependent: the CTA is resident early, and
  // reads nothing before the kernel ahead of it (the cache write) is done;
  // in the early-start mode it reads what that kernel does not write first
  const bool early = !GATHER && p.early != 0;
  if (p.wait_prior && !early) griddep_wait();

  const int cap = min(p.max_seq_len, p.max_blocks << p.bs_log2);
  int part_idx, h, b, ctx;
  if constexpr (FF) {
    // (the dynamic shared memory is free until the ring starts)
    if (!decode_item_full_first<NW>(p, cap, reinterpret_cast<int*>(smem_raw), part_idx, h, b,
                                    ctx))
      return;
  } else {
    part_idx = blockIdx.x;
    h = blockIdx.y;
    b = blockIdx.z;
    ctx = p.seq_lens[b];
    if (ctx < 0 || ctx > cap) {
      if (tid == 0 && part_idx == 0 && h == 0) atomicOr(p.err, PKV_DEVERR_SEQ_LEN);
      ctx = ctx < 0 ? 0 : cap;
    }
  }
  const int nparts = ctx > 0 ? (ctx + p.part - 1) / p.part : 1;
  if (part_idx >= nparts) return;
  const int tok0 = part_idx * p.part;
  const int tok1 = min(ctx, tok0 + p.part);
  const int npages = (tok1 - tok0 + kBS - 1) / kBS;
  const int page0 = tok0 / kBS;
  // warp partitions: warp w takes the CTA's pages [w * ppw, (w + 1) * ppw);
  // otherwise (ppw = 0) pages w, w + NW, w + 2 NW, ...
  const int ppw = GATHER ? 0 : p.wpart / kBS;

  const uint32_t raw_base = smem_u32(smem_raw);
  const uint32_t base = (raw_base + 1023u) & ~1023u;
  uint8_t* basep = smem_raw + (base - raw_base);

  if constexpr (GATHER) {
    // cache row ((block * Hkv + h) * BS + offset) of every token of the
    // partition; the rows past its end repeat the last token's row
    const int bmask = (1 << p.bs_log2) - 1;
    for (int i = tid; i < npages * kBS; i += NW * 32) {
      const int t = min(tok0 + i, tok1 - 1);
      int id = p.block_tables[(int64_t)b * p.max_blocks + (t >> p.bs_log2)];
      if (id < 0 || id >= p.num_blocks) {
        atomicOr(p.err, PKV_DEVERR_BLOCK_ID);
        id = 0;
      }
      s_ids[i] = ((id * p.Hkv + h) << p.bs_log2) + (t & bmask);
    }
  } else {
    // page rows of the tensor maps: a block of 16 << ppb_shift tokens holds
    // that many consecutive 16-token pages per KV head
    const int sub_mask = (1 << p.ppb_shift) - 1;
    for (int i = tid; i < npages; i += NW * 32) {
      const int pg = page0 + i;
      int id = p.block_tables[(int64_t)b * p.max_blocks + (pg >> p.ppb_shift)];
      if (id < 0 || id >= p.num_blocks) {
        atomicOr(p.err, PKV_DEVERR_BLOCK_ID);
        id = 0;
      }
      s_ids[i] = ((id * p.Hkv + h) << p.ppb_shift) + (pg & sub_mask);
    }
  }
  if (tid == 0) {
    if constexpr (!GATHER) {          // the gather path has no tensor maps
      prefetch_tensormap(&tmK);
      prefetch_tensormap(&tmV);
    }
#pragma unroll
    for (int w = 0; w < NW; ++w)
#pragma unroll
      for (int s = 0; s < NST; ++s) mbar_init(&bars[w][s], GATHER ? 32 : 1);
    mbar_init(&s_mbar, 1);
    fence_barrier_init();
    s_stuck = 0;
  }
  __syncthreads();

  // ---- per-warp ring: TMA loads issued by lane 0, or (gather mode) 16-byte
  // cp.async copies of the page's rows issued by all 32 lanes into the same
  // swizzled layout, each lane's copies completing on the stage's mbarrier ----
  const uint32_t wbase = base + warp * NST * STAGE;
  uint8_t* wbasep = basep + warp * NST * STAGE;
  const int nmine = ppw ? max(0, min(ppw, npages - warp * ppw))
                       : (warp < npages ? (npages - warp + NW - 1) / NW : 0);
  // the CTA's page index of this warp's k-th page
  auto page_of = [&](int k) { return ppw ? warp * ppw + k : warp + NW * k; };
  const uint8_t* kcache = static_cast<const uint8_t*>(p.k_cache);
  const uint8_t* vcache = static_cast<const uint8_t*>(p.v_cache);
  // KV pages are read once per call: mark them first to go from L2, so they
  // do not push out what is reused (block tables, queries, partials)
  const uint64_t evict_first = policy_evict_first();
  auto issue = [&](int k) {
    const int st = k % NST;
    uint64_t* bar = &bars[warp][st];
    uint8_t* dst = wbasep + st * STAGE;
    if constexpr (GATHER) {
      const int* rows = s_ids + page_of(k) * kBS;
      constexpr int CPR = Geo::ROW_BYTES / 16;             // 16-byte chunks per row
      // Copies a lane keeps in flight: NST stages of K and V. Configurations
      // up to 32 ran on GB300; one with 64 (bf16, D = 256, two stages) raised
      // an illegal-instruction fault, so the gather path stays within 32.
      static_assert(NST * 2 * kBS * CPR / 32 <= 32, "too many cp.async in flight per thread");
#pragma unroll
      for (int u = 0; u < kBS * CPR / 32; ++u) {
        const int ch = lane + 32 * u, r = ch / CPR, x = (ch % CPR) * 16;
        const uint32_t so = (x / Geo::BOX_ROW_BYTES) * Geo::BOX_BYTES +
                            Geo::swz(r, x % Geo::BOX_ROW_BYTES);
        const int64_t go = (int64_t)rows[r] * Geo::ROW_BYTES + x;
        cp_async16_hint(dst + so, kcache + go, evict_first);
        cp_async16_hint(dst + Geo::PAGE_BYTES + so, vcache + go, evict_first);
      }
      cp_async_mbar_arrive_noinc(bar);
    } else {
      const int z = s_ids[page_of(k)];
      mbar_arrive_expect_tx(bar, STAGE);
#pragma unroll
      for (int bx = 0; bx < Geo::NBOX; ++bx) {
        tma_load_3d_hint(dst + bx * Geo::BOX_BYTES, &tmK, bar, bx * Geo::BOX_ELEMS, 0, z,
                         evict_first);
        tma_load_3d_hint(dst + Geo::PAGE_BYTES + bx * Geo::BOX_BYTES, &tmV, bar,
                         bx * Geo::BOX_ELEMS, 0, z, evict_first);
      }
    }
  };
  // the page holding the newest token (position ctx - 1) is written by the
  // kernel ahead: in the early-start mode its load waits for that kernel
  const int new_pg = ctx > 0 ? (ctx - 1) / kBS - page0 : -1;
  const int new_k = ppw ? (new_pg / ppw == warp ? new_pg % ppw : -1)
                        : (new_pg % NW == warp ? new_pg / NW : -1);
  const int held = (early && new_pg >= 0 && new_pg < npages && new_k >= 0 && new_k < NST)
                       ? new_k : -1;
  if (GATHER || lane == 0)
    for (int k = 0; k < NST && k < nmine; ++k)
      if (k != held) issue(k);
  int issued = min(NST, nmine);
  if (early && p.wait_prior) {
    griddep_wait();
    if (held >= 0 && lane == 0) issue(held);
  }

  // ---- query fragments (heads in N), straight from global memory --------------------
  const uint16_t* qb = static_cast<const uint16_t*>(p.q) + ((int64_t)b * p.Hq + h * G) * D;
  uint32_t qf[NT][D / 16][2];
  int qshift;
  load_qT_frags<D, KV, QBF16, NT>(qf, qb, G, lane, qshift);

  float oacc[NT][D / 16][4];
#pragma unroll
  for (int nt = 0; nt < NT; ++nt)
#pragma unroll
    for (int t = 0; t < D / 16; ++t)
      oacc[nt][t][0] = oacc[nt][t][1] = oacc[nt][t][2] = oacc[nt][t][3] = 0.f;
  float m[NT][2], l[NT][2];
#pragma unroll
  for (int nt = 0; nt < NT; ++nt) {
    m[nt][0] = m[nt][1] = -INFINITY;
    l[nt][0] = l[nt][1] = 0.f;
  }
  // q was scaled by 2^-qshift for the f16 MMAs: scale the scores back (exact)
  const float sl2 = p.qk_scale_log2 * (KV == KV_E4M3 ? p.k_scales[h] : 1.f) * pow2f(qshift);
  const int tk0 = st_row_token<KV>(g, 0), tk8 = st_row_token<KV>(g, 1);

  for (int k = 0; k < nmine; ++k) {
    const int st = k % NST;
    bool ok = mbar_wait_bounded(&bars[warp][st], (k / NST) & 1);
    ok = __all_sync(0xffffffffu, ok);
    if (!ok) {
      if (lane == 0) atomicOr(p.err, PKV_DEVERR_TIMEOUT);
      // let what this warp still has in flight land (bounded), then stop; if
      // that wait gives up too, a late copy could still land in the ring, so
      // the CTA leaves the ring's space (the merge buffer below) alone
      bool drained = true;
      for (int kk = k + 1; kk < issued; ++kk)
        drained &= mbar_wait_bounded(&bars[warp][kk % NST], (kk / NST) & 1, 1u << 16);
      if (!__all_sync(0xffffffffu, drained) && lane == 0) s_stuck = 1;
      break;
    }
    const uint32_t kpage = wbase + st * STAGE;
    const uint32_t vpage = kpage + Geo::PAGE_BYTES;
    const int tbase = tok0 + page_of(k) * kBS;
    if (tok1 - tbase < kBS) {
      // the last page of the context: its rows past the end get weight 0, and
      // whatever they hold must not turn that into NaN, so zero them in V
      zero_page_rows<D, KV>(wbasep + st * STAGE + Geo::PAGE_BYTES, tok1 - tbase, lane);
      if constexpr (!GATHER) fence_proxy_async_smem();
      __syncwarp();
    }
    float s[NT][4];
#pragma unroll
    for (int nt = 0; nt < NT; ++nt) s[nt][0] = s[nt][1] = s[nt][2] = s[nt][3] = 0.f;
    // E4M3: take the page into registers and refill the stage at once, so the
    // next load is in flight while this page's math runs.
    E4M3PageRegs<D> pr;
    if constexpr (KV == KV_E4M3) {
      load_e4m3_page<D>(pr, kpage, vpage, lane);
      __syncwarp();
      if ((GATHER || lane == 0) && k + NST < nmine) {
        if constexpr (!GATHER) fence_proxy_async_smem();
        issue(k + NST);
      }
      kq_regs<D, NT>(s, qf, pr.k);
    } else {
      kq_page<D, KV, NT>(s, qf, kpage, lane);
    }

    // online softmax in the log2 domain, against a reference max per column
    // that moves only when the page's max outgrows it by kRefSlackLog2, so the
    // accumulators are rescaled rarely (the probabilities stay below 2^8)
    const bool v0 = tbase + tk0 < tok1, v8 = tbase + tk8 < tok1;
    float pmax[NT][2];
    bool move = false;
#pragma unroll
    for (int nt = 0; nt < NT; ++nt)
#pragma unroll
      for (int e = 0; e < 2; ++e) {
        s[nt][e] = v0 ? s[nt][e] * sl2 : -INFINITY;
        s[nt][2 + e] = v8 ? s[nt][2 + e] * sl2 : -INFINITY;
        pmax[nt][e] = col_max8(fmaxf(s[nt][e], s[nt][2 + e]));
        move |= pmax[nt][e] > m[nt][e] + kRefSlackLog2;
      }
    if (__any_sync(0xffffffffu, move)) {
#pragma unroll
      for (int nt = 0; nt < NT; ++nt)
#pragma unroll
        for (int e = 0; e < 2; ++e) {
          if (pmax[nt][e] > m[nt][e] + kRefSlackLog2) {
            const float alpha = m[nt][e] == -INFINITY ? 0.f : exp2f(m[nt][e] - pmax[nt][e]);
            m[nt][e] = pmax[nt][e];
            l[nt][e] *= alpha;
#pragma unroll
            for (int t = 0; t < D / 16; ++t) {
              oacc[nt][t][e] *= alpha;
              oacc[nt][t][2 + e] *= alpha;
            }
          }
        }
    }
#pragma unroll
    for (int nt = 0; nt < NT; ++nt)
#pragma unroll
      for (int e = 0; e < 2; ++e) {
        const float ms = m[nt][e] == -INFINITY ? 0.f : m[nt][e];
        const float p0 = exp2f(s[nt][e] - ms), p8 = exp2f(s[nt][2 + e] - ms);
        l[nt][e] += p0 + p8;
        s[nt][e] = p0;
        s[nt][2 + e] = p8;
      }
    uint32_t pb[NT][2];
    pT_frags<KV, NT>(pb, s);
    if constexpr (KV == KV_E4M3) {
      vp_regs<D, NT>(oacc, pb, pr.v);
    } else {
      vp_page<D, KV, NT>(oacc, pb, vpage, lane);
      __syncwarp();
      if ((GATHER || lane == 0) && k + NST < nmine) {
        if constexpr (!GATHER) fence_proxy_async_smem();
        issue(k + NST);
      }
    }
    issued = min(k + 1 + NST, nmine);
  }

  // ---- merge the warps of this CTA ----------------------------------------------------
#pragma unroll
  for (int nt = 0; nt < NT; ++nt)
#pragma unroll
    for (int e = 0; e < 2; ++e) {
      l[nt][e] = col_sum8(l[nt][e]);
      if (g == 0) {
        red_m[warp][8 * nt + 2 * c + e] = m[nt][e];
        red_l[warp][8 * nt + 2 * c + e] = l[nt][e];
      }
    }
  __syncthreads();  // every warp is done with its ring: the ring's space is free
  if (s_stuck) {
    // (after a timeout whose drain gave up; the error word holds the timeout)
    // no output or partial from this CTA, only its count, so that the
    // (b, h) counter still completes and comes back to zero
    if (nparts > 1 && tid == 0) {
      unsigned long long* ctr = p.done + (int64_t)b * p.Hkv + h;
      if (atom_add_acq_rel_gpu(ctr, 1ull) + 1 == (unsigned long long)nparts) *ctr = 0ull;
    }
    return;
  }
  float* obuf = reinterpret_cast<float*>(basep);   // [NW][G][D]
#pragma unroll
  for (int nt = 0; nt < NT; ++nt)
#pragma unroll
    for (int e = 0; e < 2; ++e) {
      const int hh = 8 * nt + 2 * c + e;
      if (hh < G) {
        float M = -INFINITY;
#pragma unroll
        for (int w = 0; w < NW; ++w) M = fmaxf(M, red_m[w][hh]);
        const float f = (m[nt][e] == -INFINITY) ? 0.f : exp2f(m[nt][e] - M);
        float* orow = obuf + (warp * G + hh) * D;
#pragma unroll
        for (int t = 0; t < D / 16; ++t) {
          orow[ot_row_dim<D, KV>(t, g, 0)] = oacc[nt][t][e] * f;
          orow[ot_row_dim<D, KV>(t, g, 1)] = oacc[nt][t][2 + e] * f;
        }
      }
    }
  __syncthreads();

  const float vscale = (KV == KV_E4M3) ? p.v_scales[h] : 1.f;
  const int64_t row0 = (int64_t)b * p.Hq + h * G;
  for (int idx = tid; idx < G * (D / 2); idx += NW * 32) {
    const int hh = idx / (D / 2), d = 2 * (idx % (D / 2));
    float M = -INFINITY;
#pragma unroll
    for (int w = 0; w < NW; ++w) M = fmaxf(M, red_m[w][hh]);
    float L = 0.f, o0 = 0.f, o1 = 0.f;
#pragma unroll
    for (int w = 0; w < NW; ++w) {
      if (red_m[w][hh] != -INFINITY) L += red_l[w][hh] * exp2f(red_m[w][hh] - M);
      o0 += obuf[(w * G + hh) * D + d];
      o1 += obuf[(w * G + hh) * D + d + 1];
    }
    const bool nonempty = L > 0.f;
    const float inv = nonempty ? 1.f / L : 0.f;
    if (nparts == 1) {
      *reinterpret_cast<uint32_t*>(static_cast<uint16_t*>(p.out) + (row0 + hh) * D + d) =
          pack2<QBF16>(o0 * inv * vscale, o1 * inv * vscale);
      if (d == 0 && p.out_lse != nullptr)
        p.out_lse[row0 + hh] = nonempty ? (M + log2f(L)) * kLn2 : -INFINITY;
    } else {
      const int64_t wrow = (row0 + hh) * p.max_parts + part_idx;
      *reinterpret_cast<float2*>(p.ws_o + wrow * D + d) = make_float2(o0 * inv, o1 * inv);
      if (d == 0) p.ws_lse[wrow] = nonempty ? M + log2f(L) : -INFINITY;
    }
  }
  if (nparts == 1) return;

  // ---- the CTA that completes the last partition of (b, h) merges them ------------------
  // Finished-partition counter of (b, h). The CTA that completes the count
  // merges and sets it back to zero, so the workspace is ready for the next
  // call (a CUDA-graph replay included) without a clear of its own. A count
  // at or past nparts means the counters did not start at zero. One thread
  // bumps it with release semantics after the barrier (publishing every
  // thread's partial writes) and acquire semantics (so the merging CTA,
  // after the next barrier, reads every other partition's writes).
  __syncthreads();
  unsigned long long* ctr = p.done + (int64_t)b * p.Hkv + h;
  if (tid == 0) {
    const unsigned long long before = atom_add_acq_rel_gpu(ctr, 1ull);
    if (before >= (unsigned long long)nparts) atomicOr(p.err, PKV_DEVERR_COUNTER);
    s_last = (before + 1 == (unsigned long long)nparts);
  }
  __syncthreads();
  if (!s_last) return;
  if (tid == 0) *ctr = 0ull;
  // The CTA partials of (b, h) come into shared memory (the ring's space) in
  // chunks of CH partitions. A head's partitions are consecutive rows of the
  // workspace, so a chunk is one bulk copy per head plus the chunk's
  // log2-sum-exps, all in flight before a single wait: one round trip per
  // chunk, however many partitions it holds. Each thread then owns float4
  // columns f = tid, tid + NW*32, ... of the G x D outputs and folds the
  // chunk's partitions into a running log-sum-exp (max M, sum Z, weighted
  // sum acc), rescaling when a partition's log2-sum-exp exceeds M.
  constexpr int NTH = NW * 32;
  constexpr int NF = (NH * (D / 4) + NTH - 1) / NTH;   // float4 columns per thread
  constexpr int AVAIL = Cfg::SMEM_BYTES - 1024;         // the ring's space
  const int CH = max(1, min(nparts, (AVAIL - 16) / (G * (D + 1) * 4)));
  float* s_lse = reinterpret_cast<float*>(basep);                       // [G][CH]
  float* s_o = reinterpret_cast<float*>(basep + ((G * CH * 4 + 15) & ~15));  // [G][CH][D]
  float M[NF], Z[NF];
  float4 acc[NF];
#pragma unroll
  for (int i = 0; i < NF; ++i) {
    M[i] = -INFINITY;
    Z[i] = 0.f;
    acc[i] = make_float4(0.f, 0.f, 0.f, 0.f);
  }
  const float* lse_rows = p.ws_lse + row0 * (int64_t)p.max_parts;
  for (int c0 = 0, ci = 0; c0 < nparts; c0 += CH, ++ci) {
    const int n = min(CH, nparts - c0);
    if (tid == 0) {
      // the partials were written through the generic proxy; the acquire
      // above ordered them before this thread's reads, and this fence before
      // its bulk copies
      fence_proxy_async_global();
      mbar_arrive_expect_tx(&s_mbar, (uint32_t)(G * n * D * 4));
      for (int hh = 0; hh < G; ++hh)
        bulk_load(s_o + hh * CH * D, p.ws_o + ((row0 + hh) * p.max_parts + c0) * D,
                  (uint32_t)(n * D * 4), &s_mbar);
    }
#pragma unroll 4
    for (int i = tid; i < G * n; i += NTH) {
      const int hh = i / n, sp = i - hh * n;
      s_lse[hh * CH + sp] = ldcg_f32(lse_rows + hh * p.max_parts + c0 + sp);
    }
    // the vote is also the barrier that publishes the log2-sum-exps; a CTA
    // whose copies did not all land leaves as one, after waiting once more
    // (bounded), since they target its own shared memory
    const bool landed = mbar_wait_bounded(&s_mbar, ci & 1);
    if (__syncthreads_or(!landed)) {
      if (tid == 0) atomicOr(p.err, PKV_DEVERR_TIMEOUT);
      mbar_wait_bounded(&s_mbar, ci & 1);
      return;
    }
#pragma unroll
    for (int i = 0; i < NF; ++i) {
      const int f = tid + i * NTH;
      if (f < G * (D / 4)) {
        const int hh = f / (D / 4), d4 = f - hh * (D / 4);
        for (int sp = 0; sp < n; ++sp) {
          const float ls = s_lse[hh * CH + sp];
          if (ls == -INFINITY) continue;
          if (ls > M[i]) {
            const float sc = M[i] == -INFINITY ? 0.f : exp2f(M[i] - ls);
            acc[i].x *= sc; acc[i].y *= sc; acc[i].z *= sc; acc[i].w *= sc;
            Z[i] *= sc;
            M[i] = ls;
          }
          const float w = exp2f(ls - M[i]);
          const float4 v = *reinterpret_cast<const float4*>(s_o + (hh * CH + sp) * D + d4 * 4);
          Z[i] += w;
          acc[i].x += w * v.x; acc[i].y += w * v.y; acc[i].z += w * v.z; acc[i].w += w * v.w;
        }
      }
    }
    __syncthreads();   // the next chunk reuses the staging space
  }
#pragma unroll
  for (int i = 0; i < NF; ++i) {
    const int f = tid + i * NTH;
    if (f < G * (D / 4)) {
      const int hh = f / (D / 4), d4 = f - hh * (D / 4);
      const float inv = Z[i] > 0.f ? vscale / Z[i] : 0.f;
      *reinterpret_cast<uint2*>(static_cast<uint16_t*>(p.out) + (row0 + hh) * D + d4 * 4) =
          make_uint2(pack2<QBF16>(acc[i].x * inv, acc[i].y * inv),
                     pack2<QBF16>(acc[i].z * inv, acc[i].w * inv));
      if (d4 == 0 && p.out_lse != nullptr)
        p.out_lse[row0 + hh] = Z[i] > 0.f ? (M[i] + log2f(Z[i])) * kLn2 : -INFINITY;
    }
  }
}

// TMA ring depth per warp: CTAs of kDecodeWarps warps (several resident per
// SM) keep 3 stages of E4M3 pages or 2 of 16-bit pages; whole-context CTAs of
// kDecodeWideWarps warps (an SM each) keep 3 of either.
template <int NW, int KV>
constexpr int decode_ring_stages() {
  return NW == kDecodeWideWarps ? 3 : (KV == KV_E4M3 ? 3 : 2);
}

template <bool GATHER, int D, int KV, bool QBF16, int NT, int NW, bool FF>
static pkv_status launch_decode_t(const DecodeParams& p, const CUtensorMap& tmK,
                                  const CUtensorMap& tmV, cudaStream_t stream,
                                  bool programmatic) {
  constexpr int NST = decode_ring_stages<NW, KV>();
  // warp partitions (p.wpart > 0) are planned for kDecodeWarps warps only
  static_assert(NW == kDecodeWarps || (NW == kDecodeWideWarps && !GATHER),
                "decode CTAs have kDecodeWarps warps, or kDecodeWideWarps with TMA pages");
  using Cfg = DecodeCfg<D, KV, NT, NW, NST>;
  auto kern = decode_kernel<D, KV, QBF16, NT, NW, NST, GATHER, FF>;
  int dev = 0;
  if (cudaGetDevice(&dev) != cudaSuccess || dev < 0 || dev >= 64) return PKV_ERR_CUDA;
  static std::atomic<bool> attr_set[64];  // per device; the call is idempotent
  if (!attr_set[dev]) {
    if (cudaFuncSetAttribute(kern, cudaFuncAttributeMaxDynamicSharedMemorySize,
                             Cfg::SMEM_BYTES) != cudaSuccess)
      return PKV_ERR_CUDA;
    attr_set[dev] = true;
  }
  const dim3 grid = FF ? dim3(p.grid_parts * p.Hkv * p.B) : dim3(p.grid_parts, p.Hkv, p.B);
  if (programmatic) {
    // may start while the previous kernel on the stream still runs (it
    // reads nothing that kernel writes)
    cudaLaunchAttribute attr[1];
    attr[0].id = cudaLaunchAttributeProgrammaticStreamSerialization;
    attr[0].val.programmaticStreamSerializationAllowed = 1;
    cudaLaunchConfig_t cfg = {};
    cfg.gridDim = grid;
    cfg.blockDim = dim3(NW * 32);
    cfg.dynamicSmemBytes = Cfg::SMEM_BYTES;
    cfg.stream = stream;
    cfg.attrs = attr;
    cfg.numAttrs = 1;
    return cudaLaunchKernelEx(&cfg, kern, tmK, tmV, p) == cudaSuccess ? PKV_OK : PKV_ERR_CUDA;
  }
  kern<<<grid, NW * 32, Cfg::SMEM_BYTES, stream>>>(tmK, tmV, p);
  return cudaGetLastError() == cudaSuccess ? PKV_OK : PKV_ERR_CUDA;
}

template <bool GATHER, int D, int KV, bool QBF16, int NW, bool FF>
static pkv_status launch_decode_nt(const DecodeParams& p, const CUtensorMap& tmK,
                                   const CUtensorMap& tmV, cudaStream_t stream, bool prog) {
  if constexpr (D <= 128) {
    if (p.G > 8)
      return launch_decode_t<GATHER, D, KV, QBF16, 2, NW, FF>(p, tmK, tmV, stream, prog);
  } else {
    if (p.G > 8) return PKV_ERR_UNSUPPORTED;        // 16 head columns at D = 256: not built
  }
  return launch_decode_t<GATHER, D, KV, QBF16, 1, NW, FF>(p, tmK, tmV, stream, prog);
}

template <bool GATHER, int D, int NW, bool FF>
static pkv_status launch_decode_d(const DecodeParams& p, pkv_dtype q_dtype, pkv_dtype kv_dtype,
                                  const CUtensorMap& tmK, const CUtensorMap& tmV,
                                  cudaStream_t stream, bool prog) {
  const bool qbf = (q_dtype == PKV_BF16);
  if (kv_dtype == PKV_FP8_E4M3)
    return qbf ? launch_decode_nt<GATHER, D, KV_E4M3, true, NW, FF>(p, tmK, tmV, stream, prog)
               : launch_decode_nt<GATHER, D, KV_E4M3, false, NW, FF>(p, tmK, tmV, stream, prog);
  if (kv_dtype == PKV_BF16)
    return launch_decode_nt<GATHER, D, KV_BF16, true, NW, FF>(p, tmK, tmV, stream, prog);
  return launch_decode_nt<GATHER, D, KV_F16, false, NW, FF>(p, tmK, tmV, stream, prog);
}

// GATHER: pages gathered row by row (blocks below 16 tokens); NW: warps per
// CTA; FF: full-first CTA order (decode_item_full_first).
template <bool GATHER, int NW = kDecodeWarps, bool FF = false>
pkv_status launch_decode_mode(const DecodeParams& p, int head_dim, pkv_dtype q_dtype,
                              pkv_dtype kv_dtype, const CUtensorMap& tmK, const CUtensorMap& tmV,
                              cudaStream_t stream, bool prog) {
  if constexpr (GATHER || NW == kDecodeWideWarps) {
    // rows too wide for the gather path; rings too large for a wide CTA
    if (head_dim == 256) return PKV_ERR_UNSUPPORTED;
  } else {
    if (head_dim == 256)
      return launch_decode_d<GATHER, 256, NW, FF>(p, q_dtype, kv_dtype, tmK, tmV, stream, prog);
  }
  if (head_dim == 128)
    return launch_decode_d<GATHER, 128, NW, FF>(p, q_dtype, kv_dtype, tmK, tmV, stream, prog);
  return launch_decode_d<GATHER, 64, NW, FF>(p, q_dtype, kv_dtype, tmK, tmV, stream, prog);
}
}  // namespace pkv
