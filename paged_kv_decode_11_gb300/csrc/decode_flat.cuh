// decode_flat.cuh — paged-KV decode attention with a flat warp schedule, for
// caches whose blocks hold 16, 32 or 64 tokens (pages loaded by TMA).
//
// Follows "flash attention decode (online softmax, paged KV, GQA)" and
// "Split-KV paged attention for long context" (rvLLM: High-performance LLM
// inference in Rust, Kernel Compiler Stack; Tier 2: Hand-written CUDA
// kernels; FA3 v3 Attention Kernel, "split-KV ... distributes KV tiles across
// thread blocks") and the log-sum-exp merge of partial attention (rapid_llm
// README, feature table, "Decode context parallelism").
//
// Work decomposition. The batch's K/V is a sequence of units, one per
// (sequence b, KV head h), in the order u = b * Hkv + h; unit u holds the
// ceil(ctx_b / 16) pages of its context. Counting pages (automatic split) or
// partitions of `part` tokens (explicit split) as atoms, the atoms of all
// units form one flat range of NA atoms, cut into ranges. The grid is one
// wave of resident CTAs whose warps work independently: warp w streams range
// w, which holds kFlatStaticPct percent of its even share, then claims the
// next unclaimed chunk of the rest (about kFlatTailChunks chunks per warp)
// with an atomic counter, so the warps that run faster (the speed of warps in
// one SM differs by tens of percent) take more of the tail and all finish
// together; a small batch is split evenly with no claims. A warp
// keeps its own NST-deep ring of TMA loads (K page + V page per stage,
// completion on an mbarrier) and looks the page rows up 32 pages ahead, one
// page per lane; it claims and looks up its next range before the current
// one ends, so the ring runs on across ranges. The GQA group's query heads
// sit in the MMA N dimension (decode_frags.cuh), so each K/V byte is read
// from HBM once per call.
//
// A warp's run of pages inside one unit and one range (automatic split), or
// inside one partition (explicit split), is a segment, reduced with an online
// softmax in the log2 domain. A unit that is one segment is written out
// directly. Otherwise each segment writes its normalised output and
// log2-sum-exp to a workspace slot and bumps the unit's counter; the warp
// whose bump completes the count merges the unit's slots (after its own
// pages, so its stream does not pause):
//   LSE = log2 sum_s 2^{lse_s},  out = v_scale * sum_s 2^{lse_s - LSE} o_s.
// Slots: in the automatic split, unit u's segment in range v takes slot u + v
// (unique, because range boundaries grow with v, so ranges and units advance
// together); in the explicit split
// partition p of unit u takes slot u * max_parts + p. Either way a unit's n
// slots are consecutive. Units of more than kMergeGroup slots merge in two
// levels: each group of kMergeGroup slots is merged, by the warp completing
// it, into the group's first slot, and the warp completing the last group
// merges the groups. Every counter (and the range claims) is set back to zero
// by the warp that completes it, so a workspace zero-filled once stays ready
// across calls and CUDA-graph replays.
#pragma once
#include <cuda.h>
#include "decode_frags.cuh"
#include "launch.h"

namespace pkv {

template <int D, int KV, int NW, int NST>
struct FlatCfg {
  using Geo = PageGeom<D, KV>;
  static constexpr int STAGE_BYTES = 2 * Geo::PAGE_BYTES;
  static constexpr int SMEM_BYTES = 1024 + NW * NST * STAGE_BYTES;
};

// Units a warp holds back to merge after its own pages (more are merged at once).
constexpr int kFlatPending = 8;

// A position in the flat page stream: page `pg` of unit (b, h), whose context
// holds `ctx` tokens in `npg` pages; `rbase` is the flat index of the unit's
// first atom minus the first atom of the range being walked.
struct FlatPos {
  int b, h, pg, npg, ctx, rbase;
};

// Page lookups of one range, a window of 32 positions at a time.
struct FlatWin {
  int raw_id[32];               // block-table entries (landing by cp.async)
  int raw_hs[32];               // h << 3 | page in block, -1 past the range
  FlatPos look;                 // position of the window's next first page
  int left;                     // pages of the range from `look` on
};

// Slots a warp still has to merge, once its own pages are done: n slots from
// s0, `stride` apart, of unit (b, h). ng == 0: the unit's last merge, into
// its output rows. ng > 0: a first-level group, merged into slot s0, after
// which the unit's counter of merged groups is bumped (ng groups in all).
struct PendingMerge {
  int b, h, n, stride, ng;
  long long s0, su;             // su: the unit's first slot
};

// Per-warp state that is touched rarely (kept out of registers).
struct FlatWarpState {
  int z[32];                    // current range: page rows of positions [wstart, +32)
  int nz[32];                   // next range: page rows of its positions [0, 32)
  FlatWin win[2];               // [cw]: current range, [cw ^ 1]: next range
  FlatPos nstart;               // next range: first position
  int nv;                       // next range: index; -1 none left, -2 not claimed yet
  int nnpg, npub;               // next range: pages; first window published into nz
  int cw, wstart, vcur;         // current range: lookup slot, window start, index
  long long x0cur;              // current range: first atom
  long long ks, kd, xd0, na;    // atoms per static range and per claimed chunk; first
                                // atom of the claimed chunks; atoms of the batch
  int V, Wst;                   // ranges; ranges handed out statically (one per warp)
  PendingMerge pend[kFlatPending];
  int npend;
  // the unit being streamed: (b, h), its pages and context, its first atom
  // relative to the range's, and where it entered the current range (ring
  // position kks, page pgs)
  int cb, ch, cnpg, cctx, crbase, ckks, cpgs;
};



// Range v: the static ranges 0 .. Wst-1 (ks atoms each), then the claimed
// chunks (kd atoms each) from atom xd0 on.
__device__ __forceinline__ long long range_start(const FlatWarpState& ws, long long v) {
  return v < ws.Wst ? v * ws.ks : ws.xd0 + (v - ws.Wst) * ws.kd;
}
__device__ __forceinline__ long long range_atoms(const FlatWarpState& ws, long long v) {
  return min(v < ws.Wst ? ws.ks : ws.kd, ws.na - range_start(ws, v));
}
// The range holding atom a.
__device__ __forceinline__ long long range_of(const FlatWarpState& ws, long long a) {
  return a < ws.xd0 ? a / ws.ks : ws.Wst + (a - ws.xd0) / ws.kd;
}

__device__ __forceinline__ int flat_ctx(const DecodeParams& p, int b) {
  const int ctx = p.seq_lens[b];
  return ctx < 0 ? 0 : (ctx > p.cap ? p.cap : ctx);
}
__device__ __forceinline__ int pages_of(int ctx) { return (ctx + kBS - 1) / kBS; }
__device__ __forceinline__ int atoms_of(const DecodeParams& p, int npg) {
  return p.ppp ? (npg + p.ppp - 1) / p.ppp : npg;
}

// Moves q forward by n >= 0 pages, across units (empty contexts have no
// pages and are stepped over).
__device__ __forceinline__ void flat_advance(const DecodeParams& p, FlatPos& q, int n) {
  int rem = q.pg + n;
  while (q.b < p.B && rem >= q.npg) {
    rem -= q.npg;
    q.rbase += atoms_of(p, q.npg);
    if (++q.h == p.Hkv) {
      q.h = 0;
      do {
        ++q.b;
        q.ctx = q.b < p.B ? flat_ctx(p, q.b) : 0;
        q.npg = pages_of(q.ctx);
      } while (q.b < p.B && q.npg == 0);
    }
  }
  q.pg = rem;
}

__device__ __forceinline__ FlatPos shfl_pos(const FlatPos& q, int src) {
  FlatPos r;
  r.b = __shfl_sync(0xffffffffu, q.b, src);
  r.h = __shfl_sync(0xffffffffu, q.h, src);
  r.pg = __shfl_sync(0xffffffffu, q.pg, src);
  r.npg = __shfl_sync(0xffffffffu, q.npg, src);
  r.ctx = __shfl_sync(0xffffffffu, q.ctx, src);
  r.rbase = __shfl_sync(0xffffffffu, q.rbase, src);
  return r;
}

// The position of flat atom x (x < NA), found by the whole warp with a
// prefix sum over the sequences' atom counts; rbase is relative to x.
__device__ __forceinline__ FlatPos flat_locate(const DecodeParams& p, long long x, int lane) {
  FlatPos r{};
  long long before = 0;                                  // atoms per KV head before b0
  for (int b0 = 0; b0 < p.B; b0 += 32) {
    const int b = b0 + lane;
    const int ctx = b < p.B ? flat_ctx(p, b) : 0;
    const int npg = pages_of(ctx);
    const long long a = atoms_of(p, npg);
    long long incl = a;
#pragma unroll
    for (int o = 1; o < 32; o <<= 1) {
      const long long t = __shfl_up_sync(0xffffffffu, incl, o);
      if (lane >= o) incl += t;
    }
    const long long start = (before + incl - a) * p.Hkv;       // flat atom of (b, 0, page 0)
    const unsigned hit = __ballot_sync(0xffffffffu, b < p.B && (before + incl) * p.Hkv > x);
    if (hit) {
      const long long off = x - start;                          // meaningful in the hit lane
      const long long ha = a > 0 ? off / a : 0;
      const long long j = a > 0 ? off - ha * a : 0;
      FlatPos q;
      q.b = b;
      q.h = (int)ha;
      q.pg = (int)(p.ppp ? j * p.ppp : j);
      q.npg = npg;
      q.ctx = ctx;
      q.rbase = (int)(start + ha * a - x);                      // <= 0
      r = shfl_pos(q, __ffs(hit) - 1);
      break;
    }
    before += __shfl_sync(0xffffffffu, incl, 31);
  }
  return r;
}

// Pages of the natoms atoms that start at q (same value in every lane).
__device__ __forceinline__ int flat_range_pages(const DecodeParams& p, FlatPos q, long long natoms) {
  if (!p.ppp) return (int)natoms;
  int pages = 0;
  for (long long a = 0; a < natoms; ++a) {
    const int n = min(p.ppp, q.npg - q.pg);              // a partition, or a unit's last one
    pages += n;
    flat_advance(p, q, n);
  }
  return pages;
}

// Looks up the next 32 positions of a range: lane i copies the block-table
// entry of position look + i asynchronously into w.raw_id[i] (nothing waits
// for it here) and packs (head, page in block) into w.raw_hs[i], -1 past the
// range. Also prefetches into L1 the query rows of every unit whose first page
// lies in the window, so the switch to that unit finds them close.
template <int D>
__device__ __forceinline__ void flat_window(const DecodeParams& p, FlatWin& w, int lane) {
  const int left = w.left;
  FlatPos q = w.look;
  int hsub = -1;
  if (lane < left) {
    flat_advance(p, q, lane);
    cp_async4(&w.raw_id[lane], p.block_tables + (int64_t)q.b * p.max_blocks +
                                   (q.pg >> p.ppb_shift));
    hsub = (q.h << 3) | (q.pg & ((1 << p.ppb_shift) - 1));
    if (q.pg == 0) {
      const char* qrow =
          static_cast<const char*>(p.q) + ((int64_t)q.b * p.Hq + q.h * p.G) * D * 2;
      for (int o = 0; o < p.G * D * 2; o += 128)
        asm volatile("prefetch.global.L1 [%0];" ::"l"(qrow + o));
    }
  }
  w.raw_hs[lane] = hsub;
  if (lane == 31 && left > 32) flat_advance(p, q, 1);   // position look + 32
  const FlatPos nl = shfl_pos(q, 31);
  __syncwarp();
  if (lane == 0) {
    if (left > 32) w.look = nl;
    w.left = max(0, left - 32);
  }
  __syncwarp();
}

// Makes a looked-up window usable: each lane turns its raw entry into the page
// row of the tensor maps (a block of 16 << ppb_shift tokens holds that many
// consecutive 16-token pages per KV head) in z[lane], -1 past the range. A
// block id outside the pool is flagged and replaced by block 0.
__device__ __forceinline__ void flat_publish(const DecodeParams& p, FlatWin& w, int* z,
                                             int lane) {
  cp_async_wait_all();
  const int hsub = w.raw_hs[lane];
  int row = -1;
  if (hsub >= 0) {
    int id = w.raw_id[lane];
    if (id < 0 || id >= p.num_blocks) {
      atomicOr(p.err, PKV_DEVERR_BLOCK_ID);
      id = 0;
    }
    row = ((id * p.Hkv + (hsub >> 3)) << p.ppb_shift) + (hsub & 7);
  }
  __syncwarp();
  z[lane] = row;
  __syncwarp();
}

// Output rows (b, 0 .. Hq-1) of an empty context: zeros, log-sum-exp -inf.
template <int D>
__device__ __forceinline__ void write_empty_seq(const DecodeParams& p, int b, int lane) {
  uint4* o = reinterpret_cast<uint4*>(static_cast<uint16_t*>(p.out) + (int64_t)b * p.Hq * D);
  for (int i = lane; i < p.Hq * D / 8; i += 32) o[i] = make_uint4(0u, 0u, 0u, 0u);
  if (p.out_lse != nullptr)
    for (int i = lane; i < p.Hq; i += 32) p.out_lse[(int64_t)b * p.Hq + i] = -INFINITY;
}

// What a merge reads and writes (passed by value: taking the address of the
// kernel's parameter block would move every read of it to local memory).
struct MergeArgs {
  float* ws_o;
  float* ws_lse;
  void* out;
  float* out_lse;
  unsigned long long* done;
  unsigned int* err;
  const float* v_scales;        // E4M3 caches; null otherwise
  int G, Hq, Hkv;
};

template <int KV>
__device__ __forceinline__ MergeArgs merge_args(const DecodeParams& p) {
  return MergeArgs{p.ws_o, p.ws_lse, p.out, p.out_lse, p.done, p.err,
                   KV == KV_E4M3 ? p.v_scales : nullptr, p.G, p.Hq, p.Hkv};
}

// Merges n slots s0, s0 + stride, ... by log-sum-exp. dst < 0: into the
// output rows of unit (b, h) (times vscale, the unit's V scale for an E4M3
// cache, else 1); dst >= 0: into slot dst (normalised output and
// log2-sum-exp, the slot format). Each lane owns D/32 dims of every head;
// heads go four at a time. The weights are found first (lane s holds slot
// s's), so the slot rows of four slots are in flight at once.
template <int D, bool QBF16>
__device__ __noinline__ void flat_merge(const MergeArgs a, long long s0, int n, int stride,
                                        long long dst, int b, int h, float vscale, int lane) {
  constexpr int PER = D / 32;
  const int G = a.G;
  const int64_t row0 = (int64_t)b * a.Hq + h * G;
  for (int h0 = 0; h0 < G; h0 += 4) {
    const int nh = min(4, G - h0);
    float mx[4], z[4], acc[4][PER];
#pragma unroll
    for (int j = 0; j < 4; ++j) {
      mx[j] = -INFINITY;
      z[j] = 0.f;
#pragma unroll
      for (int i = 0; i < PER; ++i) acc[j][i] = 0.f;
    }
    // the largest log2-sum-exp of each head
    for (int base = 0; base < n; base += 32) {
      const int s = base + lane;
      if (s < n)
#pragma unroll
        for (int j = 0; j < 4; ++j)
          if (j < nh)
            mx[j] = fmaxf(mx[j], ldcg_f32(a.ws_lse + (s0 + (long long)s * stride) * G + h0 + j));
    }
#pragma unroll
    for (int j = 0; j < 4; ++j)
#pragma unroll
      for (int o = 16; o > 0; o >>= 1) mx[j] = fmaxf(mx[j], __shfl_xor_sync(0xffffffffu, mx[j], o));
    for (int base = 0; base < n; base += 32) {
      const int cnt = min(32, n - base);
      const int s = base + lane;
      float w[4];
#pragma unroll
      for (int j = 0; j < 4; ++j) {
        w[j] = 0.f;
        if (s < n && j < nh) {
          const float ls = ldcg_f32(a.ws_lse + (s0 + (long long)s * stride) * G + h0 + j);
          w[j] = (ls == -INFINITY || mx[j] == -INFINITY) ? 0.f : exp2f(ls - mx[j]);
        }
        z[j] += w[j];
      }
      for (int t = 0; t < cnt; t += 4) {
#pragma unroll
        for (int tt = 0; tt < 4; ++tt) {
          if (t + tt >= cnt) break;
          const long long slot = s0 + (long long)(base + t + tt) * stride;
#pragma unroll
          for (int j = 0; j < 4; ++j) {
            const float wt = __shfl_sync(0xffffffffu, w[j], t + tt);
            if (j >= nh) continue;
            const float* o = a.ws_o + (slot * G + h0 + j) * D + lane * PER;
            if constexpr (PER % 4 == 0) {
#pragma unroll
              for (int v4 = 0; v4 < PER / 4; ++v4) {
                const float4 v = __ldcg(reinterpret_cast<const float4*>(o) + v4);
                acc[j][4 * v4] += wt * v.x;
                acc[j][4 * v4 + 1] += wt * v.y;
                acc[j][4 * v4 + 2] += wt * v.z;
                acc[j][4 * v4 + 3] += wt * v.w;
              }
            } else {
              const float2 v = __ldcg(reinterpret_cast<const float2*>(o));
              acc[j][0] += wt * v.x;
              acc[j][1] += wt * v.y;
            }
          }
        }
      }
    }
#pragma unroll
    for (int j = 0; j < 4; ++j)
#pragma unroll
      for (int o = 16; o > 0; o >>= 1) z[j] += __shfl_xor_sync(0xffffffffu, z[j], o);
    __syncwarp();                                        // every read before an in-place write
#pragma unroll
    for (int j = 0; j < 4; ++j) {
      if (j >= nh) continue;
      const float lse = z[j] > 0.f ? mx[j] + log2f(z[j]) : -INFINITY;
      if (dst < 0) {
        const float inv = z[j] > 0.f ? vscale / z[j] : 0.f;
        uint32_t* d = reinterpret_cast<uint32_t*>(static_cast<uint16_t*>(a.out) +
                                                  (row0 + h0 + j) * D + lane * PER);
#pragma unroll
        for (int i = 0; i < PER / 2; ++i)
          d[i] = pack2<QBF16>(acc[j][2 * i] * inv, acc[j][2 * i + 1] * inv);
        if (lane == 0 && a.out_lse != nullptr) a.out_lse[row0 + h0 + j] = lse * kLn2;
      } else {
        const float inv = z[j] > 0.f ? 1.f / z[j] : 0.f;
        float* d = a.ws_o + (dst * G + h0 + j) * D + lane * PER;
#pragma unroll
        for (int i = 0; i < PER; ++i) d[i] = acc[j][i] * inv;
        if (lane == 0) a.ws_lse[dst * G + h0 + j] = lse;
      }
    }
  }
}

// One lane bumps a counter (after the warp barrier) with release semantics,
// publishing every lane's earlier writes, and acquire semantics, so reads
// after the next warp barrier see every write released by earlier bumps.
// Returns the count before the bump in every lane; when the bump completes
// the count (reaches `target`) the counter is set back to zero. A count at or
// past the target means the counters did not start at zero.
__device__ __forceinline__ unsigned long long bump(unsigned long long* ctr,
                                                   unsigned long long target,
                                                   unsigned int* err, int lane) {
  __syncwarp();
  unsigned long long before = 0ull;
  if (lane == 0) {
    before = atom_add_acq_rel_gpu(ctr, 1ull);
    if (before >= target) atomicOr(err, PKV_DEVERR_COUNTER);
    if (before + 1 == target) *ctr = 0ull;
  }
  before = __shfl_sync(0xffffffffu, before, 0);
  __syncwarp();
  return before;
}

// Runs one pending merge. A first-level group is merged into its first slot,
// then the unit's counter of merged groups is bumped; the warp completing
// that count merges the groups (kMergeGroup slots apart from the unit's first
// slot) into the output rows.
template <int D, bool QBF16>
__device__ __noinline__ void flat_pending(const MergeArgs a, const PendingMerge pm, int lane) {
  const float vs = a.v_scales != nullptr ? a.v_scales[pm.h] : 1.f;
  if (pm.ng == 0) {
    flat_merge<D, QBF16>(a, pm.s0, pm.n, pm.stride, -1, pm.b, pm.h, vs, lane);
    return;
  }
  flat_merge<D, QBF16>(a, pm.s0, pm.n, 1, pm.s0, pm.b, pm.h, vs, lane);
  const long long u = (long long)pm.b * a.Hkv + pm.h;
  if (bump(a.done + u, pm.ng, a.err, lane) + 1 == (unsigned long long)pm.ng)
    flat_merge<D, QBF16>(a, pm.su, pm.ng, kMergeGroup, -1, pm.b, pm.h, vs, lane);
}

// Resident CTAs per SM the kernel is built for (registers capped to allow it).
template <int D, int KV, int NT>
constexpr int flat_min_blocks() {
  return (KV == KV_E4M3 && D <= 128 && NT == 1) ? 4 : 1;
}

template <int D, int KV, bool QBF16, int NT, int NW, int NST>
__global__ void __launch_bounds__(NW * 32, (flat_min_blocks<D, KV, NT>()))
    decode_flat_kernel(const __grid_constant__ CUtensorMap tmK,
                       const __grid_constant__ CUtensorMap tmV, const DecodeParams p) {
  using Geo = PageGeom<D, KV>;
  constexpr int STAGE = FlatCfg<D, KV, NW, NST>::STAGE_BYTES;
  extern __shared__ uint8_t smem_raw[];
  __shared__ uint64_t bars[NW][NST];
  __shared__ FlatWarpState wstate[NW];

  const int lane = threadIdx.x & 31, warp = threadIdx.x >> 5;
  const int g = lane >> 2, c = lane & 3;
  const int gw = blockIdx.x * NW + warp;
  const int W = gridDim.x * NW;
  const int G = p.G;
  FlatWarpState& ws = wstate[warp];
  // launched as a programmatic dependent: the CTA is resident early, and
  // reads nothing before the kernel ahead of it (the cache write) is done
  if (p.wait_prior) griddep_wait();

  // ---- 1. the batch's atom count; bad lengths are flagged (and clamped), the
  // rows of empty contexts written out by one warp each -----------------------------
  long long na = 0;
  for (int b0 = 0; b0 < p.B; b0 += 32) {
    const int b = b0 + lane;
    int ctx = 0;
    if (b < p.B) {
      const int raw = p.seq_lens[b];
      if ((raw < 0 || raw > p.cap) && gw == 0) atomicOr(p.err, PKV_DEVERR_SEQ_LEN);
      ctx = raw < 0 ? 0 : min(raw, p.cap);
    }
    na += __reduce_add_sync(0xffffffffu, (unsigned)atoms_of(p, pages_of(ctx)));
    unsigned empty = __ballot_sync(0xffffffffu, b < p.B && ctx == 0);
    while (empty) {
      const int be = b0 + __ffs(empty) - 1;
      empty &= empty - 1;
      if (be % W == gw) write_empty_seq<D>(p, be, lane);
    }
  }
  na *= p.Hkv;
  // the split: an even static share of kFlatStaticPct percent per warp and
  // claimed chunks for the rest; below 4 x kFlatMinPages pages (one partition
  // in the explicit split) per warp, even ranges and no claims
  const long long per = na / W;
  const long long amin = p.ppp ? 1 : p.min_atoms;
  long long ks, kd;
  int Wst, V;
  if (per < (p.ppp ? 1 : 4 * amin)) {
    ks = kd = max((na + W - 1) / W, amin);
    Wst = V = (int)((na + ks - 1) / ks);
  } else {
    ks = max(per * kFlatStaticPct / 100, 1LL);
    const long long rest = na - ks * W;
    kd = max((rest + (long long)kFlatTailChunks * W - 1) / ((long long)kFlatTailChunks * W), amin);
    Wst = W;
    V = W + (int)((rest + kd - 1) / kd);
  }
  if (gw >= Wst) return;                                  // nothing for this warp

  // ---- 2. the first range (this warp's own), its lookups and its ring --------------
  const uint32_t raw_base = smem_u32(smem_raw);
  const uint32_t base = (raw_base + 1023u) & ~1023u;
  uint8_t* wbasep = smem_raw + (base - raw_base) + warp * NST * STAGE;
  const uint32_t wbase = base + warp * NST * STAGE;
  FlatPos cur = flat_locate(p, (long long)gw * ks, lane);
  const int rn0 = flat_range_pages(p, cur, min(ks, na - (long long)gw * ks));
  if (lane == 0) {
    prefetch_tensormap(&tmK);
    prefetch_tensormap(&tmV);
#pragma unroll
    for (int s = 0; s < NST; ++s) mbar_init(&bars[warp][s], 1);
    fence_barrier_init();
    ws.ks = ks;
    ws.kd = kd;
    ws.xd0 = (long long)Wst * ks;
    ws.na = na;
    ws.V = V;
    ws.Wst = Wst;
    ws.cw = 0;
    ws.wstart = 0;
    ws.vcur = gw;
    ws.x0cur = (long long)gw * ks;
    ws.nv = V > Wst ? -2 : -1;
    ws.npub = 0;
    ws.npend = 0;
    ws.win[0].look = cur;
    ws.win[0].left = rn0;
  }
  __syncwarp();
  flat_window<D>(p, ws.win[0], lane);
  flat_publish(p, ws.win[0], ws.z, lane);
  flat_window<D>(p, ws.win[0], lane);

  // Claims the next range (the whole warp): index, first position, pages, and
  // its first window of lookups (published later, when its loads have landed).
  auto claim_next = [&]() {
    unsigned long long cl = 0ull;
    if (lane == 0) cl = atomicAdd(p.claims, 1ull);
    cl = __shfl_sync(0xffffffffu, cl, 0);
    const long long v = (long long)ws.Wst + (long long)cl;
    if (v >= ws.V) {
      // a claim past the last range: this warp is done claiming. A claim
      // number past the ranges handed out means the counter did not start at
      // zero. The last warp to get here sets both claim counters back to zero.
      __syncwarp();
      if (lane == 0) {
        if (v >= (long long)ws.V + ws.Wst) atomicOr(p.err, PKV_DEVERR_COUNTER);
        const unsigned long long done = atomicAdd(p.claims + 1, 1ull);
        if (done + 1 == (unsigned long long)ws.Wst) {
          p.claims[0] = 0ull;
          p.claims[1] = 0ull;
        }
        ws.nv = -1;
      }
      __syncwarp();
      return;
    }
    const long long x = range_start(ws, v);
    const FlatPos st = flat_locate(p, x, lane);
    const int npg = flat_range_pages(p, st, range_atoms(ws, v));
    FlatWin& w = ws.win[ws.cw ^ 1];
    __syncwarp();
    if (lane == 0) {
      ws.nv = (int)v;
      ws.nstart = st;
      ws.nnpg = npg;
      ws.npub = 0;
      w.look = st;
      w.left = npg;
    }
    __syncwarp();
    flat_window<D>(p, w, lane);
  };
  // a short first range: look up the next one at once
  if (ws.nv == -2 && rn0 <= 32 + NST) claim_next();
  if (ws.nv >= 0 && rn0 <= NST) {
    flat_publish(p, ws.win[ws.cw ^ 1], ws.nz, lane);
    if (lane == 0) ws.npub = 1;
    __syncwarp();
  }

  // ring positions are numbered over all of this warp's ranges: position j
  // uses stage j % NST; rb and rend are the current range's first and
  // one-past-last positions
  int rb = 0, rend = rn0, nxt = 0;
  // Issues every position up to `limit` that is looked up (the current range's
  // window, or the next range's first window once it is published).
  auto top_up = [&](int limit) {
    while (nxt <= limit) {
      int z;
      if (nxt < rend) {
        z = ws.z[(nxt - rb) & 31];
      } else {
        const int jn = nxt - rend;
        if (ws.nv < 0 || !ws.npub || jn >= min(32, ws.nnpg)) break;
        z = ws.nz[jn];
      }
      if (lane == 0) {
        const int st = nxt % NST;
        uint64_t* bar = &bars[warp][st];
        uint8_t* dst = wbasep + st * STAGE;
        // KV pages are read once per call: mark them first to go from L2, so
        // they do not push out what is reused (block tables, queries, partials)
        const uint64_t evict_first = policy_evict_first();
        fence_proxy_async_smem();   // the warp's reads of this stage come first
        mbar_arrive_expect_tx(bar, STAGE);
#pragma unroll
        for (int bx = 0; bx < Geo::NBOX; ++bx) {
          tma_load_3d_hint(dst + bx * Geo::BOX_BYTES, &tmK, bar, bx * Geo::BOX_ELEMS, 0, z,
                           evict_first);
          tma_load_3d_hint(dst + Geo::PAGE_BYTES + bx * Geo::BOX_BYTES, &tmV, bar,
                           bx * Geo::BOX_ELEMS, 0, z, evict_first);
        }
      }
      ++nxt;
    }
  };
  top_up(NST - 1);

  // ---- 3. stream the pages: online softmax per segment ---------------------------
  uint32_t qf[NT][D / 16][2];
  float sl2 = 0.f;
  float oacc[NT][D / 16][4];
  float m[NT][2], l[NT][2];
  auto reset = [&]() {
#pragma unroll
    for (int nt = 0; nt < NT; ++nt) {
#pragma unroll
      for (int t = 0; t < D / 16; ++t)
        oacc[nt][t][0] = oacc[nt][t][1] = oacc[nt][t][2] = oacc[nt][t][3] = 0.f;
      m[nt][0] = m[nt][1] = -INFINITY;
      l[nt][0] = l[nt][1] = 0.f;
    }
  };
  reset();
  const int tk0 = st_row_token<KV>(g, 0), tk8 = st_row_token<KV>(g, 1);
  // the query group of unit (b, h) (prefetched into L1 when its first page was
  // looked up); q is scaled by 2^-qshift for the f16 MMAs of an E4M3 cache and
  // the scores are scaled back (exact)
  auto load_unit_q = [&](int b, int h) {
    int qshift;
    const uint16_t* qb = static_cast<const uint16_t*>(p.q) + ((int64_t)b * p.Hq + h * G) * D;
    load_qT_frags<D, KV, QBF16, NT>(qf, qb, G, lane, qshift);
    sl2 = p.qk_scale_log2 * (KV == KV_E4M3 ? p.k_scales[h] : 1.f) * pow2f(qshift);
  };

  // Per-page bookkeeping is reduced to one comparison: `evt` is the next ring
  // position at which something happens (a segment ends, the lookup window
  // slides, the next range is claimed or its lookups published). uend is the
  // position of the current unit's last page in this range and lastv the
  // tokens of that page.
  int uend = 0, lastv = kBS, segk = 0, evt = 0;
  // Enters unit position q at ring position kst: the unit's bookkeeping.
  auto enter_unit = [&](const FlatPos& q, int kst) {
    const int in_range = min(q.npg - q.pg, rend - kst);
    uend = kst + in_range - 1;
    lastv = (q.npg - q.pg <= rend - kst) ? q.ctx - (q.npg - 1) * kBS : kBS;
    segk = p.ppp ? min(uend, kst + (p.ppp - q.pg % p.ppp) - 1) : uend;
    __syncwarp();
    if (lane == 0) {
      ws.cb = q.b;
      ws.ch = q.h;
      ws.cnpg = q.npg;
      ws.cctx = q.ctx;
      ws.crbase = q.rbase;
      ws.ckks = kst;
      ws.cpgs = q.pg;
    }
    __syncwarp();
  };
  // the next ring position with an event at or after kk + 1
  auto next_event = [&](int kk) {
    int e = segk;
    const int k1 = kk + 1;
    const int sl = rb + ws.wstart + 31 - NST;           // the window must slide here
    if (sl + 1 + NST < rend) e = min(e, max(sl, k1));
    const int nv = ws.nv;
    if (nv == -2) e = min(e, max(rend - 33 - NST, k1));
    if (nv >= 0 && !ws.npub) e = min(e, max(rend - 1 - NST, k1));
    return e;
  };
  load_unit_q(cur.b, cur.h);
  enter_unit(cur, 0);
  evt = next_event(-1);

  for (int kk = 0;; ++kk) {
    const int st = kk % NST;
    bool ok = mbar_wait_bounded(&bars[warp][st], (kk / NST) & 1);
    ok = __all_sync(0xffffffffu, ok);
    if (!ok) {
      if (lane == 0) atomicOr(p.err, PKV_DEVERR_TIMEOUT);
      // let what this warp may still have in flight land (each wait bounded;
      // a stage that was never issued just runs its wait out), then stop
      for (int kd = kk + 1; kd < kk + NST; ++kd)
        mbar_wait_bounded(&bars[warp][kd % NST], (kd / NST) & 1, 1u << 16);
      return;
    }
    const uint32_t kpage = wbase + st * STAGE;
    const uint32_t vpage = kpage + Geo::PAGE_BYTES;
    const int valid = kk == uend ? lastv : kBS;         // tokens of this page in the context
    if (valid < kBS) {
      // the last page of the context: its rows past the end get weight 0, and
      // whatever they hold must not turn that into NaN, so zero them in V
      zero_page_rows<D, KV>(wbasep + st * STAGE + Geo::PAGE_BYTES, valid, lane);
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
      top_up(kk + NST);
      kq_regs<D, NT>(s, qf, pr.k);
    } else {
      kq_page<D, KV, NT>(s, qf, kpage, lane);
    }

    // online softmax in the log2 domain, against a reference max per column
    // that moves only when the page's max outgrows it by kRefSlackLog2
    const bool v0 = tk0 < valid, v8 = tk8 < valid;
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
      top_up(kk + NST);
    }
    if (kk != evt) continue;

    // ---- events of this position --------------------------------------------------
    if (kk == segk) {
      // the end of a segment: this unit's last page in the range, or a
      // partition's last page
      const int cb = ws.cb, ch = ws.ch, cnpg = ws.cnpg, crbase = ws.crbase;
      const int pg = ws.cpgs + (kk - ws.ckks);          // this page
      float L[NT][2];
#pragma unroll
      for (int nt = 0; nt < NT; ++nt)
#pragma unroll
        for (int e = 0; e < 2; ++e) L[nt][e] = col_sum8(l[nt][e]);
      const long long u = (long long)cb * p.Hkv + ch;
      int n;
      long long s0, slot;
      if (p.ppp) {
        n = atoms_of(p, cnpg);
        s0 = u * p.max_parts;
        slot = s0 + pg / p.ppp;
      } else {
        // ranges holding the unit's first and last atoms
        const long long a0 = ws.x0cur + crbase;
        const long long vf = range_of(ws, a0), vl = range_of(ws, a0 + cnpg - 1);
        n = (int)(vl - vf + 1);
        s0 = u + vf;
        slot = u + ws.vcur;
      }
      // the segment's normalised output and log2-sum-exp into its slot (a
      // unit of one segment too: its one-slot merge writes the output)
#pragma unroll
      for (int nt = 0; nt < NT; ++nt)
#pragma unroll
        for (int e = 0; e < 2; ++e) {
          const int hh = 8 * nt + 2 * c + e;
          if (hh < G) {
            const float inv = L[nt][e] > 0.f ? 1.f / L[nt][e] : 0.f;
            float* orow = p.ws_o + (slot * G + hh) * D;
#pragma unroll
            for (int t = 0; t < D / 16; ++t) {
              orow[ot_row_dim<D, KV>(t, g, 0)] = oacc[nt][t][e] * inv;
              orow[ot_row_dim<D, KV>(t, g, 1)] = oacc[nt][t][2 + e] * inv;
            }
            if (g == 0)
              p.ws_lse[slot * G + hh] = L[nt][e] > 0.f ? m[nt][e] + log2f(L[nt][e]) : -INFINITY;
          }
        }
      // the warp completing the unit (one level), or one of its groups of
      // kMergeGroup slots (two levels), merges them after its own pages
      PendingMerge pm{cb, ch, n, 1, 0, s0, s0};
      bool ready;
      if (n <= kMergeGroup) {
        ready = n == 1 || bump(p.done + u, n, p.err, lane) + 1 == (unsigned long long)n;
      } else {
        const int grp = (int)(slot - s0) / kMergeGroup;
        pm.n = min(kMergeGroup, n - grp * kMergeGroup);
        pm.s0 = s0 + (long long)grp * kMergeGroup;
        pm.ng = (n + kMergeGroup - 1) / kMergeGroup;
        ready = bump(p.done1 + pm.s0, pm.n, p.err, lane) + 1 == (unsigned long long)pm.n;
      }
      if (ready) {
        const int np = ws.npend;
        if (np < kFlatPending) {
          __syncwarp();
          if (lane == 0) {
            ws.pend[np] = pm;
            ws.npend = np + 1;
          }
          __syncwarp();
        } else {
          flat_pending<D, QBF16>(merge_args<KV>(p), pm, lane);
        }
      }
      reset();

      if (kk + 1 == rend) {
        // ---- on to the next range (claimed and looked up before now) --------------
        if (ws.nv == -2) claim_next();                   // (a range of a few pages)
        if (ws.nv < 0) break;
        if (!ws.npub) {
          flat_publish(p, ws.win[ws.cw ^ 1], ws.nz, lane);
          if (lane == 0) ws.npub = 1;
        }
        const int nz_lane = ws.nz[lane];
        const FlatPos ns = ws.nstart;
        const int nnpg = ws.nnpg, nv = ws.nv;
        __syncwarp();
        ws.z[lane] = nz_lane;
        if (lane == 0) {
          ws.cw ^= 1;
          ws.wstart = 0;
          ws.vcur = nv;
          ws.x0cur = range_start(ws, nv);
          ws.nv = -2;                          // every warp claims until a claim fails
          ws.npub = 0;
        }
        __syncwarp();
        rb = rend;
        rend = rb + nnpg;
        flat_window<D>(p, ws.win[ws.cw], lane);          // the new range's second window
        load_unit_q(ns.b, ns.h);
        enter_unit(ns, kk + 1);
        if (ws.nv == -2 && nnpg <= 32 + NST) claim_next();
        if (ws.nv >= 0 && nnpg <= NST) {
          flat_publish(p, ws.win[ws.cw ^ 1], ws.nz, lane);
          if (lane == 0) ws.npub = 1;
          __syncwarp();
        }
        top_up(kk + NST);
      } else if (kk == uend) {
        // the next unit of this range
        FlatPos q{cb, ch, cnpg - 1, cnpg, ws.cctx, crbase};
        flat_advance(p, q, 1);
        load_unit_q(q.b, q.h);
        enter_unit(q, kk + 1);
      } else {
        // the next partition of this unit (the query fragments were let go at
        // the segment's end, which leaves room for its epilogue)
        load_unit_q(cb, ch);
        segk = min(uend, kk + p.ppp);
      }
    }
    // the next top_up (to position kk + 1 + NST) must find its window current
    const int ws0 = ws.wstart;
    if (kk + 1 + NST < rend && kk + 1 + NST - rb >= ws0 + 32) {
      flat_publish(p, ws.win[ws.cw], ws.z, lane);
      if (lane == 0) ws.wstart = ws0 + 32;
      flat_window<D>(p, ws.win[ws.cw], lane);
    }
    // claim the next range in time, publish its first window once it is needed
    if (ws.nv == -2 && kk + 1 + 32 + NST >= rend) claim_next();
    if (ws.nv >= 0 && !ws.npub && kk + 1 + NST >= rend) {
      flat_publish(p, ws.win[ws.cw ^ 1], ws.nz, lane);
      if (lane == 0) ws.npub = 1;
      __syncwarp();
    }
    evt = next_event(kk);
  }
  // the merges this warp completed, done now that its pages are done
  const int np = ws.npend;
  for (int i = 0; i < np; ++i) flat_pending<D, QBF16>(merge_args<KV>(p), ws.pend[i], lane);
}

#ifndef PKV_DECODE_NST_E4M3
#define PKV_DECODE_NST_E4M3 3
#endif
#ifndef PKV_DECODE_NST_16
#define PKV_DECODE_NST_16 2
#endif

// One wave of resident CTAs (at most kDecodeWorkers per SM).
template <int D, int KV, bool QBF16, int NT>
static pkv_status launch_flat_t(const DecodeParams& p, const CUtensorMap& tmK,
                                const CUtensorMap& tmV, cudaStream_t stream, bool programmatic) {
  constexpr int NW = kDecodeWarps;
  constexpr int NST = (KV == KV_E4M3) ? PKV_DECODE_NST_E4M3 : PKV_DECODE_NST_16;
  using Cfg = FlatCfg<D, KV, NW, NST>;
  auto kern = decode_flat_kernel<D, KV, QBF16, NT, NW, NST>;
  int dev = 0;
  if (cudaGetDevice(&dev) != cudaSuccess || dev < 0 || dev >= 64) return PKV_ERR_CUDA;
  static std::atomic<int> grid_ctas[64];  // per device: SMs x resident CTAs per SM
  int ctas = grid_ctas[dev];
  if (ctas == 0) {
    if (cudaFuncSetAttribute(kern, cudaFuncAttributeMaxDynamicSharedMemorySize,
                             Cfg::SMEM_BYTES) != cudaSuccess)
      return PKV_ERR_CUDA;
    int occ = 0, sms = 0;
    if (cudaOccupancyMaxActiveBlocksPerMultiprocessor(&occ, kern, NW * 32, Cfg::SMEM_BYTES) !=
            cudaSuccess ||
        cudaDeviceGetAttribute(&sms, cudaDevAttrMultiProcessorCount, dev) != cudaSuccess ||
        occ < 1)
      return PKV_ERR_CUDA;
    ctas = sms * std::min(occ, kDecodeWorkers);
    grid_ctas[dev] = ctas;
  }
  if (programmatic) {
    cudaLaunchAttribute attr[1];
    attr[0].id = cudaLaunchAttributeProgrammaticStreamSerialization;
    attr[0].val.programmaticStreamSerializationAllowed = 1;
    cudaLaunchConfig_t cfg = {};
    cfg.gridDim = dim3(ctas);
    cfg.blockDim = dim3(NW * 32);
    cfg.dynamicSmemBytes = Cfg::SMEM_BYTES;
    cfg.stream = stream;
    cfg.attrs = attr;
    cfg.numAttrs = 1;
    return cudaLaunchKernelEx(&cfg, kern, tmK, tmV, p) == cudaSuccess ? PKV_OK : PKV_ERR_CUDA;
  }
  kern<<<ctas, NW * 32, Cfg::SMEM_BYTES, stream>>>(tmK, tmV, p);
  return cudaGetLastError() == cudaSuccess ? PKV_OK : PKV_ERR_CUDA;
}

template <int D, int KV, bool QBF16>
static pkv_status launch_flat_nt(const DecodeParams& p, const CUtensorMap& tmK,
                                 const CUtensorMap& tmV, cudaStream_t stream, bool prog) {
  if constexpr (D <= 128) {
    if (p.G > 8) return launch_flat_t<D, KV, QBF16, 2>(p, tmK, tmV, stream, prog);
  } else {
    if (p.G > 8) return PKV_ERR_UNSUPPORTED;        // 16 head columns at D = 256: not built
  }
  return launch_flat_t<D, KV, QBF16, 1>(p, tmK, tmV, stream, prog);
}

template <int D>
static pkv_status launch_flat_d(const DecodeParams& p, pkv_dtype q_dtype, pkv_dtype kv_dtype,
                                const CUtensorMap& tmK, const CUtensorMap& tmV,
                                cudaStream_t stream, bool prog) {
  const bool qbf = (q_dtype == PKV_BF16);
  if (kv_dtype == PKV_FP8_E4M3)
    return qbf ? launch_flat_nt<D, KV_E4M3, true>(p, tmK, tmV, stream, prog)
               : launch_flat_nt<D, KV_E4M3, false>(p, tmK, tmV, stream, prog);
  if (kv_dtype == PKV_BF16) return launch_flat_nt<D, KV_BF16, true>(p, tmK, tmV, stream, prog);
  return launch_flat_nt<D, KV_F16, false>(p, tmK, tmV, stream, prog);
}

}  // namespace pkv
