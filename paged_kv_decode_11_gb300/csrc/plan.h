// plan.h — the split-KV plan of a decode call (host code): partition size,
// partitions per sequence and the workspace layout the decode kernels use.
#pragma once
#include <algorithm>
#include <cstddef>
#include <cstdint>
#include "launch.h"

namespace pkv {

inline size_t align256(size_t x) { return (x + 255) & ~size_t(255); }

// Split-KV plan of a decode call. With partition_tokens = 0 the partition
// is the smallest power of two from 512 to 2048 tokens that keeps the launch
// at about 3 waves of ctas_per_sm resident CTAs on every SM when contexts
// average half the maximum (below 512 tokens a CTA's start and merge cost
// more than the extra parallelism gives back); an explicit size is honoured
// as given. A larger ctas_per_sm never gives a longer partition, so the
// workspace planned with the default fits every plan.
// Workspace: [done counters B*Hkv u64 | partition outputs rows*D fp32 |
// partition log2-sum-exps rows fp32], each region 256-byte aligned, with
// rows = B * Hq * max_parts and max_parts = ceil(max_seq_len / partition).
struct DecodePlan {
  int part, max_parts;
  size_t off_done, off_o, off_lse, bytes;
};

inline DecodePlan plan_decode(int num_seqs, int num_q_heads, int num_kv_heads, int head_dim,
                              int max_seq_len, int partition_tokens, int sms,
                              int ctas_per_sm = kDecodeWorkers) {
  DecodePlan pl{};
  if (sms <= 0) sms = 148;
  if (partition_tokens > 0) {
    pl.part = partition_tokens;
  } else {
    const int64_t est = (int64_t)num_seqs * num_kv_heads * std::max(1, max_seq_len / 2);
    const int64_t target = (int64_t)sms * ctas_per_sm * 3;
    pl.part = 512;
    while (pl.part < 2048 && est / pl.part > target) pl.part *= 2;
  }
  pl.max_parts = std::max(1, (max_seq_len + pl.part - 1) / pl.part);
  const size_t units = (size_t)num_seqs * num_kv_heads;
  const size_t rows = (size_t)num_seqs * num_q_heads * (size_t)pl.max_parts;
  pl.off_done = 0;
  pl.off_o = align256(units * 8);
  pl.off_lse = pl.off_o + align256(rows * head_dim * sizeof(float));
  pl.bytes = pl.off_lse + align256(rows * sizeof(float));
  return pl;
}

// Whole-context decode: one CTA of kDecodeWideWarps warps per (sequence, KV
// head), its context one partition (no workspace partials, no cross-CTA
// merge), each warp keeping a deeper ring of pages in flight; the CTA takes an
// SM to itself. It pays when that grid is about one full wave: automatic
// partitions, pages loaded by TMA, head_dim <= 128, no other grid beside it
// (ctas_per_sm at the default), (sequence, KV head) units at most one per SM,
// and either short contexts (<= 512 tokens, where the split plan has one
// partition anyway and the extra warps shorten each warp's chain of pages) or
// at least 3/4 of the SMs busy with contexts of at most 4096 tokens (the
// longest context bounds the call, at one CTA's rate). The workspace the
// split plan sizes is always enough (this plan needs none of it).
inline bool wide_decode(int64_t units, int sms, int max_seq_len, int partition_tokens,
                        int bs_log2, int head_dim, int ctas_per_sm) {
  if (partition_tokens > 0 || bs_log2 < 4 || head_dim > 128 || ctas_per_sm != kDecodeWorkers ||
      sms <= 0 || units > sms)
    return false;
  if (max_seq_len <= 512) return true;
  return max_seq_len <= 4096 && units * 4 >= (int64_t)sms * 3;
}

// Longest-first CTA order (decode_item_full_first in decode_kernel.cuh), for
// decode planned beside a prefill grid (one resident CTA per SM) when
// contexts are split, pages are loaded by TMA and the batch is small enough
// for every CTA to rank its sequences. Measured on its own, decode loses with
// it (the equal full partitions it puts first start and end in step, so
// whole waves drain at once); beside the prefill it wins.
inline bool full_first_order(int num_seqs, int num_kv_heads, int grid_parts, int bs_log2,
                             int ctas_per_sm, bool wide) {
  return ctas_per_sm == 1 && !wide && grid_parts > 1 && bs_log2 >= 4 &&
         num_seqs <= kFullFirstMaxSeqs &&
         (int64_t)grid_parts * num_kv_heads * num_seqs < ((int64_t)1 << 31);
}

// Tokens of the partition each warp of a decode CTA reduces on its own, or 0.
// With an explicit partition size (blocks of 16 tokens or more, pages loaded
// by TMA) the kDecodeWarps warps of a CTA take consecutive partitions of one
// sequence, one each, so a CTA's start-up and its partial write are shared
// by kDecodeWarps partitions; otherwise the warps take the pages of the
// CTA's partition in turn.
inline int warp_partition_tokens(int partition_tokens, int bs_log2) {
  return (partition_tokens > 0 && bs_log2 >= 4 &&
          partition_tokens * kDecodeWarps <= kMaxPartitionTokens)
             ? partition_tokens : 0;
}

}  // namespace pkv
