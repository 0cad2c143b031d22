// plan.h — the split-KV plan of a decode call (host code): partition size,
// partitions per sequence and the workspace layout the decode kernels use.
#pragma once
#include <algorithm>
#include <cstddef>
#include <cstdint>
#include "launch.h"

namespace pkv {

inline size_t align256(size_t x) { return (x + 255) & ~size_t(255); }

// Split-KV plan of a decode call. With blocks of 16 tokens or more the flat
// warp schedule runs (decode_flat.cuh): an explicit partition size makes
// partitions of that many tokens the units of work, each written to its own
// slot; the automatic split cuts the batch's pages into equal runs, one per
// warp, so a unit's slots are at most one per warp. Blocks of fewer than 16
// tokens take the per-partition kernel, whose automatic partition is the
// smallest power of two from 512 to 2048 tokens that keeps the launch at
// about 3 waves of resident CTAs when contexts average half the maximum
// (below 512 tokens its per-CTA start and merge cost more than the extra
// parallelism gives back).
// Workspace: [range claims 2 u64 | done counters B*Hkv u64 | merge-group
// counters, one u64 per slot | slot outputs rows*D fp32 | slot log2-sum-exps
// rows fp32], each region 256-byte aligned, with slots = max(B*Hkv*max_parts,
// B*Hkv + ranges of a full grid) and rows = G * slots.
struct DecodePlan {
  int part, max_parts;
  size_t off_done, off_done1, off_o, off_lse, bytes;
};

inline DecodePlan plan_decode(int num_seqs, int num_q_heads, int num_kv_heads, int head_dim,
                       int max_seq_len, int partition_tokens, int sms) {
  DecodePlan pl{};
  if (sms <= 0) sms = 148;
  if (partition_tokens > 0) {
    pl.part = partition_tokens;
  } else {
    const int64_t est = (int64_t)num_seqs * num_kv_heads * std::max(1, max_seq_len / 2);
    const int64_t target = (int64_t)sms * kDecodeWorkers * 3;
    pl.part = 512;
    while (pl.part < 2048 && est / pl.part > target) pl.part *= 2;
  }
  pl.max_parts = std::max(1, (max_seq_len + pl.part - 1) / pl.part);
  const size_t units = (size_t)num_seqs * num_kv_heads;
  const size_t flat_slots =
      units + (size_t)sms * kDecodeWorkers * kDecodeWarps * kFlatRangesPerWarp;
  const size_t slots = std::max(units * (size_t)pl.max_parts, flat_slots);
  const size_t rows = slots * (size_t)(num_q_heads / num_kv_heads);
  pl.off_done = 256;
  pl.off_done1 = pl.off_done + align256(units * 8);
  pl.off_o = pl.off_done1 + align256(slots * 8);
  pl.off_lse = pl.off_o + align256(rows * head_dim * sizeof(float));
  pl.bytes = pl.off_lse + align256(rows * sizeof(float));
  return pl;
}

}  // namespace pkv
