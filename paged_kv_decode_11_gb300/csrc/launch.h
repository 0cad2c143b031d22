// launch.h — host-side parameter block and launchers of decode attention,
// and the constants its planner shares with the entry points (not part of
// the public ABI). launch_prefill.h and launch_cache.h hold those of the
// prefill and of the cache writes.
#pragma once
#include <cuda.h>
#include <cuda_runtime.h>
#include <atomic>
#include <cstdint>
#include "../../include/pkv.h"

namespace pkv {

constexpr int kMaxPartitionTokens = 8192;
// Largest partition of the gather path (it keeps one cache row per token in
// shared memory).
constexpr int kGatherMaxPartitionTokens = 2048;   // split-KV partition cap (block ids staged in smem)
constexpr int kDecodeWorkers = 4;           // resident decode CTAs per SM assumed by the planner
constexpr int kDecodeWarps = 4;             // warps per decode CTA
constexpr int kDecodeWideWarps = 8;         // warps per whole-context decode CTA
constexpr int kFullFirstMaxSeqs = 256;      // batches the full-first CTA order takes

struct DecodeParams {
  void* out;
  const void* q;
  const void* k_cache;        // read directly only by the gather instantiation
  const void* v_cache;
  const int32_t* block_tables;
  const int32_t* seq_lens;
  const float* k_scales;
  const float* v_scales;
  float* out_lse;
  unsigned long long* done;   // [B * Hkv] finished-partition counters (zero between calls)
  float* ws_o;                // [B * Hq, max_parts, D] fp32 partition outputs (normalised)
  float* ws_lse;              // [B * Hq, max_parts]    fp32 partition log2-sum-exp
  unsigned int* err;          // device error word
  int B, Hq, Hkv, G, max_blocks, num_blocks, max_seq_len;
  int ppb_shift;              // log2(block_size / 16): 16-token pages per block (TMA mode)
  int bs_log2;                // log2(block_size)
  int part, max_parts;        // CTA partition size (tokens) and workspace slots per sequence
  int wpart;                  // > 0: each warp of a CTA reduces its own partition of
                              // this many tokens (part = warps * wpart); 0: the warps
                              // take the CTA partition's pages round-robin
  int grid_parts;             // CTAs per (sequence, KV head) in the grid
  int wide;                   // (host routing) whole-context CTAs of kDecodeWideWarps warps
  int full_first;             // 1-D grid in full-first (longest-first) order of work items
  float qk_scale_log2;        // scale * log2(e)
  int wait_prior;             // wait for the grids ahead of it on the stream before reading
  // early start (per-partition kernel, TMA pages): the kernel ahead of it is
  // known to write nothing but the cache rows of each sequence's newest token
  // (the library's own cache write), so everything else is read, and every
  // other page is loaded, before the wait
  int early;
};

// Each launcher validates nothing (the entry points do) and returns
// PKV_ERR_CUDA on a launch failure.
// programmatic: launch as a programmatic dependent of the previous kernel on
// the stream (it may start once that kernel's CTAs have all signalled).
pkv_status launch_decode(const DecodeParams& p, int head_dim, pkv_dtype q_dtype,
                         pkv_dtype kv_dtype, const CUtensorMap& tmK, const CUtensorMap& tmV,
                         cudaStream_t stream, bool programmatic = false);
// Whole-context decode (p.wide): one CTA of kDecodeWideWarps warps per
// (sequence, KV head), head_dim 64 or 128, pages loaded by TMA.
pkv_status launch_decode_wide(const DecodeParams& p, int head_dim, pkv_dtype q_dtype,
                              pkv_dtype kv_dtype, const CUtensorMap& tmK, const CUtensorMap& tmV,
                              cudaStream_t stream, bool programmatic);
// Decode in full-first CTA order (p.full_first), pages loaded by TMA.
pkv_status launch_decode_full_first(const DecodeParams& p, int head_dim, pkv_dtype q_dtype,
                                    pkv_dtype kv_dtype, const CUtensorMap& tmK,
                                    const CUtensorMap& tmV, cudaStream_t stream,
                                    bool programmatic);
// Decode for blocks of fewer than 16 tokens (pages gathered row by row).
pkv_status launch_decode_gather(const DecodeParams& p, int head_dim, pkv_dtype q_dtype,
                                pkv_dtype kv_dtype, cudaStream_t stream, bool programmatic);

}  // namespace pkv
