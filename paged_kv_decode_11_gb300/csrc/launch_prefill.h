// launch_prefill.h — host-side parameter block and launchers of the causal
// chunked prefill (not part of the public ABI).
#pragma once
#include "launch.h"

namespace pkv {

struct PrefillParams {
  void* out;
  const void* q;
  const int32_t* block_tables;
  const int32_t* seq_lens;
  const int32_t* cu_q_lens;
  const float* k_scales;
  const float* v_scales;
  float* out_lse;
  unsigned int* err;
  int num_seqs, Hq, Hkv, G, max_blocks, num_blocks, max_q_len, q_tile;
  int q_rows;                 // rows of q and out; a chunk outside them is flagged
  int ppb_shift;              // log2(block_size / 16)
  float qk_scale_log2;
};

// Each launcher validates nothing (the entry points do) and returns
// PKV_ERR_CUDA on a launch failure.
pkv_status launch_prefill(const PrefillParams& p, int head_dim, pkv_dtype q_dtype,
                          pkv_dtype kv_dtype, const CUtensorMap& tmK, const CUtensorMap& tmV,
                          cudaStream_t stream);

// Causal chunked prefill on the fifth-generation tensor cores (16-bit caches
// at head_dim 64, 128 or 256; E4M3 caches at 64 or 128); the other cases take
// launch_prefill. may_split: the grid may pair two CTAs per query tile (a
// cluster splitting its keys) when one CTA per tile would leave more than
// half of the SMs idle.
bool prefill_tc_supported(int head_dim, pkv_dtype kv_dtype);
// query rows of one tensor-core prefill tile (the M of its MMAs): q_tile =
// kPrefillTcRows / G tokens, each with the G query heads of one KV head
constexpr int kPrefillTcRows = 128;
// tmQ: the queries as {D, Hq, rows of q} (16-bit q with a 16-bit cache; unused
// with an E4M3 cache), one box the G heads of q_tile tokens by 64 elements
pkv_status launch_prefill_tc(const PrefillParams& p, int head_dim, pkv_dtype q_dtype,
                             pkv_dtype kv_dtype, const CUtensorMap& tmQ, const CUtensorMap& tmK,
                             const CUtensorMap& tmV, cudaStream_t stream, bool may_split);

// Rows of q handled by one prefill CTA for a GQA group size G.
int prefill_q_tile(int G);

}  // namespace pkv
