// launch_cache.h — host-side parameter blocks and launchers of the cache
// writes: reshape_and_cache and the fused rotary embedding with it (not part
// of the public ABI).
#pragma once
#include "launch.h"

namespace pkv {

struct CacheWriteParams {
  const void* key;
  const void* value;
  void* k_cache;
  void* v_cache;
  const int64_t* slots;
  const float* k_scales;
  const float* v_scales;
  unsigned int* err;
  int num_tokens, Hkv, D, num_blocks;
  int bs_log2;                // log2(block_size)
};

struct RopeCacheParams {
  void* query;
  const void* key;
  const void* value;
  void* k_cache;
  void* v_cache;
  const int64_t* slots;
  const int64_t* positions;
  const float* cos_sin;
  const float* k_scales;
  const float* v_scales;
  unsigned int* err;
  int64_t max_position;
  int rot, neox, num_tokens, Hq, Hkv, D, num_blocks;
  int bs_log2;                // log2(block_size)
};

// Each launcher validates nothing (the entry points do) and returns
// PKV_ERR_CUDA on a launch failure.
pkv_status launch_cache_write(const CacheWriteParams& p, pkv_dtype src_dtype,
                              pkv_dtype kv_dtype, cudaStream_t stream);
pkv_status launch_rope_cache(const RopeCacheParams& p, pkv_dtype src_dtype, pkv_dtype kv_dtype,
                             cudaStream_t stream);

}  // namespace pkv
