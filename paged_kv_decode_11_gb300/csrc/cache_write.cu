// cache_write.cu — reshape_and_cache: scatter the K/V rows of new tokens into
// their slots of the paged cache.
//
// Follows the cache-write half of "RoPE + KV cache write -- fused, no
// intermediate alloc" (rvLLM: High-performance LLM inference in Rust, Kernel
// Compiler Stack, decode step at c=128) and the FP8 KV cache of the Litellama
// page (Features, "FP8 KV Cache"): E4M3 codes with one fp32 scale per KV head.
//
// One thread moves 8 consecutive elements of one (token, head) row: a 16-byte
// load of the source and a 16-byte (16-bit cache) or 8-byte (E4M3 cache)
// store into block slot / 16, offset slot % 16 of that head's page. Rows of
// a warp are consecutive in the source, so loads are fully coalesced; stores
// are contiguous per row.
#include <cuda_fp16.h>
#include <cuda_bf16.h>
#include "common.cuh"
#include "kv_store.cuh"
#include "launch_cache.h"

namespace pkv {

template <bool SRC_BF16, bool TO_FP8>
__global__ void __launch_bounds__(256) cache_write_kernel(const CacheWriteParams p) {
  // a decode launched behind this kernel may become resident now; it waits
  // for this grid to finish before it reads anything
  if (threadIdx.x == 0) griddep_launch_dependents();
  const int chunks = p.D / 8;
  const int64_t total = (int64_t)p.num_tokens * p.Hkv * chunks;
  const int64_t i = (int64_t)blockIdx.x * blockDim.x + threadIdx.x;
  if (i >= total) return;
  const int ch = (int)(i % chunks);
  const int64_t row = i / chunks;                 // token * Hkv + head
  const int h = (int)(row % p.Hkv);
  const int64_t t = row / p.Hkv;
  const int64_t slot = p.slots[t];
  if (slot < 0) return;
  if (slot >= ((int64_t)p.num_blocks << p.bs_log2)) {
    if (h == 0 && ch == 0) atomicOr(p.err, PKV_DEVERR_SLOT);
    return;
  }
  const int64_t dst = cache_elem(slot, h, p.Hkv, p.D, ch * 8, p.bs_log2);
  const int64_t src = row * p.D + ch * 8;
  const uint4 kin = *reinterpret_cast<const uint4*>(static_cast<const uint16_t*>(p.key) + src);
  const uint4 vin = *reinterpret_cast<const uint4*>(static_cast<const uint16_t*>(p.value) + src);
  const float ks = TO_FP8 ? p.k_scales[h] : 1.f, vs = TO_FP8 ? p.v_scales[h] : 1.f;
  store_row8<SRC_BF16, TO_FP8>(p.k_cache, dst, kin, ks);
  store_row8<SRC_BF16, TO_FP8>(p.v_cache, dst, vin, vs);
}

pkv_status launch_cache_write(const CacheWriteParams& p, pkv_dtype src_dtype, pkv_dtype kv_dtype,
                              cudaStream_t stream) {
  const int64_t total = (int64_t)p.num_tokens * p.Hkv * (p.D / 8);
  if (total == 0) return PKV_OK;
  const int threads = 256;
  const int64_t blocks = (total + threads - 1) / threads;
  if (blocks > 0x7FFFFFFF) return PKV_ERR_INVALID_ARG;
  const bool sbf = (src_dtype == PKV_BF16);
  if (kv_dtype == PKV_FP8_E4M3) {
    if (sbf) cache_write_kernel<true, true><<<(unsigned)blocks, threads, 0, stream>>>(p);
    else cache_write_kernel<false, true><<<(unsigned)blocks, threads, 0, stream>>>(p);
  } else {
    cache_write_kernel<false, false><<<(unsigned)blocks, threads, 0, stream>>>(p);
  }
  return cudaGetLastError() == cudaSuccess ? PKV_OK : PKV_ERR_CUDA;
}

}  // namespace pkv
