// noalloc.cu — paged_attn_decode_noalloc: decode attention for callers that
// cannot hand the library a workspace.
//
// Some callers cannot allocate device memory when they call attention: a
// serving engine whose memory planner has already given the whole device to
// the weights and the KV pool (an extra allocation would fail or fragment
// it), a latency-critical loop where cudaMalloc / cudaFree would synchronise
// the device and stall other streams, or a plain C host that owns no
// allocator. This entry point needs no workspace from them: the split-KV
// scratch (partition counters and fp32 partial results) lives in one
// file-scope device array of PKV_NOALLOC_SCRATCH_BYTES, which every GPU that
// loads this library holds until the process exits. Nothing here calls
// cudaMalloc, cudaFree or any allocating routine.
#include <cuda_runtime.h>
#include <cstdint>
#include <mutex>

#pragma GCC visibility push(default)
#include "../../include/pkv.h"
#pragma GCC visibility pop

namespace {

// The shared scratch. In host code this name is only a stand-in for the
// symbol; its device address comes from cudaGetSymbolAddress below.
__device__ __align__(256) unsigned char g_noalloc_scratch[PKV_NOALLOC_SCRATCH_BYTES];

constexpr int kMaxDevices = 64;
std::mutex g_mu;
void* g_scratch_addr[kMaxDevices] = {};

// Device address of the scratch on the current device, looked up once per
// device (the first call on a device does this).
void* scratch_address() {
  int dev = 0;
  if (cudaGetDevice(&dev) != cudaSuccess || dev < 0 || dev >= kMaxDevices) return nullptr;
  std::lock_guard<std::mutex> lk(g_mu);
  if (g_scratch_addr[dev] == nullptr) {
    void* p = nullptr;
    if (cudaGetSymbolAddress(&p, g_noalloc_scratch) != cudaSuccess) return nullptr;
    g_scratch_addr[dev] = p;
  }
  return g_scratch_addr[dev];
}

}  // namespace

extern "C" pkv_status paged_attn_decode_noalloc(
    void* out, const void* q, pkv_dtype q_dtype, const void* k_cache, const void* v_cache,
    pkv_dtype kv_dtype, const int32_t* block_tables, const int32_t* seq_lens, int num_seqs,
    int num_q_heads, int num_kv_heads, int head_dim, int block_size, int max_blocks_per_seq,
    int num_blocks, int max_seq_len, float scale, const float* k_scales, const float* v_scales,
    int partition_tokens, float* out_lse, void* stream) {
  const size_t need = paged_attn_decode_workspace_size(num_seqs, num_q_heads, num_kv_heads,
                                                       head_dim, max_seq_len, partition_tokens);
  if (need > (size_t)PKV_NOALLOC_SCRATCH_BYTES) return PKV_ERR_WORKSPACE;
  void* scratch = nullptr;
  if (need > 0 && num_seqs > 0) {
    scratch = scratch_address();
    if (scratch == nullptr) return PKV_ERR_CUDA;
  }
  // The shared scratch is the workspace. It starts zero-filled (a device
  // global) and every call leaves its counters at zero again.
  return paged_attn_decode(out, q, q_dtype, k_cache, v_cache, kv_dtype, block_tables, seq_lens,
                           num_seqs, num_q_heads, num_kv_heads, head_dim, block_size,
                           max_blocks_per_seq, num_blocks, max_seq_len, scale, k_scales, v_scales,
                           partition_tokens, out_lse, scratch, (size_t)PKV_NOALLOC_SCRATCH_BYTES,
                           stream);
}

extern "C" pkv_status paged_attn_decode_noalloc_reset(void* stream) {
  void* scratch = scratch_address();
  if (scratch == nullptr) return PKV_ERR_CUDA;
  // a memset of the array in place: nothing is allocated
  return cudaMemsetAsync(scratch, 0, (size_t)PKV_NOALLOC_SCRATCH_BYTES,
                         reinterpret_cast<cudaStream_t>(stream)) == cudaSuccess
             ? PKV_OK
             : PKV_ERR_CUDA;
}
