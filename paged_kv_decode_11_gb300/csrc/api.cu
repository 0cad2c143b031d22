// api.cu — the extern "C" entry points of libpkv declared in include/pkv.h:
// synchronous argument checks, TMA tensor maps over the paged cache,
// split-KV partition planning, and the kernel launches.
#include <cuda.h>
#include <cudaTypedefs.h>
#include <cuda_runtime.h>
#include <algorithm>
#include <atomic>
#include <cstdint>
#include <cstring>
#include <mutex>

#pragma GCC visibility push(default)
#include "../../include/pkv.h"
#pragma GCC visibility pop
#include "launch.h"
#include "launch_prefill.h"
#include "launch_cache.h"
#include "plan.h"
#include "ptx.cuh"

namespace pkv {

// The device error word: kernels OR PKV_DEVERR_* bits into it; read and
// cleared by pkv_get_device_error.
__device__ unsigned int g_pkv_deverr;

namespace {

constexpr int kMaxDevices = 64;

std::mutex g_mu;
unsigned int* g_err_ptr[kMaxDevices] = {};
int g_sms[kMaxDevices] = {};
PFN_cuTensorMapEncodeTiled_v12000 g_encode = nullptr;

bool current_device(int* dev) {
  if (cudaGetDevice(dev) != cudaSuccess) return false;
  return *dev >= 0 && *dev < kMaxDevices;
}

unsigned int* err_word() {
  int dev;
  if (!current_device(&dev)) return nullptr;
  std::lock_guard<std::mutex> lk(g_mu);
  if (g_err_ptr[dev] == nullptr) {
    void* p = nullptr;
    if (cudaGetSymbolAddress(&p, g_pkv_deverr) != cudaSuccess) return nullptr;
    g_err_ptr[dev] = static_cast<unsigned int*>(p);
  }
  return g_err_ptr[dev];
}

int sm_count() {
  int dev;
  if (!current_device(&dev)) return 0;
  std::lock_guard<std::mutex> lk(g_mu);
  if (g_sms[dev] == 0) {
    int n = 0;
    if (cudaDeviceGetAttribute(&n, cudaDevAttrMultiProcessorCount, dev) != cudaSuccess) return 0;
    g_sms[dev] = n;
  }
  return g_sms[dev];
}

PFN_cuTensorMapEncodeTiled_v12000 encode_fn() {
  std::lock_guard<std::mutex> lk(g_mu);
  if (g_encode == nullptr) {
    void* fn = nullptr;
    cudaDriverEntryPointQueryResult q;
    if (cudaGetDriverEntryPointByVersion("cuTensorMapEncodeTiled", &fn, 12000, cudaEnableDefault,
                                         &q) != cudaSuccess ||
        q != cudaDriverEntryPointSuccess)
      return nullptr;
    g_encode = reinterpret_cast<PFN_cuTensorMapEncodeTiled_v12000>(fn);
  }
  return g_encode;
}

// Tensor map {D, 16, num_blocks * Hkv} over a cache [num_blocks, Hkv, 16, D]:
// one box is 16 page rows by min(row bytes, 128) bytes, swizzled so that
// the fragment loads of the kernels are bank-conflict free.
// log2 of a block size the kernels take (1, 2, 4, ..., 64), or -1.
int block_log2(int block_size) {
  for (int k = 0; k <= 6; ++k)
    if (block_size == (1 << k)) return k;
  return -1;
}

// log2 of the 16-token pages in a block (0 for blocks smaller than a page).
int page_shift(int block_size) {
  const int k = block_log2(block_size);
  return k > 4 ? k - 4 : 0;
}

// Page rows and per-sequence token counts stay within int32.
bool page_rows_fit(int num_blocks, int Hkv, int block_size, int max_blocks_per_seq) {
  return (int64_t)num_blocks * Hkv * block_size < ((int64_t)1 << 31) &&
         (int64_t)max_blocks_per_seq * block_size < ((int64_t)1 << 30);
}

// A cache as the tensor maps see it: {D, 16 rows, num_blocks * Hkv * pages
// per block} (innermost first); page row z = (block * Hkv + head) * ppb + sub.
bool make_kv_tmap(CUtensorMap* m, const void* base, pkv_dtype dt, int D, int Hkv,
                  int num_blocks, int ppb_shift) {
  auto fn = encode_fn();
  if (fn == nullptr) return false;
  const int elt = dt == PKV_FP8_E4M3 ? 1 : 2;
  const int row_bytes = D * elt;
  const int box_row = row_bytes > 128 ? 128 : row_bytes;
  CUtensorMapDataType t = dt == PKV_F16    ? CU_TENSOR_MAP_DATA_TYPE_FLOAT16
                          : dt == PKV_BF16 ? CU_TENSOR_MAP_DATA_TYPE_BFLOAT16
                                           : CU_TENSOR_MAP_DATA_TYPE_UINT8;
  cuuint64_t dims[3] = {(cuuint64_t)D, 16,
                        ((cuuint64_t)num_blocks * (cuuint64_t)Hkv) << ppb_shift};
  cuuint64_t strides[2] = {(cuuint64_t)row_bytes, (cuuint64_t)row_bytes * 16};
  cuuint32_t box[3] = {(cuuint32_t)(box_row / elt), 16, 1};
  cuuint32_t es[3] = {1, 1, 1};
  CUresult r = fn(m, t, 3, const_cast<void*>(base), dims, strides, box, es,
                  CU_TENSOR_MAP_INTERLEAVE_NONE,
                  box_row == 128 ? CU_TENSOR_MAP_SWIZZLE_128B : CU_TENSOR_MAP_SWIZZLE_64B,
                  CU_TENSOR_MAP_L2_PROMOTION_L2_256B, CU_TENSOR_MAP_FLOAT_OOB_FILL_NONE);
  return r == CUDA_SUCCESS;
}

// Tensor map {D, Hq, rows} over the 16-bit queries [rows, Hq, D] of a
// prefill: one box is 64 elements (128 bytes, swizzled like the K and V boxes)
// of the G heads of one KV head over q_tile consecutive tokens, which are the
// (token, head) rows of a tensor-core query tile in the tile's row order.
// Tokens past the last row read as zeros.
bool make_q_tmap(CUtensorMap* m, const void* q, int D, int Hq, int G, int q_tile, int rows) {
  auto fn = encode_fn();
  if (fn == nullptr) return false;
  cuuint64_t dims[3] = {(cuuint64_t)D, (cuuint64_t)Hq, (cuuint64_t)rows};
  cuuint64_t strides[2] = {(cuuint64_t)D * 2, (cuuint64_t)Hq * D * 2};
  cuuint32_t box[3] = {64, (cuuint32_t)G, (cuuint32_t)q_tile};
  cuuint32_t es[3] = {1, 1, 1};
  CUresult r = fn(m, CU_TENSOR_MAP_DATA_TYPE_UINT16, 3, const_cast<void*>(q), dims, strides, box,
                  es, CU_TENSOR_MAP_INTERLEAVE_NONE, CU_TENSOR_MAP_SWIZZLE_128B,
                  CU_TENSOR_MAP_L2_PROMOTION_L2_256B, CU_TENSOR_MAP_FLOAT_OOB_FILL_NONE);
  return r == CUDA_SUCCESS;
}

bool aligned16(const void* p) { return (reinterpret_cast<uintptr_t>(p) & 15u) == 0; }

bool valid_dtypes(pkv_dtype q, pkv_dtype kv) {
  if (q != PKV_F16 && q != PKV_BF16) return false;
  return kv == q || kv == PKV_FP8_E4M3;
}

}  // namespace

// One thread waits on an mbarrier with no arrivals, through the same bounded
// wait the kernels use; when it gives up it records a timeout and returns.
__global__ void selftest_wait_kernel(unsigned int polls, unsigned int* err) {
  __shared__ uint64_t bar;
  if (threadIdx.x != 0) return;
  mbar_init(&bar, 1);
  fence_barrier_init();
  if (!mbar_wait_bounded(&bar, 0, polls)) atomicOr(err, PKV_DEVERR_TIMEOUT);
}

pkv_status launch_selftest_wait(unsigned int polls, unsigned int* err, cudaStream_t stream) {
  selftest_wait_kernel<<<1, 32, 0, stream>>>(polls, err);
  return cudaGetLastError() == cudaSuccess ? PKV_OK : PKV_ERR_CUDA;
}

}  // namespace pkv

using namespace pkv;

extern "C" {

size_t paged_attn_decode_workspace_size(int num_seqs, int num_q_heads, int num_kv_heads,
                                        int head_dim, int max_seq_len, int partition_tokens) {
  if (num_seqs < 0 || num_q_heads <= 0 || num_kv_heads <= 0 || head_dim <= 0 ||
      max_seq_len < 0 || partition_tokens < 0 || partition_tokens % 16 != 0 ||
      partition_tokens > kMaxPartitionTokens)
    return 0;
  return plan_decode(num_seqs, num_q_heads, num_kv_heads, head_dim, max_seq_len,
                     partition_tokens, sm_count())
      .bytes;
}

}  // extern "C"

namespace {

// A decode call checked and planned, ready to enqueue (one kernel launch).
struct DecodeCall {
  DecodeParams p;
  CUtensorMap tmK, tmV;
  int head_dim;
  pkv_dtype q_dtype, kv_dtype;
  bool empty;
};

pkv_status decode_setup(void* out, const void* q, pkv_dtype q_dtype, const void* k_cache,
                        const void* v_cache, pkv_dtype kv_dtype, const int32_t* block_tables,
                        const int32_t* seq_lens, int num_seqs, int num_q_heads, int num_kv_heads,
                        int head_dim, int block_size, int max_blocks_per_seq, int num_blocks,
                        int max_seq_len, float scale, const float* k_scales,
                        const float* v_scales, int partition_tokens, float* out_lse,
                        void* workspace, size_t workspace_bytes, DecodeCall* call,
                        int plan_ctas_per_sm = kDecodeWorkers) {
  call->empty = true;
  if (num_seqs < 0 || num_q_heads <= 0 || num_kv_heads <= 0 || max_seq_len < 0 ||
      max_blocks_per_seq <= 0 || num_blocks <= 0 || partition_tokens < 0)
    return PKV_ERR_INVALID_ARG;
  if (num_q_heads % num_kv_heads != 0) return PKV_ERR_INVALID_ARG;
  if (partition_tokens % 16 != 0 || partition_tokens > kMaxPartitionTokens)
    return PKV_ERR_INVALID_ARG;
  if (!valid_dtypes(q_dtype, kv_dtype)) return PKV_ERR_UNSUPPORTED;
  if (head_dim != 64 && head_dim != 128 && head_dim != 256) return PKV_ERR_UNSUPPORTED;
  const int bs_log2 = block_log2(block_size);
  if (bs_log2 < 0) return PKV_ERR_UNSUPPORTED;
  const int shift = page_shift(block_size);
  if (!page_rows_fit(num_blocks, num_kv_heads, block_size, max_blocks_per_seq))
    return PKV_ERR_INVALID_ARG;
  // blocks below a page are gathered per token, with at most this many per
  // partition and rows of at most 256 bytes
  if (bs_log2 < 4 && (partition_tokens > kGatherMaxPartitionTokens || head_dim > 128))
    return PKV_ERR_UNSUPPORTED;
  const int G = num_q_heads / num_kv_heads;
  if (G > 16 || (head_dim > 128 && G > 8)) return PKV_ERR_UNSUPPORTED;
  if (num_seqs > 65535 || num_kv_heads > 65535) return PKV_ERR_UNSUPPORTED;
  if (num_seqs == 0) return PKV_OK;
  call->empty = false;
  if (!out || !q || !k_cache || !v_cache || !block_tables || !seq_lens)
    return PKV_ERR_INVALID_ARG;
  if (kv_dtype == PKV_FP8_E4M3 && (!k_scales || !v_scales)) return PKV_ERR_INVALID_ARG;
  if (!aligned16(out) || !aligned16(q) || !aligned16(k_cache) || !aligned16(v_cache))
    return PKV_ERR_INVALID_ARG;

  const int sms = sm_count();
  const DecodePlan pl = plan_decode(num_seqs, num_q_heads, num_kv_heads, head_dim, max_seq_len,
                                    partition_tokens, sms, plan_ctas_per_sm);
  if (workspace == nullptr || workspace_bytes < pl.bytes ||
      (reinterpret_cast<uintptr_t>(workspace) & 255u) != 0)
    return PKV_ERR_WORKSPACE;
  call->tmK = CUtensorMap{};
  call->tmV = CUtensorMap{};
  if (bs_log2 >= 4 &&
      (!make_kv_tmap(&call->tmK, k_cache, kv_dtype, head_dim, num_kv_heads, num_blocks, shift) ||
       !make_kv_tmap(&call->tmV, v_cache, kv_dtype, head_dim, num_kv_heads, num_blocks, shift)))
    return PKV_ERR_CUDA;
  unsigned int* err = err_word();
  if (err == nullptr) return PKV_ERR_CUDA;
  char* ws = static_cast<char*>(workspace);
  call->head_dim = head_dim;
  call->q_dtype = q_dtype;
  call->kv_dtype = kv_dtype;
  DecodeParams& p = call->p;
  p = DecodeParams{};
  p.out = out;
  p.q = q;
  p.k_cache = k_cache;
  p.v_cache = v_cache;
  p.block_tables = block_tables;
  p.seq_lens = seq_lens;
  p.k_scales = k_scales;
  p.v_scales = v_scales;
  p.out_lse = out_lse;
  p.done = reinterpret_cast<unsigned long long*>(ws + pl.off_done);
  p.ws_o = reinterpret_cast<float*>(ws + pl.off_o);
  p.ws_lse = reinterpret_cast<float*>(ws + pl.off_lse);
  p.err = err;
  p.B = num_seqs;
  p.Hq = num_q_heads;
  p.Hkv = num_kv_heads;
  p.G = G;
  p.max_blocks = max_blocks_per_seq;
  p.num_blocks = num_blocks;
  p.max_seq_len = max_seq_len;
  p.ppb_shift = shift;
  p.bs_log2 = bs_log2;
  p.part = pl.part;
  p.max_parts = pl.max_parts;
  p.wpart = warp_partition_tokens(partition_tokens, bs_log2);
  if (p.wpart > 0) p.part = p.wpart * kDecodeWarps;
  p.wide = wide_decode((int64_t)num_seqs * num_kv_heads, sms, max_seq_len, partition_tokens,
                       bs_log2, head_dim, plan_ctas_per_sm) ? 1 : 0;
  if (p.wide) p.part = std::max(16, (max_seq_len + 15) / 16 * 16);   // one partition
  p.grid_parts = std::max(1, (max_seq_len + p.part - 1) / p.part);
  p.full_first = full_first_order(num_seqs, num_kv_heads, p.grid_parts, bs_log2,
                                  plan_ctas_per_sm, p.wide != 0) ? 1 : 0;
  p.qk_scale_log2 = scale * 1.4426950408889634f;  // log2(e)
  p.wait_prior = 1;
  return PKV_OK;
}

// Decode is always launched as a programmatic dependent of the kernel ahead
// of it on the stream. With wait_prior it waits for that kernel before
// reading anything (behind a cache write: its launch overlaps the write);
// without, it runs beside it (behind the prefill of the same step, whose
// inputs it does not touch).
// early: the kernel just ahead on the stream is this library's cache write of
// each sequence's newest token (paged_attn_decode_step), so the decode reads
// its inputs and loads every other page before waiting for it.
pkv_status decode_launch(const DecodeCall& c, cudaStream_t stream, bool beside_prior,
                         bool early = false) {
  if (c.empty) return PKV_OK;
  DecodeParams p = c.p;
  p.wait_prior = beside_prior ? 0 : 1;
  p.early = early ? 1 : 0;
  return launch_decode(p, c.head_dim, c.q_dtype, c.kv_dtype, c.tmK, c.tmV, stream, true);
}


struct PrefillCall {
  PrefillParams p;
  CUtensorMap tmQ, tmK, tmV;
  int head_dim;
  pkv_dtype q_dtype, kv_dtype;
  bool empty;
};

pkv_status prefill_setup(void* out, const void* q, pkv_dtype q_dtype, const void* k_cache,
                         const void* v_cache, pkv_dtype kv_dtype, const int32_t* block_tables,
                         const int32_t* seq_lens, const int32_t* cu_q_lens, int num_seqs,
                         int total_q_tokens, int max_q_len, int num_q_heads, int num_kv_heads,
                         int head_dim, int block_size, int max_blocks_per_seq, int num_blocks,
                         float scale, const float* k_scales, const float* v_scales,
                         float* out_lse, int q_rows, PrefillCall* call) {
  call->empty = true;
  if (num_seqs < 0 || total_q_tokens < 0 || max_q_len < 0 || num_q_heads <= 0 ||
      num_kv_heads <= 0 || max_blocks_per_seq <= 0 || num_blocks <= 0)
    return PKV_ERR_INVALID_ARG;
  if (num_q_heads % num_kv_heads != 0) return PKV_ERR_INVALID_ARG;
  if (!valid_dtypes(q_dtype, kv_dtype)) return PKV_ERR_UNSUPPORTED;
  if (head_dim != 64 && head_dim != 128 && head_dim != 256) return PKV_ERR_UNSUPPORTED;
  const int bs_log2 = block_log2(block_size);
  if (bs_log2 < 4) return PKV_ERR_UNSUPPORTED;
  const int shift = page_shift(block_size);
  if (!page_rows_fit(num_blocks, num_kv_heads, block_size, max_blocks_per_seq))
    return PKV_ERR_INVALID_ARG;
  const int G = num_q_heads / num_kv_heads;
  if (G > 16 || (head_dim > 128 && G > 8)) return PKV_ERR_UNSUPPORTED;
  if (num_seqs > 65535 || num_kv_heads > 65535) return PKV_ERR_UNSUPPORTED;
  if (num_seqs == 0 || total_q_tokens == 0 || max_q_len == 0) return PKV_OK;
  call->empty = false;
  if (!out || !q || !k_cache || !v_cache || !block_tables || !seq_lens || !cu_q_lens)
    return PKV_ERR_INVALID_ARG;
  if (kv_dtype == PKV_FP8_E4M3 && (!k_scales || !v_scales)) return PKV_ERR_INVALID_ARG;
  if (!aligned16(out) || !aligned16(q) || !aligned16(k_cache) || !aligned16(v_cache))
    return PKV_ERR_INVALID_ARG;
  if (!make_kv_tmap(&call->tmK, k_cache, kv_dtype, head_dim, num_kv_heads, num_blocks, shift) ||
      !make_kv_tmap(&call->tmV, v_cache, kv_dtype, head_dim, num_kv_heads, num_blocks, shift))
    return PKV_ERR_CUDA;
  call->tmQ = CUtensorMap{};
  if (kv_dtype != PKV_FP8_E4M3 && prefill_tc_supported(head_dim, kv_dtype) &&
      !make_q_tmap(&call->tmQ, q, head_dim, num_q_heads, G, kPrefillTcRows / G, q_rows))
    return PKV_ERR_CUDA;
  unsigned int* err = err_word();
  if (err == nullptr) return PKV_ERR_CUDA;
  call->head_dim = head_dim;
  call->q_dtype = q_dtype;
  call->kv_dtype = kv_dtype;
  PrefillParams& p = call->p;
  p = PrefillParams{};
  p.out = out;
  p.q = q;
  p.block_tables = block_tables;
  p.seq_lens = seq_lens;
  p.cu_q_lens = cu_q_lens;
  p.k_scales = k_scales;
  p.v_scales = v_scales;
  p.out_lse = out_lse;
  p.err = err;
  p.num_seqs = num_seqs;
  p.Hq = num_q_heads;
  p.Hkv = num_kv_heads;
  p.G = G;
  p.max_blocks = max_blocks_per_seq;
  p.num_blocks = num_blocks;
  p.max_q_len = max_q_len;
  p.q_tile = prefill_q_tile(G);
  p.q_rows = q_rows;
  p.ppb_shift = shift;
  p.qk_scale_log2 = scale * 1.4426950408889634f;  // log2(e)
  return PKV_OK;
}

// beside_decode: a decode grid is launched right behind this one to run on
// the SMs it leaves free
pkv_status prefill_launch(const PrefillCall& c, cudaStream_t stream, bool beside_decode) {
  if (c.empty) return PKV_OK;
  if (prefill_tc_supported(c.head_dim, c.kv_dtype))
    return launch_prefill_tc(c.p, c.head_dim, c.q_dtype, c.kv_dtype, c.tmQ, c.tmK, c.tmV, stream,
                             !beside_decode);
  return launch_prefill(c.p, c.head_dim, c.q_dtype, c.kv_dtype, c.tmK, c.tmV, stream);
}

}  // namespace

extern "C" {

pkv_status paged_attn_decode(void* out, const void* q, pkv_dtype q_dtype, const void* k_cache,
                             const void* v_cache, pkv_dtype kv_dtype, const int32_t* block_tables,
                             const int32_t* seq_lens, int num_seqs, int num_q_heads,
                             int num_kv_heads, int head_dim, int block_size,
                             int max_blocks_per_seq, int num_blocks, int max_seq_len, float scale,
                             const float* k_scales, const float* v_scales, int partition_tokens,
                             float* out_lse, void* workspace, size_t workspace_bytes,
                             void* stream) {
  DecodeCall c;
  pkv_status st = decode_setup(out, q, q_dtype, k_cache, v_cache, kv_dtype, block_tables,
                               seq_lens, num_seqs, num_q_heads, num_kv_heads, head_dim,
                               block_size, max_blocks_per_seq, num_blocks, max_seq_len, scale,
                               k_scales, v_scales, partition_tokens, out_lse, workspace,
                               workspace_bytes, &c);
  if (st != PKV_OK || c.empty) return st;
  const cudaStream_t s = reinterpret_cast<cudaStream_t>(stream);
  return decode_launch(c, s, false);
}

pkv_status paged_attn_decode_step(const void* key, const void* value,
                                  const int64_t* slot_mapping, void* out, const void* q,
                                  pkv_dtype q_dtype, void* k_cache, void* v_cache,
                                  pkv_dtype kv_dtype, const int32_t* block_tables,
                                  const int32_t* seq_lens, int num_seqs, int num_q_heads,
                                  int num_kv_heads, int head_dim, int block_size,
                                  int max_blocks_per_seq, int num_blocks, int max_seq_len,
                                  float scale, const float* k_scales, const float* v_scales,
                                  int partition_tokens, float* out_lse, void* workspace,
                                  size_t workspace_bytes, void* stream) {
  DecodeCall c;
  pkv_status st = decode_setup(out, q, q_dtype, k_cache, v_cache, kv_dtype, block_tables,
                               seq_lens, num_seqs, num_q_heads, num_kv_heads, head_dim,
                               block_size, max_blocks_per_seq, num_blocks, max_seq_len, scale,
                               k_scales, v_scales, partition_tokens, out_lse, workspace,
                               workspace_bytes, &c);
  if (st != PKV_OK) return st;
  // checked in full before anything is enqueued
  if (num_seqs > 0 && (!key || !value || !slot_mapping || !aligned16(key) || !aligned16(value)))
    return PKV_ERR_INVALID_ARG;
  st = reshape_and_cache(key, value, q_dtype, k_cache, v_cache, kv_dtype, slot_mapping, num_seqs,
                         num_kv_heads, head_dim, block_size, num_blocks, k_scales, v_scales,
                         stream);
  if (st != PKV_OK || c.empty) return st;
  return decode_launch(c, reinterpret_cast<cudaStream_t>(stream), false, true);
}

pkv_status paged_attn_prefill_chunk(void* out, const void* q, pkv_dtype q_dtype,
                                    const void* k_cache, const void* v_cache, pkv_dtype kv_dtype,
                                    const int32_t* block_tables, const int32_t* seq_lens,
                                    const int32_t* cu_q_lens, int num_seqs, int total_q_tokens,
                                    int max_q_len, int num_q_heads, int num_kv_heads,
                                    int head_dim, int block_size, int max_blocks_per_seq,
                                    int num_blocks, float scale, const float* k_scales,
                                    const float* v_scales, float* out_lse, void* stream) {
  PrefillCall c;
  pkv_status st = prefill_setup(out, q, q_dtype, k_cache, v_cache, kv_dtype, block_tables,
                                seq_lens, cu_q_lens, num_seqs, total_q_tokens, max_q_len,
                                num_q_heads, num_kv_heads, head_dim, block_size,
                                max_blocks_per_seq, num_blocks, scale, k_scales, v_scales,
                                out_lse, total_q_tokens, &c);
  if (st != PKV_OK || c.empty) return st;
  return prefill_launch(c, reinterpret_cast<cudaStream_t>(stream), false);
}

pkv_status paged_attn_varlen(void* out, const void* q, pkv_dtype q_dtype, const void* k_cache,
                             const void* v_cache, pkv_dtype kv_dtype, const int32_t* block_tables,
                             const int32_t* seq_lens, const int32_t* query_start_loc,
                             int num_seqs, int num_decode_seqs, int total_q_tokens,
                             int max_q_len, int max_decode_seq_len, int num_q_heads,
                             int num_kv_heads, int head_dim, int block_size,
                             int max_blocks_per_seq, int num_blocks, float scale,
                             const float* k_scales, const float* v_scales, int partition_tokens,
                             float* out_lse, void* workspace, size_t workspace_bytes,
                             void* stream) {
  if (num_seqs < 0 || num_decode_seqs < 0 || num_decode_seqs > num_seqs ||
      total_q_tokens < num_decode_seqs || max_blocks_per_seq <= 0 || num_kv_heads <= 0)
    return PKV_ERR_INVALID_ARG;
  const int n_pf = num_seqs - num_decode_seqs;
  if (n_pf > 0 && query_start_loc == nullptr) return PKV_ERR_INVALID_ARG;
  if (!aligned16(out) || !aligned16(q)) return PKV_ERR_INVALID_ARG;
  const int32_t* pf_tables = block_tables ? block_tables + (size_t)num_decode_seqs *
                                                               max_blocks_per_seq
                                          : nullptr;
  DecodeCall dc;
  PrefillCall pc;
  // with chunks in the call, the prefill grid holds SMs while decode runs, and
  // automatic decode partitions are planned for one resident CTA per SM
  // (longer partitions: the mixed step 2-5 us faster; the same plan slowed a
  // decode call that has the GPU to itself)
  pkv_status st = decode_setup(out, q, q_dtype, k_cache, v_cache, kv_dtype, block_tables,
                               seq_lens, num_decode_seqs, num_q_heads, num_kv_heads, head_dim,
                               block_size, max_blocks_per_seq, num_blocks, max_decode_seq_len,
                               scale, k_scales, v_scales, partition_tokens, out_lse, workspace,
                               workspace_bytes, &dc, n_pf > 0 ? 1 : kDecodeWorkers);
  if (st != PKV_OK) return st;
  // the chunks' query rows follow the decode rows; their offsets in
  // query_start_loc[num_decode_seqs ..] are absolute rows of q and out
  st = prefill_setup(out, q, q_dtype, k_cache, v_cache, kv_dtype, pf_tables,
                     seq_lens ? seq_lens + num_decode_seqs : nullptr,
                     query_start_loc ? query_start_loc + num_decode_seqs : nullptr, n_pf,
                     total_q_tokens - num_decode_seqs, max_q_len, num_q_heads, num_kv_heads,
                     head_dim, block_size, max_blocks_per_seq, num_blocks, scale, k_scales,
                     v_scales, out_lse, total_q_tokens, &pc);
  if (st != PKV_OK) return st;
  const cudaStream_t s = reinterpret_cast<cudaStream_t>(stream);
  // the prefill chunks, then decode launched as a programmatic dependent of
  // the prefill kernel, whose CTAs release it as they start, so both kinds of
  // work share the GPU without a second stream
  if ((st = prefill_launch(pc, s, !dc.empty)) != PKV_OK) return st;
  return decode_launch(dc, s, !pc.empty);
}

pkv_status reshape_and_cache(const void* key, const void* value, pkv_dtype src_dtype,
                             void* k_cache, void* v_cache, pkv_dtype kv_dtype,
                             const int64_t* slot_mapping, int num_tokens, int num_kv_heads,
                             int head_dim, int block_size, int num_blocks,
                             const float* k_scales, const float* v_scales, void* stream) {
  if (num_tokens < 0 || num_kv_heads <= 0 || num_blocks <= 0) return PKV_ERR_INVALID_ARG;
  if (!valid_dtypes(src_dtype, kv_dtype)) return PKV_ERR_UNSUPPORTED;
  if (head_dim != 64 && head_dim != 128 && head_dim != 256) return PKV_ERR_UNSUPPORTED;
  const int bs_log2 = block_log2(block_size);
  if (bs_log2 < 0) return PKV_ERR_UNSUPPORTED;
  if (num_tokens == 0) return PKV_OK;
  if (!key || !value || !k_cache || !v_cache || !slot_mapping) return PKV_ERR_INVALID_ARG;
  if (kv_dtype == PKV_FP8_E4M3 && (!k_scales || !v_scales)) return PKV_ERR_INVALID_ARG;
  if (!aligned16(key) || !aligned16(value) || !aligned16(k_cache) || !aligned16(v_cache))
    return PKV_ERR_INVALID_ARG;
  unsigned int* err = err_word();
  if (err == nullptr) return PKV_ERR_CUDA;
  CacheWriteParams p{};
  p.key = key;
  p.value = value;
  p.k_cache = k_cache;
  p.v_cache = v_cache;
  p.slots = slot_mapping;
  p.k_scales = k_scales;
  p.v_scales = v_scales;
  p.err = err;
  p.num_tokens = num_tokens;
  p.Hkv = num_kv_heads;
  p.D = head_dim;
  p.num_blocks = num_blocks;
  p.bs_log2 = bs_log2;
  return launch_cache_write(p, src_dtype, kv_dtype, reinterpret_cast<cudaStream_t>(stream));
}

pkv_status rope_reshape_and_cache(void* query, const void* key, const void* value,
                                  pkv_dtype src_dtype, void* k_cache, void* v_cache,
                                  pkv_dtype kv_dtype, const int64_t* slot_mapping,
                                  const int64_t* positions, const float* cos_sin_cache,
                                  int max_position, int rot_dim, int neox_style, int num_tokens,
                                  int num_q_heads, int num_kv_heads, int head_dim, int block_size,
                                  int num_blocks, const float* k_scales, const float* v_scales,
                                  void* stream) {
  if (num_tokens < 0 || num_q_heads <= 0 || num_kv_heads <= 0 || num_blocks <= 0 ||
      max_position <= 0)
    return PKV_ERR_INVALID_ARG;
  if (!valid_dtypes(src_dtype, kv_dtype)) return PKV_ERR_UNSUPPORTED;
  if (head_dim != 64 && head_dim != 128 && head_dim != 256) return PKV_ERR_UNSUPPORTED;
  const int bs_log2 = block_log2(block_size);
  if (bs_log2 < 0) return PKV_ERR_UNSUPPORTED;
  if (rot_dim < 16 || rot_dim > head_dim || rot_dim % 16 != 0) return PKV_ERR_INVALID_ARG;
  if (num_tokens == 0) return PKV_OK;
  if (!query || !key || !value || !k_cache || !v_cache || !slot_mapping || !positions ||
      !cos_sin_cache)
    return PKV_ERR_INVALID_ARG;
  if (kv_dtype == PKV_FP8_E4M3 && (!k_scales || !v_scales)) return PKV_ERR_INVALID_ARG;
  if (!aligned16(query) || !aligned16(key) || !aligned16(value) || !aligned16(k_cache) ||
      !aligned16(v_cache) || !aligned16(cos_sin_cache))
    return PKV_ERR_INVALID_ARG;
  unsigned int* err = err_word();
  if (err == nullptr) return PKV_ERR_CUDA;
  RopeCacheParams p{};
  p.query = query;
  p.key = key;
  p.value = value;
  p.k_cache = k_cache;
  p.v_cache = v_cache;
  p.slots = slot_mapping;
  p.positions = positions;
  p.cos_sin = cos_sin_cache;
  p.k_scales = k_scales;
  p.v_scales = v_scales;
  p.err = err;
  p.max_position = max_position;
  p.rot = rot_dim;
  p.neox = neox_style != 0;
  p.num_tokens = num_tokens;
  p.Hq = num_q_heads;
  p.Hkv = num_kv_heads;
  p.D = head_dim;
  p.num_blocks = num_blocks;
  p.bs_log2 = bs_log2;
  return launch_rope_cache(p, src_dtype, kv_dtype, reinterpret_cast<cudaStream_t>(stream));
}

pkv_status pkv_selftest_bounded_wait(unsigned int polls, void* stream) {
  if (polls < 1 || polls > (1u << 20)) return PKV_ERR_INVALID_ARG;
  unsigned int* err = err_word();
  if (err == nullptr) return PKV_ERR_CUDA;
  return launch_selftest_wait(polls, err, reinterpret_cast<cudaStream_t>(stream));
}

pkv_status pkv_get_device_error(void* stream, unsigned int* bits) {
  if (cudaStreamSynchronize(reinterpret_cast<cudaStream_t>(stream)) != cudaSuccess)
    return PKV_ERR_CUDA;
  unsigned int* err = err_word();
  if (err == nullptr) return PKV_ERR_CUDA;
  unsigned int v = 0;
  if (cudaMemcpy(&v, err, sizeof(v), cudaMemcpyDeviceToHost) != cudaSuccess) return PKV_ERR_CUDA;
  if (v != 0 && cudaMemset(err, 0, sizeof(v)) != cudaSuccess) return PKV_ERR_CUDA;
  if (bits) *bits = v;
  return v ? PKV_ERR_DEVICE_CHECK : PKV_OK;
}

const char* pkv_status_string(pkv_status s) {
  switch (s) {
    case PKV_OK: return "ok";
    case PKV_ERR_INVALID_ARG: return "invalid argument";
    case PKV_ERR_UNSUPPORTED: return "unsupported configuration";
    case PKV_ERR_WORKSPACE: return "workspace missing or too small";
    case PKV_ERR_CUDA: return "CUDA error";
    case PKV_ERR_DEVICE_CHECK: return "device-side check failed";
  }
  return "unknown status";
}

}  // extern "C"
