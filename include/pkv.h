/*
 * pkv.h — C ABI of libpkv: attention over a paged KV cache for one
 * continuous-batching step, on one GB300 (sm_103a).
 *
 * What the operations are (the source pages name them, they print no API):
 *  - "Efficient management of attention key and value memory with
 *    PagedAttention" (Welcome to vLLM, feature list): K/V of every sequence
 *    live in fixed-size physical blocks reached through a per-sequence block
 *    table; "per-step KV bookkeeping handed to the kernels" (Litellama,
 *    Architecture tree, executor/attention_metadata.py).
 *  - "flash attention decode (online softmax, paged KV, GQA)" and
 *    "Split-KV paged attention for long context" (rvLLM: High-performance
 *    LLM inference in Rust, Kernel Compiler Stack / Tier 2: Hand-written CUDA
 *    kernels; FA3 v3 Attention Kernel).
 *  - partial attention "merged by log-sum-exp" (rapid_llm README, feature
 *    table, row "Decode context parallelism"), done here over KV partitions
 *    of one GPU.
 *  - "RoPE + KV cache write -- fused, no intermediate alloc" (rvLLM, Kernel
 *    Compiler Stack, decode step at c=128): rope_reshape_and_cache below; its
 *    cache-write half alone is reshape_and_cache.
 *  - "FP8 KV Cache" (Litellama, Features; rvLLM, Optional Features):
 *    E4M3 codes with one fp32 scale per KV head for K and one for V.
 *  - "Chunked Prefill ... 512-token chunks" (Litellama, Features): causal
 *    attention of a chunk of new query tokens over the same paged cache.
 *
 * Conventions shared by every entry point
 *  - All pointers are DEVICE pointers unless stated; the caller owns every
 *    buffer. The library allocates no device memory and keeps no per-call
 *    state. Its library-wide state: per device, the device error word, the
 *    scratch array of paged_attn_decode_noalloc (PKV_NOALLOC_SCRATCH_BYTES,
 *    a file-scope device array held by every GPU that loads the library),
 *    the cached SM count and the one-time kernel attribute and grid-size
 *    settings; process-wide, the driver's tensor-map encoder entry point.
 *  - `stream` is a cudaStream_t passed as an opaque pointer (NULL = the
 *    legacy default stream). Work is only enqueued; nothing synchronises,
 *    except pkv_get_device_error.
 *  - Argument checks are synchronous: a bad argument returns a status and
 *    nothing is launched. A launch failure returns PKV_ERR_CUDA.
 *  - Data-dependent checks run on the device (block ids outside
 *    [0, num_blocks), slots outside the pool, seq_lens above the stated
 *    maximum). A failing check skips the access, sets a bit in the device
 *    error word and never traps; pkv_get_device_error reads the word.
 *  - Tensors are dense and row-major. Every base pointer must be 16-byte
 *    aligned.
 *  - Layouts (B = num_seqs, Hq = num_q_heads, Hkv = num_kv_heads,
 *    G = Hq / Hkv, D = head_dim, BS = block_size):
 *      q            [B, Hq, D]                       q dtype
 *      out          [B, Hq, D]                       q dtype
 *      k_cache      [num_blocks, Hkv, BS, D]          kv dtype (same for v)
 *      block_tables int32 [B, max_blocks_per_seq]
 *      seq_lens     int32 [B]  context length INCLUDING the new token, whose
 *                              K/V reshape_and_cache has already written
 *    Logical token j of sequence b lives in physical block
 *    block_tables[b][j / BS] at offset j % BS. Query head h reads KV head
 *    h / G. Within a block each KV head's BS x D run is contiguous; the
 *    kernels read it as BS / 16 consecutive pages of 16 tokens, or gather a
 *    16-token page row by row when BS < 16 (BS = 1 is token-level paging).
 *  - Cache slots past a sequence's context (the rest of its last block) may
 *    hold anything, NaN included: they are read with weight 0 and their
 *    values are zeroed before they meet that weight.
 *  - E4M3 caches run f16 tensor-core MMAs on the codes widened to f16
 *    (exact). A bf16 q is scaled by a power of two 2^-e, rounded to f16, and
 *    the scores are multiplied back by 2^e: e is chosen per sequence and KV
 *    head in decode (per query row in prefill) so that the largest |q|
 *    element lands in [2^14, 2^15). Any finite bf16 q works (no overflow to
 *    inf). Elements within 2^-28 of the largest of their group convert
 *    exactly; smaller ones fall into f16's subnormal range and move by at
 *    most 2^-39 of the largest.
 *  - Supported: D in {64, 128, 256}; BS a power of two from 1 to 64 (decode
 *    and the cache writes; prefill, and decode at D = 256, need BS >= 16);
 *    G <= 16 (G <= 8 at D = 256); q dtype F16 or BF16; KV
 *    dtype equal to the q dtype, or FP8_E4M3 with per-KV-head fp32 scales
 *    (dequantised value = code * scale).
 */
#ifndef PKV_H
#define PKV_H

#include <stddef.h>
#include <stdint.h>

#ifdef __cplusplus
extern "C" {
#endif

typedef enum {
  PKV_OK = 0,
  PKV_ERR_INVALID_ARG = 1,   /* null pointer, bad size, misaligned pointer */
  PKV_ERR_UNSUPPORTED = 2,   /* valid but not built: D, BS, G or dtype pair */
  PKV_ERR_WORKSPACE = 3,     /* workspace missing or smaller than required */
  PKV_ERR_CUDA = 4,          /* a CUDA runtime call or a launch failed */
  PKV_ERR_DEVICE_CHECK = 5   /* a device-side check failed (see below) */
} pkv_status;

typedef enum { PKV_F16 = 0, PKV_BF16 = 1, PKV_FP8_E4M3 = 2 } pkv_dtype;

/* Bits of the device error word. */
#define PKV_DEVERR_BLOCK_ID   0x1u  /* block table entry outside [0, num_blocks) */
#define PKV_DEVERR_SLOT       0x2u  /* slot >= num_blocks * block_size */
#define PKV_DEVERR_SEQ_LEN    0x4u  /* seq_len < 0 or above the stated maximum */
#define PKV_DEVERR_TIMEOUT    0x8u  /* a bounded wait on an async copy gave up */
#define PKV_DEVERR_QLEN       0x10u /* prefill: chunk longer than its context, or outside q's rows */
#define PKV_DEVERR_POSITION   0x20u /* rotary: position outside [0, max_position) */
#define PKV_DEVERR_COUNTER    0x40u /* decode: workspace counters were not zero */

/*
 * paged_attn_decode_workspace_size
 *   Bytes of device workspace paged_attn_decode needs for these sizes: the
 *   per-(sequence, KV head) partition counters and the fp32 partial outputs
 *   and log-sum-exps of the split-KV partitions. partition_tokens: as passed
 *   to paged_attn_decode (0 = automatic; the automatic size depends on the
 *   current device's SM count, so query on the device that will run the
 *   call). Returns 0 for invalid sizes.
 */
size_t paged_attn_decode_workspace_size(int num_seqs, int num_q_heads,
                                        int num_kv_heads, int head_dim,
                                        int max_seq_len, int partition_tokens);

/*
 * paged_attn_decode — one query token per sequence against its paged K/V.
 *   For each sequence b and query head h (KV head g = h / G):
 *     s_j   = scale * k_scale[g] * <q[b,h,:], Kcode_j>          j < seq_lens[b]
 *     out   = v_scale[g] * sum_j softmax(s)_j * Vcode_j          (q dtype, RNE)
 *     lse   = log(sum_j exp(s_j))                                (natural log)
 *   (k_scale = v_scale = 1 unless kv_dtype is FP8_E4M3.)
 *   Each context is cut into partitions (of `partition_tokens` tokens, a
 *   multiple of 16 up to 8192, or 0 = automatic sizes); each partition is
 *   reduced with an online softmax and the partitions of a sequence are
 *   merged by log-sum-exp in the same kernel launch. With 0, a batch whose
 *   (sequence, KV head) pairs fit one per SM may be planned as one partition
 *   per context (on head_dim <= 128 with blocks of 16 tokens or more): the
 *   same attention, summed in another order than a split plan.
 *   seq_lens[b] == 0 gives out = 0 and lse = -inf.
 *   max_seq_len: upper bound on every seq_lens[b] (sizes the plan); a larger
 *   seq_len sets PKV_DEVERR_SEQ_LEN and is clamped.
 *   k_scales, v_scales: fp32 [Hkv], required for FP8 KV, ignored otherwise.
 *   out_lse: optional fp32 [B, Hq] (NULL to skip).
 *   workspace: 256-byte aligned device buffer of at least
 *   paged_attn_decode_workspace_size() bytes, always required. Zero-fill it
 *   once before its first use: each call sets the per-(sequence, KV head)
 *   partition counters it used back to zero (CUDA-graph replays included),
 *   so a call enqueues nothing but its kernel. A call that ends with a
 *   device error may leave counters set; zero the workspace again before
 *   reusing it (PKV_DEVERR_COUNTER reports counters found non-zero). Two
 *   calls that share a workspace must not overlap on the GPU.
 *   The kernel is launched as a programmatic dependent of the kernel ahead
 *   of it on `stream`: it may become resident while that kernel runs, and
 *   reads no input before that kernel has finished.
 */
pkv_status paged_attn_decode(void* out, const void* q, pkv_dtype q_dtype,
                             const void* k_cache, const void* v_cache,
                             pkv_dtype kv_dtype, const int32_t* block_tables,
                             const int32_t* seq_lens, int num_seqs,
                             int num_q_heads, int num_kv_heads, int head_dim,
                             int block_size, int max_blocks_per_seq,
                             int num_blocks, int max_seq_len, float scale,
                             const float* k_scales, const float* v_scales,
                             int partition_tokens, float* out_lse,
                             void* workspace, size_t workspace_bytes,
                             void* stream);

/*
 * paged_attn_decode_step — one decode step of attention: the cache write of
 * every sequence's new token, then decode attention, in one call ("RoPE + KV
 * cache write" followed by "Flash Attention Decode", rvLLM: High-performance
 * LLM inference in Rust, Kernel Compiler Stack, decode step).
 *   key, value: [num_seqs, Hkv, D] in the q dtype, the new token of each
 *   sequence; slot_mapping: int64 [num_seqs], its slot. The step's contract:
 *   row b is sequence b's token at position seq_lens[b] - 1 (slot_mapping[b]
 *   is that position's slot, or < 0 to write nothing). Everything else is as
 *   reshape_and_cache followed by paged_attn_decode on `stream`, with the same
 *   results. Because the library itself writes the cache just ahead of the
 *   attention kernel, and only those rows, the attention kernel reads its
 *   inputs and loads every page but the newest token's before the cache write
 *   has finished (the separate calls must wait for it first).
 *   All arguments are checked before anything is enqueued.
 */
pkv_status paged_attn_decode_step(const void* key, const void* value,
                                  const int64_t* slot_mapping, void* out, const void* q,
                                  pkv_dtype q_dtype, void* k_cache, void* v_cache,
                                  pkv_dtype kv_dtype, const int32_t* block_tables,
                                  const int32_t* seq_lens, int num_seqs, int num_q_heads,
                                  int num_kv_heads, int head_dim, int block_size,
                                  int max_blocks_per_seq, int num_blocks, int max_seq_len,
                                  float scale, const float* k_scales, const float* v_scales,
                                  int partition_tokens, float* out_lse, void* workspace,
                                  size_t workspace_bytes, void* stream);

/* Size of the scratch array paged_attn_decode_noalloc uses (32 MiB). */
#define PKV_NOALLOC_SCRATCH_BYTES (32u << 20)

/*
 * paged_attn_decode_noalloc — paged_attn_decode without a caller workspace.
 *   The source pages have no counterpart to this call; it exists for callers
 *   that cannot allocate device memory at the point where they run
 *   attention: an engine whose memory planner has already handed the whole
 *   device to weights and the KV pool, a latency-critical loop that cannot
 *   afford cudaMalloc/cudaFree (they can synchronise the device), or a plain
 *   C host with no allocator of its own.
 *   Same arguments, results and errors as paged_attn_decode, minus the
 *   workspace: the split-KV scratch is one device array of
 *   PKV_NOALLOC_SCRATCH_BYTES inside the library, held by every GPU that
 *   loads the library until the process exits. Sizes whose
 *   paged_attn_decode_workspace_size() exceeds PKV_NOALLOC_SCRATCH_BYTES are
 *   rejected with PKV_ERR_WORKSPACE before anything is launched.
 *   Nothing here allocates. The first call on a device looks up the array's
 *   device address (cudaGetSymbolAddress); make that first call before any
 *   stream capture. The array starts zero-filled and each call leaves the
 *   counters it used at zero. Every call on a device shares the one array,
 *   so calls that overlap on the GPU (on different streams, or from
 *   different threads) race: serialise them. After a race, or a call that
 *   reported a device error, clear the array with
 *   paged_attn_decode_noalloc_reset before the next call.
 */
pkv_status paged_attn_decode_noalloc(void* out, const void* q, pkv_dtype q_dtype,
                                     const void* k_cache, const void* v_cache,
                                     pkv_dtype kv_dtype,
                                     const int32_t* block_tables,
                                     const int32_t* seq_lens, int num_seqs,
                                     int num_q_heads, int num_kv_heads,
                                     int head_dim, int block_size,
                                     int max_blocks_per_seq, int num_blocks,
                                     int max_seq_len, float scale,
                                     const float* k_scales,
                                     const float* v_scales,
                                     int partition_tokens, float* out_lse,
                                     void* stream);

/*
 * paged_attn_decode_noalloc_reset — the way back to a clean scratch array for
 * paged_attn_decode_noalloc. The source pages have no counterpart to this
 * call either. Its callers cannot clear the library's array themselves, yet
 * its partition counters must be zero when a call starts; a call that ended
 * with a device error (PKV_DEVERR_TIMEOUT, for instance), or two calls that
 * overlapped on the GPU, can leave some set, and every later call on that
 * device is then flagged with PKV_DEVERR_COUNTER or merges stale partials.
 * This enqueues on `stream` one cudaMemsetAsync that zero-fills the whole
 * array of the current device (PKV_NOALLOC_SCRATCH_BYTES; it allocates
 * nothing). Call it, on the stream the decode calls use, after such an error
 * and before the next paged_attn_decode_noalloc; it must not overlap a
 * noalloc call on the GPU. Like the decode call, its first use on a device
 * looks up the array's address, so make that first call outside any stream
 * capture. PKV_ERR_CUDA if the lookup or the memset fails.
 */
pkv_status paged_attn_decode_noalloc_reset(void* stream);

/*
 * paged_attn_prefill_chunk — causal attention of a chunk of new query
 * tokens of each sequence over that sequence's paged cache.
 *   Sequence n owns query rows cu_q_lens[n] .. cu_q_lens[n+1]-1 of q/out
 *   ([total_q_tokens, Hq, D]); its chunk length L_n = cu_q_lens[n+1] -
 *   cu_q_lens[n] and seq_lens[n] is its whole context INCLUDING the chunk
 *   (whose K/V reshape_and_cache has already written), so P_n = seq_lens[n]
 *   - L_n tokens precede it. Query row i of the chunk sits at absolute
 *   position P_n + i and attends keys 0 .. P_n + i (causal, aligned to the
 *   bottom right). Same scores, scales and output dtype as decode.
 *   max_q_len: upper bound on every L_n (sizes the grid).
 *   out_lse: optional fp32 [total_q_tokens, Hq].
 *   A chunk with L_n > seq_lens[n], or whose rows do not lie within the
 *   total_q_tokens rows of q and out, sets PKV_DEVERR_QLEN and is skipped.
 *   Launch: one CTA per tile of query rows; when those would occupy at most
 *   half of the SMs, a cluster of two CTAs per tile, each over half of the
 *   tile's keys, merged by log-sum-exp on chip (tensor-core kernel: 16-bit
 *   caches at D 64/128/256, E4M3 caches at D 64/128). With an E4M3 cache a
 *   bf16 q goes to f16 MMAs as described at the top of this file.
 */
pkv_status paged_attn_prefill_chunk(void* out, const void* q,
                                    pkv_dtype q_dtype, const void* k_cache,
                                    const void* v_cache, pkv_dtype kv_dtype,
                                    const int32_t* block_tables,
                                    const int32_t* seq_lens,
                                    const int32_t* cu_q_lens, int num_seqs,
                                    int total_q_tokens, int max_q_len,
                                    int num_q_heads, int num_kv_heads,
                                    int head_dim, int block_size,
                                    int max_blocks_per_seq, int num_blocks,
                                    float scale, const float* k_scales,
                                    const float* v_scales, float* out_lse,
                                    void* stream);

/*
 * paged_attn_varlen — attention for a whole continuous-batching step in one
 * call: decode sequences and prefill chunks over the same paged cache
 * ("Continuous batching" and "Chunked Prefill", Litellama, Features).
 *   Sequences [0, num_decode_seqs) are decode sequences, one query row each:
 *   q rows 0 .. num_decode_seqs-1. Sequences [num_decode_seqs, num_seqs) are
 *   prefill chunks: query_start_loc int32 [num_seqs + 1] holds the first q row
 *   of every sequence (query_start_loc[i] = i for the decode sequences) and
 *   query_start_loc[num_seqs] = total_q_tokens.
 *   q, out: [total_q_tokens, Hq, D]; out_lse (optional): fp32
 *   [total_q_tokens, Hq]. block_tables [num_seqs, max_blocks_per_seq] and
 *   seq_lens [num_seqs] as for decode and prefill (seq_lens include the new
 *   tokens, already cached by reshape_and_cache).
 *   Decode rows are computed by paged_attn_decode's kernel (max_decode_seq_len
 *   bounds their seq_lens and sizes the split; the workspace is
 *   paged_attn_decode_workspace_size(num_decode_seqs, Hq, Hkv, D,
 *   max_decode_seq_len, partition_tokens) bytes). With an explicit
 *   partition_tokens they equal a separate paged_attn_decode call bit for
 *   bit; with partition_tokens = 0 and chunks in the call, the automatic
 *   partitions are sized for one resident decode CTA per SM (the prefill
 *   grid holds SMs meanwhile), so they may round differently from a
 *   separate call. Chunk rows are the causal attention of
 *   paged_attn_prefill_chunk (max_q_len bounds every chunk); a chunk call of
 *   its own may use other tile shapes and sum in another order.
 *   Everything is enqueued on `stream`: the prefill kernel, then the decode
 *   kernel launched as a programmatic dependent of the prefill kernel, so
 *   decode CTAs start on the room the prefill grid leaves instead of
 *   waiting for it to finish (the workspace's split-KV counters reset
 *   themselves, as for paged_attn_decode). Block sizes: >= 16 when there
 *   are chunks.
 */
pkv_status paged_attn_varlen(void* out, const void* q, pkv_dtype q_dtype,
                             const void* k_cache, const void* v_cache,
                             pkv_dtype kv_dtype, const int32_t* block_tables,
                             const int32_t* seq_lens,
                             const int32_t* query_start_loc, int num_seqs,
                             int num_decode_seqs, int total_q_tokens,
                             int max_q_len, int max_decode_seq_len,
                             int num_q_heads, int num_kv_heads, int head_dim,
                             int block_size, int max_blocks_per_seq,
                             int num_blocks, float scale,
                             const float* k_scales, const float* v_scales,
                             int partition_tokens, float* out_lse,
                             void* workspace, size_t workspace_bytes,
                             void* stream);

/*
 * reshape_and_cache — write the K/V rows of new tokens into their slots.
 *   key, value: [num_tokens, Hkv, D] in src_dtype (F16 or BF16).
 *   slot_mapping: int64 [num_tokens]; slot s names block s / BS, offset
 *   s % BS; s < 0 means "write nothing" (padding tokens).
 *   For every token t and KV head h, the D values land in
 *   k_cache[s / BS][h][s % BS][:] (same for v_cache):
 *     kv_dtype == src_dtype : bit copy
 *     kv_dtype == FP8_E4M3  : code = E4M3(x / k_scales[h]) with the division
 *                             done as one correctly rounded fp32 operation
 *                             and the conversion rounding to nearest even,
 *                             saturating at +-448 (NaN stays NaN).
 *   A slot >= num_blocks * BS sets PKV_DEVERR_SLOT and is skipped.
 */
pkv_status reshape_and_cache(const void* key, const void* value,
                             pkv_dtype src_dtype, void* k_cache, void* v_cache,
                             pkv_dtype kv_dtype, const int64_t* slot_mapping,
                             int num_tokens, int num_kv_heads, int head_dim,
                             int block_size, int num_blocks,
                             const float* k_scales, const float* v_scales,
                             void* stream);

/*
 * rope_reshape_and_cache — the rotary position embedding of the new tokens'
 * queries and keys, fused with the cache write of their keys and values
 * (rvLLM, Kernel Compiler Stack, "RoPE + KV cache write -- fused, no
 * intermediate alloc"). The rotation is the rotary embedding of RoFormer:
 * each pair of dims of a head is turned by the angle of the token's position.
 *   query:  [num_tokens, Hq, D] src_dtype, rotated IN PLACE.
 *   key, value: [num_tokens, Hkv, D] src_dtype, read only; the rotated key
 *           is not stored anywhere but in the cache.
 *   positions: int64 [num_tokens], the token's position in its sequence.
 *   cos_sin_cache: fp32 [max_position, rot_dim]; row p holds rot_dim/2
 *           cosines, then rot_dim/2 sines (the model's rotary table).
 *   rot_dim: rotated dims per head, a multiple of 16 in [16, D]; dims from
 *           rot_dim on pass through unchanged.
 *   neox_style: nonzero = pair i is dims (i, i + rot_dim/2) (rotate-half);
 *           zero = pair i is dims (2i, 2i+1) (interleaved).
 *   For pair (x1, x2) and (c, s) = row positions[t], entries i, rot_dim/2+i:
 *     y1 = x1 c - x2 s,  y2 = x2 c + x1 s
 *   with both products exact in double, one rounding of the sum to double
 *   and one round-to-nearest-even to src_dtype. The key's rotated row, in
 *   src_dtype, and the value row are then written to slot_mapping[t] exactly
 *   as reshape_and_cache writes them (bit copy, or the E4M3 encode with
 *   k_scales / v_scales). Slot < 0: the query is still rotated, nothing is
 *   written. A position outside [0, max_position) sets PKV_DEVERR_POSITION:
 *   that token's query is left as it was and nothing is written; a slot
 *   >= num_blocks * BS sets PKV_DEVERR_SLOT and writes nothing.
 */
pkv_status rope_reshape_and_cache(void* query, const void* key, const void* value,
                                  pkv_dtype src_dtype, void* k_cache, void* v_cache,
                                  pkv_dtype kv_dtype, const int64_t* slot_mapping,
                                  const int64_t* positions, const float* cos_sin_cache,
                                  int max_position, int rot_dim, int neox_style,
                                  int num_tokens, int num_q_heads, int num_kv_heads,
                                  int head_dim, int block_size, int num_blocks,
                                  const float* k_scales, const float* v_scales,
                                  void* stream);

/*
 * pkv_get_device_error — synchronises `stream`, then reads and clears the
 * device error word of the current device. Returns PKV_OK when no check
 * failed since the last read, else PKV_ERR_DEVICE_CHECK with the PKV_DEVERR_*
 * bits in *bits (bits may be NULL). PKV_ERR_CUDA if the sync fails.
 */
pkv_status pkv_get_device_error(void* stream, unsigned int* bits);

/* Static, human-readable name of a status. */
const char* pkv_status_string(pkv_status status);

/*
 * pkv_selftest_bounded_wait — checks the failure path every kernel's waits
 * share: enqueues on `stream` one CTA whose thread waits on a shared-memory
 * mbarrier that nothing ever arrives at, with the library's bounded wait
 * limited to `polls` polls (1 .. 2^20). The wait gives up, sets
 * PKV_DEVERR_TIMEOUT in the device error word and the kernel returns; the
 * context stays usable. PKV_ERR_INVALID_ARG for polls outside the range.
 */
pkv_status pkv_selftest_bounded_wait(unsigned int polls, void* stream);

#ifdef __cplusplus
}
#endif

#endif /* PKV_H */
