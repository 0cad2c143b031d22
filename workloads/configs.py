"""The five synthetic workloads, as plain data.

Each workload is shaped like one the serving pages describe: one decode step of
one attention layer over a paged KV cache (Welcome to vLLM, feature list:
PagedAttention, continuous batching, chunked prefill, prefix caching), with the
FP8 KV cache of the Litellama page (Features, "FP8 KV Cache") and the 512-token
prefill chunks of the same page (Features, "Chunked Prefill").

Fields
  B, Hq, Hkv, D, BS     sequences, query heads, KV heads, head_dim, block size
  dtype                 "f16" | "bf16": dtype of q, out and the new K/V rows
  kv                    "same" | "fp8": cache dtype (same as q, or E4M3 codes)
  ctx                   ("fixed", [..]) or ("uniform", lo, hi): context lengths,
                        including the token decoded this step
  pool                  ("blocks", n) a pool of n blocks, or ("scale", f) a pool
                        of ceil(f * blocks needed) blocks
  partition_tokens      split-KV partition size handed to the decode call
                        (0 = the library's automatic choice)
  shared_prefix         (n_seqs, tokens): the first n_seqs sequences reach their
                        first `tokens` tokens through identical block ids
  prefill               (L, P): one extra sequence with a chunk of L new query
                        tokens on P cached tokens
"""

CONFIGS = {
    # B4, ctx {17, 64, 100, 255}, 8/2 heads, D64, fp16, 128-block pool.
    "tiny": dict(
        B=4, Hq=8, Hkv=2, D=64, BS=16, dtype="f16", kv="same",
        ctx=("fixed", [17, 64, 100, 255]), pool=("blocks", 128),
        partition_tokens=0, shared_prefix=None, prefill=None),
    # Qwen2.5-7B-shaped layer: B32, 28/4 heads (G=7), D128, bf16,
    # ctx U[512, 2048], pool 1.25x the blocks needed, 32 new tokens cached.
    "qwen2.5-7b": dict(
        B=32, Hq=28, Hkv=4, D=128, BS=16, dtype="bf16", kv="same",
        ctx=("uniform", 512, 2048), pool=("scale", 1.25),
        partition_tokens=0, shared_prefix=None, prefill=None),
    # Llama-3-8B-shaped layer with an FP8 E4M3 cache: B128, 32/8 heads, D128,
    # bf16 q, per-KV-head fp32 scales absmax/448, ctx U[1024, 8192].
    "llama3-8b-fp8": dict(
        B=128, Hq=32, Hkv=8, D=128, BS=16, dtype="bf16", kv="fp8",
        ctx=("uniform", 1024, 8192), pool=("scale", 1.25),
        partition_tokens=0, shared_prefix=None, prefill=None),
    # Long-context split-KV decode: B4, ctx 32K..128K, 32/8 heads, D128,
    # bf16, partitions of 512 tokens.
    "long-ctx": dict(
        B=4, Hq=32, Hkv=8, D=128, BS=16, dtype="bf16", kv="same",
        ctx=("fixed", [32768, 65536, 98304, 131072]), pool=("scale", 1.25),
        partition_tokens=512, shared_prefix=None, prefill=None),
    # Mixed continuous-batching step: 64 decode seqs ctx U[256, 4096] (16 of
    # them share a 1024-token prefix) + one 512-token chunk on 1500 cached
    # tokens; 16/8 heads, D128, bf16; 576 new tokens cached.
    "mixed": dict(
        B=64, Hq=16, Hkv=8, D=128, BS=16, dtype="bf16", kv="same",
        ctx=("uniform", 256, 4096), pool=("scale", 1.25),
        partition_tokens=0, shared_prefix=(16, 1024), prefill=(512, 1500)),
}

# The workload the benchmark times: the FP8-KV Llama-3-8B-shaped decode step.
BENCH_CONFIG = "llama3-8b-fp8"
