"""One attention-layer pass of a continuous-batching step, composed from the
three C-ABI calls (argument marshalling and stream plumbing only).

A decode step writes the new token of every sequence into its slot
(reshape_and_cache) and then runs decode attention over the paged cache
("RoPE + KV cache write" followed by "Flash Attention Decode", rvLLM:
High-performance LLM inference in Rust, Kernel Compiler Stack). A mixed
step also carries a chunked-prefill chunk (Litellama, Features, "Chunked
Prefill"): after one cache write of every new token, decode and the prefill
chunk run on two streams, so the bandwidth-bound decode and the
compute-bound prefill overlap on the GPU.
"""
from __future__ import annotations

from typing import Optional

import numpy as np
import torch

from . import _binding as B


def _dev(a, device="cuda"):
    if isinstance(a, np.ndarray):
        a = torch.from_numpy(np.ascontiguousarray(a))
    return a.to(device).contiguous()


class DecodeStep:
    """Device-resident inputs of one decode step and its outputs."""

    def __init__(self, k_cache, v_cache, q, new_k, new_v, new_slots, block_tables, seq_lens,
                 scale, max_seq_len, k_scales=None, v_scales=None, partition_tokens=0):
        self.k_cache, self.v_cache = k_cache, v_cache
        self.q = q
        self.new_k, self.new_v, self.new_slots = new_k, new_v, new_slots
        self.block_tables, self.seq_lens = block_tables, seq_lens
        self.scale, self.max_seq_len = float(scale), int(max_seq_len)
        self.k_scales, self.v_scales = k_scales, v_scales
        self.partition_tokens = int(partition_tokens)
        self.out = torch.empty_like(q)
        self.lse = torch.empty(q.shape[:2], dtype=torch.float32, device=q.device)
        Bn, Hq, D = q.shape
        ws = B.paged_attn_decode_workspace_size(Bn, Hq, k_cache.shape[1], D, self.max_seq_len,
                                                self.partition_tokens)
        self.workspace = torch.empty(max(ws, 256), dtype=torch.uint8, device=q.device)

    @classmethod
    def from_case(cls, case, k_cache, v_cache):
        ks = vs = None
        if case.kv_fp8:
            ks, vs = _dev(case.k_scales), _dev(case.v_scales)
        nd = case.B       # the decode tokens are the first B new rows
        return cls(k_cache, v_cache, _dev(case.q), _dev(case.new_k[:nd]), _dev(case.new_v[:nd]),
                   _dev(case.new_slots[:nd]), _dev(case.block_tables), _dev(case.seq_lens),
                   case.scale, case.max_seq_len, ks, vs, case.partition_tokens)

    def write_cache(self, stream=None):
        B.reshape_and_cache(self.new_k, self.new_v, self.k_cache, self.v_cache, self.new_slots,
                            self.k_scales, self.v_scales, stream=stream)

    def attend(self, stream=None):
        B.paged_attn_decode(self.out, self.q, self.k_cache, self.v_cache, self.block_tables,
                            self.seq_lens, self.scale, self.max_seq_len, self.k_scales,
                            self.v_scales, partition_tokens=self.partition_tokens,
                            out_lse=self.lse, workspace=self.workspace, stream=stream)

    def run(self, stream=None):
        self.write_cache(stream)
        self.attend(stream)

    # host <-> device traffic of one step, for end-to-end timing
    def inputs(self):
        return [self.q, self.new_k, self.new_v, self.new_slots, self.block_tables, self.seq_lens]

    def outputs(self):
        return [self.out]


class MixedStep:
    """Decode of many sequences plus one prefill chunk, sharing one cache."""

    def __init__(self, decode: DecodeStep, all_new_k, all_new_v, all_new_slots, pf_q,
                 pf_block_tables, pf_seq_lens, pf_cu_q_lens, pf_max_q_len):
        self.decode = decode
        self.all_new_k, self.all_new_v, self.all_new_slots = all_new_k, all_new_v, all_new_slots
        self.pf_q = pf_q
        self.pf_block_tables, self.pf_seq_lens, self.pf_cu_q_lens = (pf_block_tables, pf_seq_lens,
                                                                     pf_cu_q_lens)
        self.pf_max_q_len = int(pf_max_q_len)
        self.prefill_out = torch.empty_like(pf_q)
        self.prefill_lse = torch.empty(pf_q.shape[:2], dtype=torch.float32, device=pf_q.device)
        self.side = torch.cuda.Stream(device=pf_q.device)
        self.ev_written = torch.cuda.Event()
        self.ev_prefill = torch.cuda.Event()

    @classmethod
    def from_case(cls, case, k_cache, v_cache):
        d = DecodeStep.from_case(case, k_cache, v_cache)
        pf = case.prefill
        return cls(d, _dev(case.new_k), _dev(case.new_v), _dev(case.new_slots), _dev(pf.q),
                   _dev(pf.block_tables), _dev(pf.seq_lens), _dev(pf.cu_q_lens), pf.L)

    @property
    def out(self):
        return self.decode.out

    def run(self, stream: Optional[torch.cuda.Stream] = None):
        main = stream or torch.cuda.current_stream()
        d = self.decode
        B.reshape_and_cache(self.all_new_k, self.all_new_v, d.k_cache, d.v_cache,
                            self.all_new_slots, d.k_scales, d.v_scales, stream=main)
        self.ev_written.record(main)
        self.side.wait_event(self.ev_written)
        # prefill first: its CTAs take their SMs, and the persistent decode
        # grid claims work on whatever room is left, then everywhere
        B.paged_attn_prefill_chunk(self.prefill_out, self.pf_q, d.k_cache, d.v_cache,
                                   self.pf_block_tables, self.pf_seq_lens, self.pf_cu_q_lens,
                                   d.scale, self.pf_max_q_len, d.k_scales, d.v_scales,
                                   out_lse=self.prefill_lse, stream=self.side)
        d.attend(stream=main)
        self.ev_prefill.record(self.side)
        main.wait_event(self.ev_prefill)

    def inputs(self):
        d = self.decode
        return [d.q, self.all_new_k, self.all_new_v, self.all_new_slots, d.block_tables,
                d.seq_lens, self.pf_q, self.pf_block_tables, self.pf_seq_lens, self.pf_cu_q_lens]

    def outputs(self):
        return [self.decode.out, self.prefill_out]
