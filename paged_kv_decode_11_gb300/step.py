"""One attention-layer pass of a continuous-batching step, composed from the
three C-ABI calls (argument marshalling and stream plumbing only).

A decode step writes the new token of every sequence into its slot
(reshape_and_cache) and then runs decode attention over the paged cache
("RoPE + KV cache write" followed by "Flash Attention Decode", rvLLM:
High-performance LLM inference in Rust, Kernel Compiler Stack). A mixed
step also carries a chunked-prefill chunk (Litellama, Features, "Chunked
Prefill"): after one cache write of every new token, the bandwidth-bound
decode and the compute-bound prefill chunk overlap on the GPU, either
through one paged_attn_varlen call on one stream or through the two entry
points on two streams.
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


def _pack(obj, names):
    """Moves the named tensor attributes of obj into one device buffer (each
    at a 256-byte aligned offset) and points the attributes at views of it,
    so a step's inputs arrive with one host-to-device copy. Returns the buffer."""
    ts = [getattr(obj, n) for n in names]
    offs, total = [], 0
    for t in ts:
        offs.append(total)
        total += (t.numel() * t.element_size() + 255) & ~255
    buf = torch.empty(max(total, 256), dtype=torch.uint8, device=ts[0].device)
    for n, t, o in zip(names, ts, offs):
        nb = t.numel() * t.element_size()
        v = buf[o:o + nb].view(t.dtype).view(t.shape)
        v.copy_(t)
        setattr(obj, n, v)
    return buf


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
        self.workspace = torch.zeros(max(ws, 256), dtype=torch.uint8, device=q.device)
        self.in_buf = _pack(self, ["q", "new_k", "new_v", "new_slots", "block_tables",
                                   "seq_lens"])

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
        """The whole step in one call (paged_attn_decode_step): the cache write
        of the new tokens, then attention, which starts before the write ends."""
        B.paged_attn_decode_step(self.new_k, self.new_v, self.new_slots, self.out, self.q,
                                 self.k_cache, self.v_cache, self.block_tables, self.seq_lens,
                                 self.scale, self.max_seq_len, self.k_scales, self.v_scales,
                                 partition_tokens=self.partition_tokens, out_lse=self.lse,
                                 workspace=self.workspace, stream=stream)

    # host <-> device traffic of one step, for end-to-end timing: the inputs
    # live in one buffer, so one copy brings them all
    def inputs(self):
        return [self.in_buf]

    def outputs(self):
        return [self.out]


class MixedStep:
    """Decode of many sequences plus one prefill chunk, sharing one cache.

    mode "varlen" (default): one cache write of every new token, then one
    paged_attn_varlen call over the whole batch (decode rows first, then the
    chunk), which overlaps the two kinds of work on one stream. mode
    "streams": the same two kernels through the separate entry points, the
    chunk on a second stream."""

    def __init__(self, decode: DecodeStep, all_new_k, all_new_v, all_new_slots, pf_q,
                 pf_block_tables, pf_seq_lens, pf_cu_q_lens, pf_max_q_len, mode: str = "varlen"):
        assert mode in ("varlen", "streams")
        self.mode = mode
        self.decode = decode
        self.all_new_k, self.all_new_v, self.all_new_slots = all_new_k, all_new_v, all_new_slots
        self.pf_q = pf_q
        self.pf_block_tables, self.pf_seq_lens, self.pf_cu_q_lens = (pf_block_tables, pf_seq_lens,
                                                                     pf_cu_q_lens)
        self.pf_max_q_len = int(pf_max_q_len)
        d = decode
        nd, L = d.q.shape[0], pf_q.shape[0]
        dev = pf_q.device
        if mode == "varlen":
            # one batch: decode rows, then the chunk rows
            self.q_all = torch.cat([d.q, pf_q]).contiguous()
            self.out_all = torch.empty_like(self.q_all)
            self.lse_all = torch.empty(self.q_all.shape[:2], dtype=torch.float32, device=dev)
            width = max(d.block_tables.shape[1], pf_block_tables.shape[1])
            bt = torch.zeros((nd + pf_block_tables.shape[0], width), dtype=torch.int32, device=dev)
            bt[:nd, :d.block_tables.shape[1]] = d.block_tables
            bt[nd:, :pf_block_tables.shape[1]] = pf_block_tables
            self.bt_all = bt
            self.seq_lens_all = torch.cat([d.seq_lens, pf_seq_lens]).contiguous()
            self.qsl = torch.cat([torch.arange(nd, dtype=torch.int32, device=dev),
                                  pf_cu_q_lens.to(torch.int32) + nd]).contiguous()
            self.prefill_out = self.out_all[nd:]
            self.prefill_lse = self.lse_all[nd:]
            self.in_buf = _pack(self, ["q_all", "all_new_k", "all_new_v", "all_new_slots",
                                       "bt_all", "seq_lens_all", "qsl"])
        else:
            self.prefill_out = torch.empty_like(pf_q)
            self.prefill_lse = torch.empty(pf_q.shape[:2], dtype=torch.float32, device=dev)
            self.side = torch.cuda.Stream(device=dev)
            self.ev_written = torch.cuda.Event()
            self.ev_prefill = torch.cuda.Event()
            self.in_buf = _pack(self, ["all_new_k", "all_new_v", "all_new_slots", "pf_q",
                                       "pf_block_tables", "pf_seq_lens", "pf_cu_q_lens"])

    @classmethod
    def from_case(cls, case, k_cache, v_cache, mode: str = "varlen"):
        d = DecodeStep.from_case(case, k_cache, v_cache)
        pf = case.prefill
        return cls(d, _dev(case.new_k), _dev(case.new_v), _dev(case.new_slots), _dev(pf.q),
                   _dev(pf.block_tables), _dev(pf.seq_lens), _dev(pf.cu_q_lens), pf.L, mode)

    @property
    def out(self):
        if self.mode == "varlen":
            return self.out_all[:self.decode.q.shape[0]]
        return self.decode.out

    def run(self, stream: Optional[torch.cuda.Stream] = None):
        main = stream or torch.cuda.current_stream()
        d = self.decode
        B.reshape_and_cache(self.all_new_k, self.all_new_v, d.k_cache, d.v_cache,
                            self.all_new_slots, d.k_scales, d.v_scales, stream=main)
        if self.mode == "varlen":
            B.paged_attn_varlen(self.out_all, self.q_all, d.k_cache, d.v_cache, self.bt_all,
                                self.seq_lens_all, self.qsl, d.q.shape[0], d.scale,
                                self.pf_max_q_len, d.max_seq_len, d.k_scales, d.v_scales,
                                partition_tokens=d.partition_tokens, out_lse=self.lse_all,
                                workspace=d.workspace, stream=main)
            return
        self.ev_written.record(main)
        self.side.wait_event(self.ev_written)
        # prefill first: its CTAs take their SMs, decode fills the rest
        B.paged_attn_prefill_chunk(self.prefill_out, self.pf_q, d.k_cache, d.v_cache,
                                   self.pf_block_tables, self.pf_seq_lens, self.pf_cu_q_lens,
                                   d.scale, self.pf_max_q_len, d.k_scales, d.v_scales,
                                   out_lse=self.prefill_lse, stream=self.side)
        d.attend(stream=main)
        self.ev_prefill.record(self.side)
        main.wait_event(self.ev_prefill)

    def prefill(self, stream: Optional[torch.cuda.Stream] = None):
        """The chunk alone through paged_attn_prefill_chunk (the cache already holds it)."""
        d = self.decode
        B.paged_attn_prefill_chunk(self.prefill_out, self.pf_q, d.k_cache, d.v_cache,
                                   self.pf_block_tables, self.pf_seq_lens, self.pf_cu_q_lens,
                                   d.scale, self.pf_max_q_len, d.k_scales, d.v_scales,
                                   out_lse=self.prefill_lse,
                                   stream=stream or torch.cuda.current_stream())

    def inputs(self):
        if self.mode == "varlen":
            return [self.in_buf]
        return [self.decode.in_buf, self.in_buf]

    def outputs(self):
        if self.mode == "varlen":
            return [self.out_all]
        return [self.decode.out, self.prefill_out]
