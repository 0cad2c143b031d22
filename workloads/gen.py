"""Seeded synthetic inputs for paged-KV attention.

This module is shared by the CUDA path's callers (tests, bench) and by the
oracle's tests. It draws numbers and lays out the paged pool; it holds none of
the attention arithmetic and none of the cache-write arithmetic (each side
quantises to FP8 with its own code).

Recipe (all draws seeded):
  * metadata (context lengths, block placement) from numpy's PCG64
    (`numpy.random.default_rng(seed)`): ctx ~ U[lo, hi] with `rng.integers`,
    physical block ids = `rng.permutation(pool)` taken in order;
  * values (q, every cached K/V row, every new K/V row) ~ N(0, 1), drawn in
    fp32 with a seeded `torch.Generator` on the requested device, then rounded
    to nearest even to the q dtype with `Tensor.to`;
  * FP8 scales: one fp32 scale per KV head for K and one for V, equal to the
    absolute maximum of that head's K (or V) values, over every token the
    cache will hold, divided by 448 (the E4M3 maximum);
  * block-table entries past a sequence's last block name a poison block, a
    valid block filled with NaN (16-bit caches) or the E4M3 NaN code 0x7F;
    every block no sequence owns is poison too; the slots of a sequence's last
    block beyond its context hold a large finite sentinel (60.0, or code
    0x7E = 448 for FP8), so a read past the context shows as a large error.

Rotary tables (`rope_cos_sin`) are model inputs, like weights: row p holds
cos and sin of p * base^(-2i/rot) for i < rot/2, the angles taken in double
and rounded to fp32 once.

A decode step caches, for every sequence, positions 0 .. ctx-2 ("fill" rows,
already in the cache before the step) and writes position ctx-1 ("new" rows,
written by the step's reshape_and_cache). The prefill chunk's sequence has P
fill rows and L new rows. Shared-prefix sequences reach the same physical
blocks for their first `tokens` positions; those rows are cached once.
"""
from __future__ import annotations

import math
from dataclasses import dataclass, field
from typing import Optional

import numpy as np
import torch

from .configs import CONFIGS

TORCH_DTYPES = {"f16": torch.float16, "bf16": torch.bfloat16}
E4M3_NAN_CODE = 0x7F
E4M3_MAX_CODE = 0x7E          # +448
SENTINEL = 60.0
_ROWS_PER_DRAW = 1 << 15       # tokens drawn per torch.randn call


@dataclass
class PrefillPart:
    q: torch.Tensor                 # [L, Hq, D]
    cu_q_lens: np.ndarray           # int32 [2]
    seq_lens: np.ndarray            # int32 [1]   P + L
    block_tables: np.ndarray        # int32 [1, max_blocks]
    L: int
    P: int


@dataclass
class Case:
    name: str
    cfg: dict
    B: int
    Hq: int
    Hkv: int
    D: int
    BS: int
    dtype: str                      # "f16" | "bf16"
    kv_fp8: bool
    scale: np.float32               # 1/sqrt(D) as fp32
    partition_tokens: int
    seq_lens: np.ndarray            # int32 [B]
    block_tables: np.ndarray        # int32 [B, max_blocks_per_seq]
    num_blocks: int
    max_blocks_per_seq: int
    poison_block: int
    q: torch.Tensor                 # [B, Hq, D]
    fill_k: torch.Tensor            # [Tf, Hkv, D]
    fill_v: torch.Tensor
    fill_slots: np.ndarray          # int64 [Tf]
    new_k: torch.Tensor             # [Tn, Hkv, D]
    new_v: torch.Tensor
    new_slots: np.ndarray           # int64 [Tn]
    new_positions: np.ndarray       # int64 [Tn] the new rows' positions in their sequences
    tail_slots: np.ndarray          # int64: slots past a context in its last block
    k_scales: Optional[np.ndarray]  # fp32 [Hkv] (FP8 only)
    v_scales: Optional[np.ndarray]
    prefill: Optional[PrefillPart] = None
    shared_blocks: Optional[np.ndarray] = None
    device: str = "cpu"
    _slot_rows: Optional[np.ndarray] = field(default=None, repr=False)

    @property
    def G(self) -> int:
        return self.Hq // self.Hkv

    @property
    def torch_dtype(self) -> torch.dtype:
        return TORCH_DTYPES[self.dtype]

    @property
    def max_seq_len(self) -> int:
        return int(self.seq_lens.max()) if self.B else 0

    @property
    def kv_elem_bytes(self) -> int:
        return 1 if self.kv_fp8 else 2

    def kv_bytes_logical(self) -> int:
        """K+V bytes one decode call reads by definition (every context
        token of every sequence, per KV head)."""
        return int(self.seq_lens.astype(np.int64).sum()) * self.Hkv * self.D * 2 * self.kv_elem_bytes

    def kv_bytes_unique(self) -> int:
        """As kv_bytes_logical, but blocks reached by several sequences
        counted once."""
        if self.shared_blocks is None:
            return self.kv_bytes_logical()
        n_sh = self.cfg["shared_prefix"][0]
        tok = self.cfg["shared_prefix"][1]
        dup = (n_sh - 1) * tok
        return (int(self.seq_lens.astype(np.int64).sum()) - dup) * self.Hkv * self.D * 2 * self.kv_elem_bytes

    def slot_rows(self) -> np.ndarray:
        """slot -> row of the concatenated [fill; new] value arrays (-1 if no
        token was written there)."""
        if self._slot_rows is None:
            m = np.full(self.num_blocks * self.BS, -1, np.int64)
            tf = len(self.fill_slots)
            m[self.fill_slots] = np.arange(tf, dtype=np.int64)
            ok = self.new_slots >= 0
            m[self.new_slots[ok]] = tf + np.arange(len(self.new_slots), dtype=np.int64)[ok]
            self._slot_rows = m
        return self._slot_rows

    def logical_rows(self, block_table_row: np.ndarray, ctx: int) -> np.ndarray:
        """Rows of [fill; new] holding logical tokens 0..ctx-1 of the sequence
        whose block-table row is given."""
        j = np.arange(ctx, dtype=np.int64)
        slots = block_table_row[j // self.BS].astype(np.int64) * self.BS + j % self.BS
        return self.slot_rows()[slots]


def _gen(seed: int, stream: int, device: str) -> torch.Generator:
    g = torch.Generator(device=device)
    g.manual_seed((seed * 1_000_003 + stream * 7919) & 0x7FFF_FFFF_FFFF)
    return g


def _normal(n_tok: int, Hkv: int, D: int, dtype: torch.dtype, g: torch.Generator,
            device: str) -> torch.Tensor:
    out = torch.empty((n_tok, Hkv, D), dtype=dtype, device=device)
    for s in range(0, n_tok, _ROWS_PER_DRAW):
        e = min(n_tok, s + _ROWS_PER_DRAW)
        out[s:e] = torch.randn((e - s, Hkv, D), generator=g, device=device,
                               dtype=torch.float32).to(dtype)
    return out


def _absmax_per_head(*ts: torch.Tensor) -> np.ndarray:
    m = None
    for t in ts:
        if t.shape[0] == 0:
            continue
        a = t.abs().amax(dim=(0, 2)).float().cpu()
        m = a if m is None else torch.maximum(m, a)
    return m.numpy().astype(np.float32)


def make_case(name: str | dict = "tiny", seed: int = 0, device: str = "cpu",
              **overrides) -> Case:
    """Build one workload. `name` is a key of CONFIGS or a config dict;
    keyword overrides replace config fields (used by tests for edge shapes)."""
    if isinstance(name, dict):
        cfg = dict(name)
        cname = cfg.get("name", "custom")
    else:
        cfg = dict(CONFIGS[name])
        cname = name
    cfg.update(overrides)
    B, Hq, Hkv, D, BS = cfg["B"], cfg["Hq"], cfg["Hkv"], cfg["D"], cfg["BS"]
    assert Hq % Hkv == 0
    dtype = cfg["dtype"]
    tdt = TORCH_DTYPES[dtype]
    kv_fp8 = cfg["kv"] == "fp8"
    rng = np.random.default_rng(seed)

    # --- context lengths ---------------------------------------------------
    kind = cfg["ctx"][0]
    if kind == "fixed":
        ctx = np.asarray(cfg["ctx"][1], dtype=np.int64)
        assert len(ctx) == B
        hi = int(ctx.max()) if B else 0
    else:
        lo, hi = cfg["ctx"][1], cfg["ctx"][2]
        ctx = rng.integers(lo, hi + 1, size=B).astype(np.int64)
    sp = cfg.get("shared_prefix")
    if sp is not None:
        n_sh, sp_tok = sp
        assert sp_tok % BS == 0
        ctx[:n_sh] = np.maximum(ctx[:n_sh], sp_tok + 1)
    hi = max(hi, int(ctx.max()) if B else 0)
    pf = cfg.get("prefill")
    nblk = -(-ctx // BS)                          # blocks per sequence
    max_blocks = max(1, -(-hi // BS))

    # --- block placement ---------------------------------------------------
    n_shared = (sp[1] // BS) if sp is not None else 0
    need = int(nblk.sum()) - (max(0, sp[0] - 1) * n_shared if sp is not None else 0)
    pf_blocks = (-(-(pf[0] + pf[1]) // BS)) if pf is not None else 0
    need += pf_blocks + 1                         # + the poison block
    pool = cfg["pool"]
    num_blocks = pool[1] if pool[0] == "blocks" else int(math.ceil(pool[1] * need))
    assert num_blocks >= need, "pool smaller than the blocks the workload needs"
    perm = rng.permutation(num_blocks).astype(np.int64)
    cursor = 0

    def take(n):
        nonlocal cursor
        r = perm[cursor:cursor + n]
        cursor += n
        return r

    shared = take(n_shared) if sp is not None else None
    poison = int(take(1)[0])
    tables = np.full((B, max_blocks), poison, dtype=np.int32)
    for b in range(B):
        nb = int(nblk[b])
        if sp is not None and b < sp[0]:
            tables[b, :n_shared] = shared
            tables[b, n_shared:nb] = take(nb - n_shared)
        else:
            tables[b, :nb] = take(nb)

    prefill = None
    if pf is not None:
        L, P = pf
        pf_table = np.full((1, max(1, pf_blocks)), poison, dtype=np.int32)
        pf_table[0, :pf_blocks] = take(pf_blocks)

    # --- slots ---------------------------------------------------------------
    def slots_of(row, positions):
        return row[positions // BS].astype(np.int64) * BS + positions % BS

    fill_slots, new_slots, tail, new_pos = [], [], [], []
    for b in range(B):
        c = int(ctx[b])
        start = sp[1] if (sp is not None and 0 < b < sp[0]) else 0
        fill_slots.append(slots_of(tables[b], np.arange(start, c - 1, dtype=np.int64)))
        if c > 0:
            new_slots.append(slots_of(tables[b], np.array([c - 1], np.int64)))
            new_pos.append(np.array([c - 1], np.int64))
        tail.append(slots_of(tables[b], np.arange(c, int(nblk[b]) * BS, dtype=np.int64)))
    if pf is not None:
        fill_slots.append(slots_of(pf_table[0], np.arange(0, P, dtype=np.int64)))
        new_slots.append(slots_of(pf_table[0], np.arange(P, P + L, dtype=np.int64)))
        new_pos.append(np.arange(P, P + L, dtype=np.int64))
        tail.append(slots_of(pf_table[0], np.arange(P + L, pf_blocks * BS, dtype=np.int64)))
    cat = lambda xs: np.concatenate(xs) if xs else np.zeros(0, np.int64)
    fill_slots, new_slots, tail_slots = cat(fill_slots), cat(new_slots), cat(tail)
    new_positions = cat(new_pos)

    # --- values --------------------------------------------------------------
    q = torch.randn((B, Hq, D), generator=_gen(seed, 1, device), device=device,
                    dtype=torch.float32).to(tdt)
    fill_k = _normal(len(fill_slots), Hkv, D, tdt, _gen(seed, 2, device), device)
    fill_v = _normal(len(fill_slots), Hkv, D, tdt, _gen(seed, 3, device), device)
    new_k = _normal(len(new_slots), Hkv, D, tdt, _gen(seed, 4, device), device)
    new_v = _normal(len(new_slots), Hkv, D, tdt, _gen(seed, 5, device), device)
    if pf is not None:
        pq = torch.randn((L, Hq, D), generator=_gen(seed, 6, device), device=device,
                         dtype=torch.float32).to(tdt)
        prefill = PrefillPart(q=pq, cu_q_lens=np.array([0, L], np.int32),
                              seq_lens=np.array([P + L], np.int32),
                              block_tables=pf_table, L=L, P=P)

    k_scales = v_scales = None
    if kv_fp8:
        e4m3_max = np.float32(448.0)
        k_scales = (_absmax_per_head(fill_k, new_k) / e4m3_max).astype(np.float32)
        v_scales = (_absmax_per_head(fill_v, new_v) / e4m3_max).astype(np.float32)

    return Case(
        name=cname, cfg=cfg, B=B, Hq=Hq, Hkv=Hkv, D=D, BS=BS, dtype=dtype,
        kv_fp8=kv_fp8, scale=np.float32(1.0 / math.sqrt(D)),
        partition_tokens=int(cfg.get("partition_tokens", 0)),
        seq_lens=ctx.astype(np.int32), block_tables=tables,
        num_blocks=num_blocks, max_blocks_per_seq=max_blocks,
        poison_block=poison, q=q, fill_k=fill_k, fill_v=fill_v,
        fill_slots=fill_slots, new_k=new_k, new_v=new_v, new_slots=new_slots,
        new_positions=new_positions,
        tail_slots=tail_slots, k_scales=k_scales, v_scales=v_scales,
        prefill=prefill, shared_blocks=shared, device=device)


def rope_cos_sin(max_position: int, rot_dim: int, base: float = 10000.0) -> np.ndarray:
    """A model's rotary table, fp32 [max_position, rot_dim]: row p is
    cos(p w_i) for i < rot_dim/2, then sin(p w_i), with w_i = base^(-2i/rot_dim)
    (angles in double, one rounding to fp32)."""
    assert rot_dim % 2 == 0
    i = np.arange(rot_dim // 2, dtype=np.float64)
    w = base ** (-2.0 * i / rot_dim)
    ang = np.arange(max_position, dtype=np.float64)[:, None] * w[None, :]
    return np.concatenate([np.cos(ang), np.sin(ang)], axis=1).astype(np.float32)


def empty_cache(case: Case, device: Optional[str] = None):
    """The pool before any token is written: poison everywhere, sentinel in
    the tail slots. Returns (k_cache, v_cache) of shape
    [num_blocks, Hkv, BS, D]; uint8 E4M3 codes for FP8, else the q dtype."""
    device = device or case.device
    shape = (case.num_blocks, case.Hkv, case.BS, case.D)
    if case.kv_fp8:
        k = torch.full(shape, E4M3_NAN_CODE, dtype=torch.uint8, device=device)
        sent = E4M3_MAX_CODE
    else:
        k = torch.full(shape, float("nan"), dtype=case.torch_dtype, device=device)
        sent = SENTINEL
    v = k.clone()
    if len(case.tail_slots):
        ts = torch.as_tensor(case.tail_slots, device=device)
        blk, off = ts // case.BS, ts % case.BS
        for c in (k, v):
            c[blk, :, off, :] = sent
    return k, v
