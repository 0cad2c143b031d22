"""Brute-force dense attention with torch fp64, for pinning the oracle.

Independent of the oracle: K/V are taken from the generator's source rows in
logical order (never through the paged cache), FP8 values are quantised with
torch's own float8_e4m3fn conversion, GQA uses repeat_interleave and the
softmax is torch.softmax.
"""
import numpy as np
import torch


def source_rows(case):
    """fp64 [Tf+Tn, Hkv, D] K and V source values, as the cache will hold
    them (FP8: torch's E4M3 rounding of x / scale, times the scale)."""
    k = torch.cat([case.fill_k.cpu(), case.new_k.cpu()]).double()
    v = torch.cat([case.fill_v.cpu(), case.new_v.cpu()]).double()
    if case.kv_fp8:
        ks = torch.as_tensor(case.k_scales, dtype=torch.float32)[None, :, None]
        vs = torch.as_tensor(case.v_scales, dtype=torch.float32)[None, :, None]
        kq = (k.float() / ks).to(torch.float8_e4m3fn).double() * ks.double()
        vq = (v.float() / vs).to(torch.float8_e4m3fn).double() * vs.double()
        return kq, vq
    return k, v


def dense_attention(q, K, V, scale, causal_offset=None):
    """q [Lq, Hq, D], K/V [Lk, Hkv, D] fp64. Returns (out [Lq, Hq, D],
    lse [Lq, Hq]). causal_offset P: query row i sees keys 0..P+i."""
    Lq, Hq, D = q.shape
    Hkv = K.shape[1]
    G = Hq // Hkv
    Kx = K.repeat_interleave(G, dim=1)            # [Lk, Hq, D]
    Vx = V.repeat_interleave(G, dim=1)
    s = torch.einsum("qhd,khd->hqk", q.double(), Kx) * float(scale)
    if causal_offset is not None:
        i = torch.arange(Lq)[:, None]
        j = torch.arange(K.shape[0])[None, :]
        s = s.masked_fill((j > causal_offset + i)[None], float("-inf"))
    p = torch.softmax(s, dim=-1)
    out = torch.einsum("hqk,khd->qhd", p, Vx)
    lse = torch.logsumexp(s, dim=-1).transpose(0, 1)
    return out, lse


def dense_decode(case, b, K_all, V_all):
    rows = case.logical_rows(case.block_tables[b], int(case.seq_lens[b]))
    K, V = K_all[rows], V_all[rows]
    out, lse = dense_attention(case.q[b:b + 1].cpu().double(), K, V, np.float64(case.scale))
    return out[0], lse[0]
