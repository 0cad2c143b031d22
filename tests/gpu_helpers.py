"""Shared plumbing of the GPU parity tests: run the CUDA path through the C
ABI binding, run the oracle on the same seeded inputs, compare."""
import numpy as np
import torch

import paged_kv_decode_11_gb300 as P
from oracle import oracle as O
from workloads import empty_cache

# Output tolerances (max abs error against the fp64 oracle).
TOL = {"f16": 2e-3, "bf16": 1e-2, "fp8": 1e-2}
LSE_TOL = 1e-3


def tol(case):
    return TOL["fp8"] if case.kv_fp8 else TOL[case.dtype]


def dev(a, dtype=None):
    if isinstance(a, np.ndarray):
        t = torch.from_numpy(np.ascontiguousarray(a))
    else:
        t = a
    if dtype is not None:
        t = t.to(dtype)
    return t.contiguous().cuda()


def scales(case):
    if not case.kv_fp8:
        return None, None
    return dev(case.k_scales), dev(case.v_scales)


def product_cache(case, write_new=True):
    """The CUDA path's cache: the poisoned pool, every fill row (and the
    step's new rows) written by the library's reshape_and_cache."""
    kc, vc = empty_cache(case, "cuda")
    ks, vs = scales(case)
    parts = [(case.fill_k, case.fill_v, case.fill_slots)]
    if write_new:
        parts.append((case.new_k, case.new_v, case.new_slots))
    for k, v, sl in parts:
        if len(sl):
            P.reshape_and_cache(dev(k), dev(v), kc, vc, dev(sl), ks, vs)
    return kc, vc


def oracle_cache(case, seqs=None):
    """The oracle's cache. With `seqs`, only the rows those decode sequences
    read are written (enough for sampled comparisons of big workloads)."""
    kc, vc = empty_cache(case, "cpu")
    allk = torch.cat([case.fill_k.cpu(), case.new_k.cpu()])
    allv = torch.cat([case.fill_v.cpu(), case.new_v.cpu()])
    slots = np.concatenate([case.fill_slots, case.new_slots])
    if seqs is None:
        rows = np.arange(len(slots))
    else:
        rows = np.unique(np.concatenate(
            [case.logical_rows(case.block_tables[b], int(case.seq_lens[b])) for b in seqs]))
    rows = torch.as_tensor(rows)
    rc = O.reshape_and_cache(allk[rows].contiguous(), allv[rows].contiguous(), kc, vc,
                             slots[rows.numpy()], case.k_scales, case.v_scales)
    assert rc == 0
    return kc, vc


def run_decode(case, kc, vc, partition_tokens=None, block_tables=None, seq_lens=None, q=None,
               max_seq_len=None, want_lse=True):
    q = dev(case.q) if q is None else q
    out = torch.empty_like(q)
    lse = torch.empty(q.shape[:2], dtype=torch.float32, device="cuda") if want_lse else None
    ks, vs = scales(case)
    bt = dev(case.block_tables if block_tables is None else block_tables)
    sl = dev(case.seq_lens if seq_lens is None else seq_lens)
    pt = case.partition_tokens if partition_tokens is None else partition_tokens
    msl = case.max_seq_len if max_seq_len is None else max_seq_len
    P.paged_attn_decode(out, q, kc, vc, bt, sl, float(case.scale), msl, ks, vs,
                        partition_tokens=pt, out_lse=lse)
    return out, lse


def run_prefill(case, kc, vc):
    pf = case.prefill
    q = dev(pf.q)
    out = torch.empty_like(q)
    lse = torch.empty(q.shape[:2], dtype=torch.float32, device="cuda")
    ks, vs = scales(case)
    P.paged_attn_prefill_chunk(out, q, kc, vc, dev(pf.block_tables), dev(pf.seq_lens),
                               dev(pf.cu_q_lens), float(case.scale), pf.L, ks, vs, out_lse=lse)
    return out, lse


def oracle_decode(case, kc, vc, sel=None, part_tokens=0):
    return O.decode(case.q.cpu(), kc, vc, case.block_tables, case.seq_lens, case.scale,
                    case.k_scales, case.v_scales, sel=sel, part_tokens=part_tokens)


def assert_close(got, want, atol, what):
    g = got.double().cpu().numpy() if isinstance(got, torch.Tensor) else got
    finite = np.isfinite(want)
    assert np.array_equal(np.isfinite(g), finite), f"{what}: non-finite pattern differs"
    err = np.abs(g[finite] - want[finite]).max() if finite.any() else 0.0
    assert err <= atol, f"{what}: max abs error {err:.3e} > {atol:.1e}"
    return err


def check_device_ok():
    bits = P.pkv_get_device_error()
    assert bits == 0, f"device error bits {bits:#x}"
