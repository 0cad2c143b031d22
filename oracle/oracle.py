"""ctypes front end of the fp64 C oracle (oracle.c).

TEST INFRASTRUCTURE ONLY: imported by the tests, by the smoke check and by the
bench's CPU-baseline leg, never by the product path. It shares no code with
the CUDA path. Inputs are host (CPU) torch tensors or numpy arrays; results
are float64 numpy arrays.
"""
from __future__ import annotations

import ctypes
import os
import platform
import subprocess
from typing import Optional

import numpy as np
import torch

_HERE = os.path.dirname(os.path.abspath(__file__))
_SRC = os.path.join(_HERE, "oracle.c")
_OUT = os.path.join(_HERE, "_build", f"liboracle_{platform.machine()}.so")
_lib = None

F16, BF16, E4M3 = 0, 1, 2
_DT = {torch.float16: F16, torch.bfloat16: BF16, torch.uint8: E4M3}


def build(force: bool = False) -> str:
    """Compile oracle.c with gcc (fp64, -O2, OpenMP, no fast-math)."""
    if (not force and os.path.exists(_OUT)
            and os.path.getmtime(_OUT) >= os.path.getmtime(_SRC)):
        return _OUT
    os.makedirs(os.path.dirname(_OUT), exist_ok=True)
    tmp = _OUT + f".tmp{os.getpid()}"
    subprocess.check_call(["gcc", "-O2", "-fopenmp", "-fPIC", "-shared", "-std=c11",
                           "-fno-fast-math", "-ffp-contract=off", _SRC, "-o", tmp, "-lm"])
    os.replace(tmp, _OUT)
    return _OUT


def lib():
    global _lib
    if _lib is None:
        L = ctypes.CDLL(build())
        P, I, D, I64 = ctypes.c_void_p, ctypes.c_int, ctypes.c_double, ctypes.c_int64
        L.pkvo_f16_value.restype = D
        L.pkvo_f16_value.argtypes = [ctypes.c_uint16]
        L.pkvo_bf16_value.restype = D
        L.pkvo_bf16_value.argtypes = [ctypes.c_uint16]
        L.pkvo_e4m3_value.restype = D
        L.pkvo_e4m3_value.argtypes = [ctypes.c_uint8]
        L.pkvo_e4m3_encode.restype = ctypes.c_uint8
        L.pkvo_e4m3_encode.argtypes = [ctypes.c_float]
        L.pkvo_f16_encode.restype = ctypes.c_uint16
        L.pkvo_f16_encode.argtypes = [D]
        L.pkvo_bf16_encode.restype = ctypes.c_uint16
        L.pkvo_bf16_encode.argtypes = [D]
        L.pkvo_rope.restype = I
        L.pkvo_rope.argtypes = [P, I, I, I, I, P, P, I64, I, I, P]
        L.pkvo_rope_reshape_and_cache.restype = I
        L.pkvo_rope_reshape_and_cache.argtypes = [P, P, P, I, P, P, I, P, P, P, I64, I, I, I, I,
                                                  I, I, I, I, P, P, P]
        L.pkvo_set_threads.argtypes = [I]
        L.pkvo_get_threads.restype = I
        L.pkvo_reshape_and_cache.restype = I
        L.pkvo_reshape_and_cache.argtypes = [P, P, I, P, P, I, P, I, I, I, I, I, P, P]
        L.pkvo_decode.restype = I
        L.pkvo_decode.argtypes = [P, P, P, I, P, P, I, P, P, I, I, I, I, I, I, I64, D,
                                  P, P, P, I, I, I, I]
        L.pkvo_prefill_chunk.restype = I
        L.pkvo_prefill_chunk.argtypes = [P, P, P, I, P, P, I, P, P, P, I, I, I, I, I, I,
                                         I64, D, P, P]
        _lib = L
    return _lib


def _ptr(a) -> Optional[int]:
    if a is None:
        return None
    if isinstance(a, torch.Tensor):
        assert a.device.type == "cpu" and a.is_contiguous()
        return a.data_ptr()
    assert a.flags["C_CONTIGUOUS"]
    return a.ctypes.data


def _np(a, dt):
    return None if a is None else np.ascontiguousarray(np.asarray(a, dtype=dt))


def set_threads(n: int) -> None:
    lib().pkvo_set_threads(int(n))


def threads() -> int:
    return int(lib().pkvo_get_threads())


def f16_value(bits: int) -> float:
    return lib().pkvo_f16_value(bits)


def bf16_value(bits: int) -> float:
    return lib().pkvo_bf16_value(bits)


def e4m3_value(code: int) -> float:
    return lib().pkvo_e4m3_value(code)


def e4m3_encode(y: float) -> int:
    return int(lib().pkvo_e4m3_encode(float(np.float32(y))))


def f16_encode(v: float) -> int:
    """Bits of the binary16 nearest to v (ties to even)."""
    return int(lib().pkvo_f16_encode(float(v)))


def bf16_encode(v: float) -> int:
    """Bits of the bfloat16 nearest to v (ties to even)."""
    return int(lib().pkvo_bf16_encode(float(v)))


def rope(x, positions, cos_sin, rot_dim: int, neox: bool = True):
    """Rotary embedding of rows x [T, H, D] (fp16/bf16, CPU) by their tokens'
    positions with the fp32 table cos_sin [max_position, rot_dim] (cosines,
    then sines). Returns (rotated rows, same dtype; flags: 2 if a position was
    outside the table)."""
    T, H, D = x.shape
    pos = _np(positions, np.int64)
    cs = _np(cos_sin, np.float32)
    out = torch.empty_like(x)
    rc = lib().pkvo_rope(_ptr(x), _DT[x.dtype], T, H, D, _ptr(pos), _ptr(cs), int(cs.shape[0]),
                         int(rot_dim), int(bool(neox)), _ptr(out))
    return out, int(rc)


def rope_reshape_and_cache(q, key, value, k_cache, v_cache, slots, positions, cos_sin,
                           rot_dim: int, neox: bool = True, k_scales=None, v_scales=None):
    """The fused step: rotated queries (returned) and the rotated keys plus
    the values written into the caches in place. Returns (q_out, flags) with
    flags bit 1 = a slot outside the pool, bit 2 = a position outside the
    table."""
    T, Hq, D = q.shape
    nb, hkv, bs, _ = k_cache.shape
    pos = _np(positions, np.int64)
    sl = _np(slots, np.int64)
    cs = _np(cos_sin, np.float32)
    ks, vs = _np(k_scales, np.float32), _np(v_scales, np.float32)
    q_out = torch.empty_like(q)
    rc = lib().pkvo_rope_reshape_and_cache(
        _ptr(q), _ptr(key), _ptr(value), _DT[q.dtype], _ptr(k_cache), _ptr(v_cache),
        _DT[k_cache.dtype], _ptr(sl), _ptr(pos), _ptr(cs), int(cs.shape[0]), int(rot_dim),
        int(bool(neox)), T, Hq, hkv, D, bs, nb, _ptr(ks), _ptr(vs), _ptr(q_out))
    if rc < 0:
        raise MemoryError("oracle rope_reshape_and_cache: out of host memory")
    return q_out, int(rc)


def reshape_and_cache(key, value, k_cache, v_cache, slots, k_scales=None, v_scales=None) -> int:
    """Writes key/value [T, Hkv, D] into the caches [num_blocks, Hkv, BS, D]
    in place. Returns 0, or -1 when some slot was outside the pool."""
    nb, hkv, bs, d = k_cache.shape
    slots = _np(slots, np.int64)
    ks, vs = _np(k_scales, np.float32), _np(v_scales, np.float32)
    return lib().pkvo_reshape_and_cache(
        _ptr(key), _ptr(value), _DT[key.dtype], _ptr(k_cache), _ptr(v_cache),
        _DT[k_cache.dtype], _ptr(slots), int(len(slots)), hkv, d, bs, nb,
        _ptr(ks), _ptr(vs))


def decode(q, k_cache, v_cache, block_tables, seq_lens, scale, k_scales=None,
           v_scales=None, sel=None, part_tokens: int = 0, heads=None):
    """fp64 decode attention. q [B, Hq, D]; caches [num_blocks, Hkv, BS, D].
    Returns (out [nsel, nh, D], lse [nsel, nh]) for the selected sequences
    and the query-head range `heads` = (lo, hi) (default: all heads)."""
    B, Hq, D = q.shape
    h_lo, h_hi = (0, Hq) if heads is None else heads
    nb, hkv, bs, _ = k_cache.shape
    bt = _np(block_tables, np.int32)
    sl = _np(seq_lens, np.int32)
    sel_a = None if sel is None else _np(sel, np.int32)
    nsel = B if sel is None else len(sel_a)
    out = np.zeros((nsel, h_hi - h_lo, D), np.float64)
    lse = np.zeros((nsel, h_hi - h_lo), np.float64)
    ks, vs = _np(k_scales, np.float32), _np(v_scales, np.float32)
    rc = lib().pkvo_decode(
        _ptr(out), _ptr(lse), _ptr(q), _DT[q.dtype], _ptr(k_cache), _ptr(v_cache),
        _DT[k_cache.dtype], _ptr(bt), _ptr(sl), B, Hq, hkv, D, bs, bt.shape[1], nb,
        float(scale), _ptr(ks), _ptr(vs), _ptr(sel_a), nsel, int(part_tokens), h_lo, h_hi)
    if rc != 0:
        raise ValueError("oracle decode: block id outside the pool")
    return out, lse


def prefill_chunk(q, k_cache, v_cache, block_tables, seq_lens, cu_q_lens, scale,
                  k_scales=None, v_scales=None):
    """fp64 causal chunked-prefill attention. q [total_q, Hq, D].
    Returns (out [total_q, Hq, D], lse [total_q, Hq])."""
    T, Hq, D = q.shape
    nb, hkv, bs, _ = k_cache.shape
    bt = _np(block_tables, np.int32)
    sl = _np(seq_lens, np.int32)
    cu = _np(cu_q_lens, np.int32)
    out = np.zeros((T, Hq, D), np.float64)
    lse = np.zeros((T, Hq), np.float64)
    ks, vs = _np(k_scales, np.float32), _np(v_scales, np.float32)
    rc = lib().pkvo_prefill_chunk(
        _ptr(out), _ptr(lse), _ptr(q), _DT[q.dtype], _ptr(k_cache), _ptr(v_cache),
        _DT[k_cache.dtype], _ptr(bt), _ptr(sl), _ptr(cu), len(sl), Hq, hkv, D, bs,
        bt.shape[1], nb, float(scale), _ptr(ks), _ptr(vs))
    if rc == -2:
        raise ValueError("oracle prefill: chunk longer than its context")
    if rc != 0:
        raise ValueError("oracle prefill: block id outside the pool")
    return out, lse


def fill_cache(case):
    """The oracle's own cache for a generated case: the poisoned pool with
    every fill row and every new row written by the oracle's cache write."""
    from workloads import empty_cache
    k, v = empty_cache(case, "cpu")
    ks, vs = case.k_scales, case.v_scales
    for kk, vv, sl in ((case.fill_k, case.fill_v, case.fill_slots),
                       (case.new_k, case.new_v, case.new_slots)):
        if len(sl):
            rc = reshape_and_cache(kk.cpu().contiguous(), vv.cpu().contiguous(), k, v, sl, ks, vs)
            assert rc == 0
    return k, v
