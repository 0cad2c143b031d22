"""Thin ctypes binding of libpkv (include/pkv.h), same names as the C ABI.

Only argument marshalling happens here: torch tensors become device pointers,
shapes and dtype codes; every step of the computation runs in the library's
CUDA kernels. There is no fallback: if libpkv.so is missing or a call
returns an error status, a RuntimeError is raised.
"""
from __future__ import annotations

import ctypes
import os
from typing import Optional

import torch

HERE = os.path.dirname(os.path.abspath(__file__))
LIB_PATH = os.path.join(HERE, "libpkv.so")

PKV_F16, PKV_BF16, PKV_FP8_E4M3 = 0, 1, 2
STATUS = {0: "ok", 1: "invalid argument", 2: "unsupported configuration",
          3: "workspace missing or too small", 4: "CUDA error", 5: "device-side check failed"}
DEVERR_BITS = {0x1: "block id", 0x2: "slot", 0x4: "seq_len", 0x8: "timeout", 0x10: "chunk length or rows",
               0x20: "rotary position", 0x40: "workspace counters not zero"}

# Every symbol include/pkv.h declares.
EXPORTS = ("paged_attn_decode_workspace_size", "paged_attn_decode", "paged_attn_decode_step",
           "paged_attn_decode_noalloc", "paged_attn_decode_noalloc_reset",
           "paged_attn_prefill_chunk", "paged_attn_varlen", "reshape_and_cache",
           "rope_reshape_and_cache", "pkv_get_device_error", "pkv_status_string",
           "pkv_selftest_bounded_wait")

_lib = None


class PkvError(RuntimeError):
    def __init__(self, fn: str, status: int, bits: int = 0):
        msg = f"{fn}: {STATUS.get(status, status)}"
        if bits:
            msg += " (" + ", ".join(v for k, v in DEVERR_BITS.items() if bits & k) + ")"
        super().__init__(msg)
        self.status = status
        self.bits = bits


def load(path: str = LIB_PATH):
    """Load libpkv.so and declare its signatures. Raises if it is absent."""
    global _lib
    if _lib is not None:
        return _lib
    if not os.path.exists(path):
        raise RuntimeError(f"libpkv.so not built ({path}); run paged_kv_decode_11_gb300.build.build()")
    L = ctypes.CDLL(path)
    P, I, F, S = ctypes.c_void_p, ctypes.c_int, ctypes.c_float, ctypes.c_size_t
    L.paged_attn_decode_workspace_size.restype = S
    L.paged_attn_decode_workspace_size.argtypes = [I, I, I, I, I, I]
    L.paged_attn_decode.restype = I
    L.paged_attn_decode.argtypes = [P, P, I, P, P, I, P, P, I, I, I, I, I, I, I, I, F, P, P, I, P,
                                    P, S, P]
    L.paged_attn_decode_step.restype = I
    L.paged_attn_decode_step.argtypes = [P, P, P, P, P, I, P, P, I, P, P, I, I, I, I, I, I, I, I,
                                         F, P, P, I, P, P, S, P]
    L.paged_attn_decode_noalloc.restype = I
    L.paged_attn_decode_noalloc.argtypes = [P, P, I, P, P, I, P, P, I, I, I, I, I, I, I, I, F, P,
                                            P, I, P, P]
    L.paged_attn_decode_noalloc_reset.restype = I
    L.paged_attn_decode_noalloc_reset.argtypes = [P]
    L.paged_attn_prefill_chunk.restype = I
    L.paged_attn_prefill_chunk.argtypes = [P, P, I, P, P, I, P, P, P, I, I, I, I, I, I, I, I, I,
                                           F, P, P, P, P]
    L.paged_attn_varlen.restype = I
    L.paged_attn_varlen.argtypes = [P, P, I, P, P, I, P, P, P, I, I, I, I, I, I, I, I, I, I, I, F,
                                    P, P, I, P, P, S, P]
    L.reshape_and_cache.restype = I
    L.reshape_and_cache.argtypes = [P, P, I, P, P, I, P, I, I, I, I, I, P, P, P]
    L.rope_reshape_and_cache.restype = I
    L.rope_reshape_and_cache.argtypes = [P, P, P, I, P, P, I, P, P, P, I, I, I, I, I, I, I, I,
                                         I, P, P, P]
    L.pkv_get_device_error.restype = I
    L.pkv_get_device_error.argtypes = [P, ctypes.POINTER(ctypes.c_uint)]
    L.pkv_status_string.restype = ctypes.c_char_p
    L.pkv_status_string.argtypes = [I]
    L.pkv_selftest_bounded_wait.restype = I
    L.pkv_selftest_bounded_wait.argtypes = [ctypes.c_uint, P]
    _lib = L
    return L


def dtype_code(t: torch.Tensor) -> int:
    if t.dtype == torch.float16:
        return PKV_F16
    if t.dtype == torch.bfloat16:
        return PKV_BF16
    if t.dtype in (torch.uint8, torch.float8_e4m3fn):
        return PKV_FP8_E4M3
    raise TypeError(f"unsupported dtype {t.dtype}")


def _dev_ptr(t: Optional[torch.Tensor], name: str) -> Optional[int]:
    if t is None:
        return None
    if not t.is_cuda:
        raise ValueError(f"{name} must be a CUDA tensor")
    if not t.is_contiguous():
        raise ValueError(f"{name} must be contiguous")
    return t.data_ptr()


def _stream(stream) -> Optional[int]:
    if stream is None:
        return torch.cuda.current_stream().cuda_stream
    if isinstance(stream, torch.cuda.Stream):
        return stream.cuda_stream
    return int(stream)


def _check(fn: str, status: int):
    if status != 0:
        raise PkvError(fn, status)


def paged_attn_decode_workspace_size(num_seqs: int, num_q_heads: int, num_kv_heads: int,
                                     head_dim: int, max_seq_len: int,
                                     partition_tokens: int = 0) -> int:
    return int(load().paged_attn_decode_workspace_size(num_seqs, num_q_heads, num_kv_heads,
                                                        head_dim, max_seq_len, partition_tokens))


def paged_attn_decode(out: torch.Tensor, q: torch.Tensor, k_cache: torch.Tensor,
                      v_cache: torch.Tensor, block_tables: torch.Tensor, seq_lens: torch.Tensor,
                      scale: float, max_seq_len: int, k_scales: Optional[torch.Tensor] = None,
                      v_scales: Optional[torch.Tensor] = None, partition_tokens: int = 0,
                      out_lse: Optional[torch.Tensor] = None,
                      workspace: Optional[torch.Tensor] = None, stream=None) -> None:
    """out[B, Hq, D] <- decode attention of q[B, Hq, D] over the paged cache
    k_cache/v_cache[num_blocks, Hkv, BS, D]. Without a workspace tensor, a
    zero-filled one is allocated with torch on every call (an allocation and a
    fill kernel per call): pass one and reuse it across calls."""
    B, Hq, D = q.shape
    nb, hkv, bs, d2 = k_cache.shape
    assert d2 == D and out.shape == q.shape and out.dtype == q.dtype
    assert block_tables.dtype == torch.int32 and seq_lens.dtype == torch.int32
    if workspace is None:
        ws = paged_attn_decode_workspace_size(B, Hq, hkv, D, max_seq_len, partition_tokens)
        workspace = torch.zeros(max(ws, 256), dtype=torch.uint8, device=q.device)
    st = load().paged_attn_decode(
        _dev_ptr(out, "out"), _dev_ptr(q, "q"), dtype_code(q), _dev_ptr(k_cache, "k_cache"),
        _dev_ptr(v_cache, "v_cache"), dtype_code(k_cache), _dev_ptr(block_tables, "block_tables"),
        _dev_ptr(seq_lens, "seq_lens"), B, Hq, hkv, D, bs, block_tables.shape[1], nb,
        int(max_seq_len), float(scale), _dev_ptr(k_scales, "k_scales"),
        _dev_ptr(v_scales, "v_scales"), int(partition_tokens), _dev_ptr(out_lse, "out_lse"),
        _dev_ptr(workspace, "workspace"), workspace.numel() * workspace.element_size(),
        _stream(stream))
    _check("paged_attn_decode", st)


def paged_attn_decode_step(key: torch.Tensor, value: torch.Tensor, slot_mapping: torch.Tensor,
                           out: torch.Tensor, q: torch.Tensor, k_cache: torch.Tensor,
                           v_cache: torch.Tensor, block_tables: torch.Tensor,
                           seq_lens: torch.Tensor, scale: float, max_seq_len: int,
                           k_scales: Optional[torch.Tensor] = None,
                           v_scales: Optional[torch.Tensor] = None, partition_tokens: int = 0,
                           out_lse: Optional[torch.Tensor] = None,
                           workspace: Optional[torch.Tensor] = None, stream=None) -> None:
    """One decode step: key/value[B, Hkv, D] (each sequence's new token, at
    position seq_lens[b] - 1) written to their slots, then decode attention of
    q[B, Hq, D] into out, in one call (the attention kernel starts before the
    cache write has finished). Same workspace rule as paged_attn_decode."""
    B, Hq, D = q.shape
    nb, hkv, bs, d2 = k_cache.shape
    assert d2 == D and out.shape == q.shape and out.dtype == q.dtype
    assert key.shape == (B, hkv, D) and value.shape == key.shape and key.dtype == q.dtype
    assert slot_mapping.dtype == torch.int64 and slot_mapping.shape[0] == B
    assert block_tables.dtype == torch.int32 and seq_lens.dtype == torch.int32
    if workspace is None:
        ws = paged_attn_decode_workspace_size(B, Hq, hkv, D, max_seq_len, partition_tokens)
        workspace = torch.zeros(max(ws, 256), dtype=torch.uint8, device=q.device)
    st = load().paged_attn_decode_step(
        _dev_ptr(key, "key"), _dev_ptr(value, "value"), _dev_ptr(slot_mapping, "slot_mapping"),
        _dev_ptr(out, "out"), _dev_ptr(q, "q"), dtype_code(q), _dev_ptr(k_cache, "k_cache"),
        _dev_ptr(v_cache, "v_cache"), dtype_code(k_cache), _dev_ptr(block_tables, "block_tables"),
        _dev_ptr(seq_lens, "seq_lens"), B, Hq, hkv, D, bs, block_tables.shape[1], nb,
        int(max_seq_len), float(scale), _dev_ptr(k_scales, "k_scales"),
        _dev_ptr(v_scales, "v_scales"), int(partition_tokens), _dev_ptr(out_lse, "out_lse"),
        _dev_ptr(workspace, "workspace"), workspace.numel() * workspace.element_size(),
        _stream(stream))
    _check("paged_attn_decode_step", st)


def paged_attn_decode_noalloc(out: torch.Tensor, q: torch.Tensor, k_cache: torch.Tensor,
                              v_cache: torch.Tensor, block_tables: torch.Tensor,
                              seq_lens: torch.Tensor, scale: float, max_seq_len: int,
                              k_scales: Optional[torch.Tensor] = None,
                              v_scales: Optional[torch.Tensor] = None, partition_tokens: int = 0,
                              out_lse: Optional[torch.Tensor] = None, stream=None) -> None:
    """Like paged_attn_decode, for callers that cannot allocate: the split-KV
    scratch is the library's own fixed device array (PKV_NOALLOC_SCRATCH_BYTES),
    so no workspace is passed and nothing is allocated. Calls that overlap on
    the GPU share that array and race."""
    B, Hq, D = q.shape
    nb, hkv, bs, d2 = k_cache.shape
    assert d2 == D and out.shape == q.shape and out.dtype == q.dtype
    assert block_tables.dtype == torch.int32 and seq_lens.dtype == torch.int32
    st = load().paged_attn_decode_noalloc(
        _dev_ptr(out, "out"), _dev_ptr(q, "q"), dtype_code(q), _dev_ptr(k_cache, "k_cache"),
        _dev_ptr(v_cache, "v_cache"), dtype_code(k_cache), _dev_ptr(block_tables, "block_tables"),
        _dev_ptr(seq_lens, "seq_lens"), B, Hq, hkv, D, bs, block_tables.shape[1], nb,
        int(max_seq_len), float(scale), _dev_ptr(k_scales, "k_scales"),
        _dev_ptr(v_scales, "v_scales"), int(partition_tokens), _dev_ptr(out_lse, "out_lse"),
        _stream(stream))
    _check("paged_attn_decode_noalloc", st)


def paged_attn_decode_noalloc_reset(stream=None) -> None:
    """Zero-fill the scratch array of paged_attn_decode_noalloc on the current
    device (one cudaMemsetAsync on `stream`, nothing allocated): the way back
    after a device error or an overlap left its partition counters set."""
    _check("paged_attn_decode_noalloc_reset",
           load().paged_attn_decode_noalloc_reset(_stream(stream)))


def paged_attn_prefill_chunk(out: torch.Tensor, q: torch.Tensor, k_cache: torch.Tensor,
                             v_cache: torch.Tensor, block_tables: torch.Tensor,
                             seq_lens: torch.Tensor, cu_q_lens: torch.Tensor, scale: float,
                             max_q_len: int, k_scales: Optional[torch.Tensor] = None,
                             v_scales: Optional[torch.Tensor] = None,
                             out_lse: Optional[torch.Tensor] = None, stream=None) -> None:
    """out[T, Hq, D] <- causal chunked-prefill attention of q[T, Hq, D]."""
    T, Hq, D = q.shape
    nb, hkv, bs, _ = k_cache.shape
    n = seq_lens.shape[0]
    assert cu_q_lens.dtype == torch.int32 and cu_q_lens.shape[0] == n + 1
    st = load().paged_attn_prefill_chunk(
        _dev_ptr(out, "out"), _dev_ptr(q, "q"), dtype_code(q), _dev_ptr(k_cache, "k_cache"),
        _dev_ptr(v_cache, "v_cache"), dtype_code(k_cache), _dev_ptr(block_tables, "block_tables"),
        _dev_ptr(seq_lens, "seq_lens"), _dev_ptr(cu_q_lens, "cu_q_lens"), n, T, int(max_q_len),
        Hq, hkv, D, bs, block_tables.shape[1], nb, float(scale), _dev_ptr(k_scales, "k_scales"),
        _dev_ptr(v_scales, "v_scales"), _dev_ptr(out_lse, "out_lse"), _stream(stream))
    _check("paged_attn_prefill_chunk", st)


def paged_attn_varlen(out: torch.Tensor, q: torch.Tensor, k_cache: torch.Tensor,
                      v_cache: torch.Tensor, block_tables: torch.Tensor, seq_lens: torch.Tensor,
                      query_start_loc: torch.Tensor, num_decode_seqs: int, scale: float,
                      max_q_len: int, max_decode_seq_len: int,
                      k_scales: Optional[torch.Tensor] = None,
                      v_scales: Optional[torch.Tensor] = None, partition_tokens: int = 0,
                      out_lse: Optional[torch.Tensor] = None,
                      workspace: Optional[torch.Tensor] = None, stream=None) -> None:
    """out[T, Hq, D] <- attention of a whole step: q rows 0..num_decode_seqs-1
    are the decode sequences, the rest the prefill chunks that
    query_start_loc [num_seqs + 1] delimits. One call, one stream. Without a
    workspace tensor, a zero-filled one is allocated with torch on every call
    (an allocation and a fill kernel per call): pass one and reuse it."""
    T, Hq, D = q.shape
    nb, hkv, bs, _ = k_cache.shape
    n = seq_lens.shape[0]
    assert out.shape == q.shape and query_start_loc.shape[0] == n + 1
    assert query_start_loc.dtype == torch.int32 and seq_lens.dtype == torch.int32
    if workspace is None:
        ws = paged_attn_decode_workspace_size(num_decode_seqs, Hq, hkv, D, max_decode_seq_len,
                                              partition_tokens)
        workspace = torch.zeros(max(ws, 256), dtype=torch.uint8, device=q.device)
    st = load().paged_attn_varlen(
        _dev_ptr(out, "out"), _dev_ptr(q, "q"), dtype_code(q), _dev_ptr(k_cache, "k_cache"),
        _dev_ptr(v_cache, "v_cache"), dtype_code(k_cache), _dev_ptr(block_tables, "block_tables"),
        _dev_ptr(seq_lens, "seq_lens"), _dev_ptr(query_start_loc, "query_start_loc"), n,
        int(num_decode_seqs), T, int(max_q_len), int(max_decode_seq_len), Hq, hkv, D, bs,
        block_tables.shape[1], nb, float(scale), _dev_ptr(k_scales, "k_scales"),
        _dev_ptr(v_scales, "v_scales"), int(partition_tokens), _dev_ptr(out_lse, "out_lse"),
        _dev_ptr(workspace, "workspace"), workspace.numel() * workspace.element_size(),
        _stream(stream))
    _check("paged_attn_varlen", st)


def reshape_and_cache(key: torch.Tensor, value: torch.Tensor, k_cache: torch.Tensor,
                      v_cache: torch.Tensor, slot_mapping: torch.Tensor,
                      k_scales: Optional[torch.Tensor] = None,
                      v_scales: Optional[torch.Tensor] = None, stream=None) -> None:
    """Write key/value[T, Hkv, D] into their slots of the paged cache."""
    T, hkv, D = key.shape
    nb, hkv2, bs, _ = k_cache.shape
    assert hkv2 == hkv and slot_mapping.dtype == torch.int64
    st = load().reshape_and_cache(
        _dev_ptr(key, "key"), _dev_ptr(value, "value"), dtype_code(key),
        _dev_ptr(k_cache, "k_cache"), _dev_ptr(v_cache, "v_cache"), dtype_code(k_cache),
        _dev_ptr(slot_mapping, "slot_mapping"), T, hkv, D, bs, nb,
        _dev_ptr(k_scales, "k_scales"), _dev_ptr(v_scales, "v_scales"), _stream(stream))
    _check("reshape_and_cache", st)


def rope_reshape_and_cache(query: torch.Tensor, key: torch.Tensor, value: torch.Tensor,
                           k_cache: torch.Tensor, v_cache: torch.Tensor,
                           slot_mapping: torch.Tensor, positions: torch.Tensor,
                           cos_sin_cache: torch.Tensor, rot_dim: Optional[int] = None,
                           neox_style: bool = True, k_scales: Optional[torch.Tensor] = None,
                           v_scales: Optional[torch.Tensor] = None, stream=None) -> None:
    """Rotate query [T, Hq, D] in place and key [T, Hkv, D] by their
    positions with the fp32 table cos_sin_cache [max_position, rot_dim], and
    write the rotated keys and the values into their cache slots."""
    T, Hq, D = query.shape
    nb, hkv, bs, _ = k_cache.shape
    assert key.shape == (T, hkv, D) and value.shape == key.shape
    assert slot_mapping.dtype == torch.int64 and positions.dtype == torch.int64
    assert cos_sin_cache.dtype == torch.float32 and cos_sin_cache.dim() == 2
    rot = cos_sin_cache.shape[1] if rot_dim is None else int(rot_dim)
    assert cos_sin_cache.shape[1] == rot
    st = load().rope_reshape_and_cache(
        _dev_ptr(query, "query"), _dev_ptr(key, "key"), _dev_ptr(value, "value"),
        dtype_code(query), _dev_ptr(k_cache, "k_cache"), _dev_ptr(v_cache, "v_cache"),
        dtype_code(k_cache), _dev_ptr(slot_mapping, "slot_mapping"),
        _dev_ptr(positions, "positions"), _dev_ptr(cos_sin_cache, "cos_sin_cache"),
        cos_sin_cache.shape[0], rot, int(bool(neox_style)), T, Hq, hkv, D, bs, nb,
        _dev_ptr(k_scales, "k_scales"), _dev_ptr(v_scales, "v_scales"), _stream(stream))
    _check("rope_reshape_and_cache", st)


def pkv_get_device_error(stream=None) -> int:
    """Synchronise the stream, read and clear the device error word; returns
    its PKV_DEVERR_* bits (0 when every device-side check passed)."""
    bits = ctypes.c_uint(0)
    st = load().pkv_get_device_error(_stream(stream), ctypes.byref(bits))
    if st not in (0, 5):
        raise PkvError("pkv_get_device_error", st)
    return int(bits.value)


def pkv_status_string(status: int) -> str:
    return load().pkv_status_string(int(status)).decode()


def pkv_selftest_bounded_wait(polls: int, stream=None) -> None:
    """Enqueue the bounded-wait self-test (a wait that nothing satisfies gives
    up after `polls` polls and sets the timeout bit of the device error word)."""
    _check("pkv_selftest_bounded_wait",
           load().pkv_selftest_bounded_wait(int(polls), _stream(stream)))
