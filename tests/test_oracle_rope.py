"""Pins of the oracle's rotary embedding and of the fused rotary + cache write
(CPU only), against what the definitions fix: numpy's binary16 rounding, a
brute-force nearest-bfloat16 search, complex multiplication, closed forms and
the relative-position property of rotary embeddings."""
import math

import numpy as np
import pytest
import torch

from oracle import oracle as O
from workloads import make_case, empty_cache, rope_cos_sin


def _bf16_from_bits(b):
    return float(np.array([int(b) << 16], np.uint32).view(np.float32)[0])


def nearest_bf16_bits(v: float) -> int:
    """Brute force: among the bfloat16 codes around v, the one nearest to v,
    ties to the even code (bfloat16 is the top half of a binary32)."""
    if v == 0.0:
        return 0x8000 if math.copysign(1.0, v) < 0 else 0
    u = int(np.array([v], np.float32).view(np.uint32)[0]) >> 16
    best, best_d = None, None
    for c in (u - 1, u, u + 1):
        c &= 0xFFFF
        x = _bf16_from_bits(c)
        if not math.isfinite(x):
            continue
        d = abs(v - x)
        if best is None or d < best_d or (d == best_d and (c & 1) == 0):
            best, best_d = c, d
    return best


# ---- rounding to the 16-bit formats ------------------------------------------

def test_f16_encode_round_trips_every_finite_code():
    for c in range(65536):
        v = O.f16_value(c)
        if math.isfinite(v):
            assert O.f16_encode(v) == c, hex(c)


def test_f16_encode_matches_numpy_direct_rounding():
    rng = np.random.default_rng(5)
    vals = np.concatenate([
        rng.standard_normal(4000) * 10.0 ** rng.integers(-9, 5, 4000),
        rng.standard_normal(500) * 6e-8,                     # subnormal range
        np.array([65504.0, 65519.99, 65520.0, 70000.0, -65520.0, 2.0 ** -25, 2.0 ** -24,
                  3 * 2.0 ** -26, 0.0, -0.0]),
    ])
    with np.errstate(over="ignore"):
        want = vals.astype(np.float16).view(np.uint16)       # numpy rounds double -> half directly
    got = np.array([O.f16_encode(v) for v in vals], np.uint16)
    assert np.array_equal(got, want)


def test_bf16_encode_round_trips_and_is_nearest():
    for c in list(range(0, 0x7F80, 7)) + list(range(0x8000, 0xFF80, 13)):
        assert O.bf16_encode(_bf16_from_bits(c)) == c
    rng = np.random.default_rng(6)
    vals = rng.standard_normal(3000) * 10.0 ** rng.integers(-30, 30, 3000)
    for v in vals:
        assert O.bf16_encode(float(v)) == nearest_bf16_bits(float(v)), v


def test_bf16_encode_rounds_once_from_double():
    # halfway between 1.0 (0x3F80) and the next bfloat16 ties to the even code
    mid = 1.0 + 2.0 ** -8
    assert O.bf16_encode(mid) == 0x3F80
    assert O.bf16_encode(1.0 + 3 * 2.0 ** -8) == 0x3F82      # tie between 0x3F81 and 0x3F82
    # just above the midpoint: rounding to binary32 first would land on the
    # midpoint and tie down; one rounding from double goes up
    assert O.bf16_encode(mid + 2.0 ** -40) == 0x3F81
    assert O.bf16_encode(mid - 2.0 ** -40) == 0x3F80
    # the largest finite value is (2 - 2^-7) 2^127 with an odd significand; its
    # half ulp is 2^119: the tie rounds to infinity, anything below to the max
    big = _bf16_from_bits(0x7F7F)
    assert O.bf16_encode(big + 2.0 ** 119) == 0x7F80
    assert O.bf16_encode(big + 2.0 ** 119 - 2.0 ** 100) == 0x7F7F
    assert O.bf16_encode(-(big + 2.0 ** 120)) == 0xFF80


# ---- rotary embedding -----------------------------------------------------------

def _rows(T, H, D, dtype, seed):
    g = torch.Generator().manual_seed(seed)
    return torch.randn((T, H, D), generator=g).to(dtype)


def _complex_rope(x, pos, cs, rot, neox):
    """Rotation as complex multiplication: pair (x1, x2) as x1 + i x2 times
    c + i s of the token's table row; returns float64 [T, H, D]."""
    xd = x.double().numpy()
    out = xd.copy()
    half = rot // 2
    i1 = np.arange(half) if neox else 2 * np.arange(half)
    i2 = i1 + half if neox else i1 + 1
    rows = cs[pos].astype(np.float64)                         # [T, rot]
    w = (rows[:, :half] + 1j * rows[:, half:])[:, None, :]    # [T, 1, half]
    z = (xd[..., i1] + 1j * xd[..., i2]) * w
    out[..., i1] = z.real
    out[..., i2] = z.imag
    return out


@pytest.mark.parametrize("neox", [True, False])
@pytest.mark.parametrize("rot", [128, 64, 32])
def test_rope_f16_equals_complex_rotation_rounded(neox, rot):
    T, H, D = 37, 3, 128
    cs = rope_cos_sin(4096, rot, 10000.0)
    pos = np.random.default_rng(1).integers(0, 4096, T)
    x = _rows(T, H, D, torch.float16, 2)
    got, flags = O.rope(x, pos, cs, rot, neox)
    assert flags == 0
    want = _complex_rope(x, pos, cs, rot, neox).astype(np.float16)   # numpy: one rounding
    assert np.array_equal(got.numpy().view(np.uint16), want.view(np.uint16))


@pytest.mark.parametrize("neox", [True, False])
def test_rope_bf16_is_nearest_to_complex_rotation(neox):
    T, H, D, rot = 19, 2, 64, 64
    cs = rope_cos_sin(1 << 15, rot, 500000.0)
    pos = np.random.default_rng(3).integers(0, 1 << 15, T)
    x = _rows(T, H, D, torch.bfloat16, 4)
    got, _ = O.rope(x, pos, cs, rot, neox)
    exact = _complex_rope(x, pos, cs, rot, neox)
    gb = got.view(torch.int16).numpy().astype(np.int64) & 0xFFFF
    for idx in np.ndindex(exact.shape):
        assert gb[idx] == nearest_bf16_bits(float(exact[idx])), idx


def test_rope_position_zero_is_identity():
    cs = rope_cos_sin(8, 128)
    x = _rows(5, 4, 128, torch.bfloat16, 7)
    for neox in (True, False):
        got, _ = O.rope(x, np.zeros(5, np.int64), cs, 128, neox)
        assert torch.equal(got.view(torch.int16), x.view(torch.int16))


@pytest.mark.parametrize("neox", [True, False])
def test_rope_of_unit_vectors_gives_table_entries(neox):
    D = rot = 64
    half = rot // 2
    cs = rope_cos_sin(300, rot)
    p = 257
    x = torch.zeros((half, 1, D), dtype=torch.float16)
    for i in range(half):
        x[i, 0, i if neox else 2 * i] = 1.0
    got, _ = O.rope(x, np.full(half, p, np.int64), cs, rot, neox)
    g = got.double().numpy()
    c16 = cs[p, :half].astype(np.float16).astype(np.float64)
    s16 = cs[p, half:].astype(np.float16).astype(np.float64)
    for i in range(half):
        a, b = (i, i + half) if neox else (2 * i, 2 * i + 1)
        assert g[i, 0, a] == c16[i] and g[i, 0, b] == s16[i]
        others = np.delete(g[i, 0], [a, b])
        assert np.all(others == 0.0)


def test_rope_scores_depend_only_on_relative_position():
    D = rot = 128
    cs = rope_cos_sin(5000, rot, 10000.0)
    q = _rows(1, 1, D, torch.float16, 8)
    k = _rows(1, 1, D, torch.float16, 9)

    def score(m, n):
        qr, _ = O.rope(q, np.array([m]), cs, rot, True)
        kr, _ = O.rope(k, np.array([n]), cs, rot, True)
        return float((qr.double() * kr.double()).sum())

    s0 = score(40, 17)
    for shift in (1, 100, 3000):
        assert abs(score(40 + shift, 17 + shift) - s0) < 2e-2
    assert abs(score(40, 17) - score(17, 40)) > 1e-3          # not symmetric in general


def test_rope_partial_rotary_copies_the_rest():
    cs = rope_cos_sin(64, 32)
    x = _rows(6, 2, 128, torch.bfloat16, 10)
    pos = np.arange(6) * 9
    got, _ = O.rope(x, pos, cs, 32, True)
    assert torch.equal(got[..., 32:].view(torch.int16), x[..., 32:].view(torch.int16))
    head, _ = O.rope(x[..., :32].contiguous(), pos, cs, 32, True)
    assert torch.equal(got[..., :32].view(torch.int16), head.view(torch.int16))


def test_rope_flags_position_outside_table_and_leaves_row():
    cs = rope_cos_sin(16, 64)
    x = _rows(3, 2, 64, torch.float16, 11)
    got, flags = O.rope(x, np.array([3, 16, -1]), cs, 64, True)
    assert flags == 2
    assert torch.equal(got[1:].view(torch.int16), x[1:].view(torch.int16))
    assert not torch.equal(got[0].view(torch.int16), x[0].view(torch.int16))


# ---- the fused step -------------------------------------------------------------

@pytest.mark.parametrize("fp8", [False, True])
def test_fused_step_equals_rope_then_cache_write(fp8):
    c = make_case("tiny", 0, kv="fp8" if fp8 else "same")
    cs = rope_cos_sin(512, c.D)
    T = len(c.new_slots)
    g = torch.Generator().manual_seed(12)
    q = torch.randn((T, c.Hq, c.D), generator=g).to(c.torch_dtype)
    k, v = c.new_k.cpu().contiguous(), c.new_v.cpu().contiguous()
    pos = c.new_positions
    slots = c.new_slots.copy()
    slots[1] = -1                                            # a token that is not cached
    kc1, vc1 = empty_cache(c, "cpu")
    q1, flags = O.rope_reshape_and_cache(q, k, v, kc1, vc1, slots, pos, cs, c.D, True,
                                         c.k_scales, c.v_scales)
    assert flags == 0
    qr, _ = O.rope(q, pos, cs, c.D, True)
    kr, _ = O.rope(k, pos, cs, c.D, True)
    kc2, vc2 = empty_cache(c, "cpu")
    assert O.reshape_and_cache(kr, v, kc2, vc2, slots, c.k_scales, c.v_scales) == 0
    assert torch.equal(q1.view(torch.int16), qr.view(torch.int16))
    assert torch.equal(kc1.view(torch.uint8), kc2.view(torch.uint8))
    assert torch.equal(vc1.view(torch.uint8), vc2.view(torch.uint8))
    # the uncached token left its slot as it was
    kc0, _ = empty_cache(c, "cpu")
    s = int(c.new_slots[1])
    assert torch.equal(kc1[s // c.BS, :, s % c.BS].view(torch.uint8),
                       kc0[s // c.BS, :, s % c.BS].view(torch.uint8))


def test_fused_step_flags_bad_position_and_slot():
    c = make_case("tiny", 1)
    cs = rope_cos_sin(64, c.D)
    T = len(c.new_slots)
    q = torch.zeros((T, c.Hq, c.D), dtype=c.torch_dtype)
    pos = np.minimum(c.new_positions, 63)
    pos[0] = 64                                              # outside the table
    slots = c.new_slots.copy()
    slots[2] = c.num_blocks * c.BS                           # outside the pool
    kc, vc = empty_cache(c, "cpu")
    kc0 = kc.clone()
    _, flags = O.rope_reshape_and_cache(q, c.new_k.cpu().contiguous(), c.new_v.cpu().contiguous(),
                                        kc, vc, slots, pos, cs, c.D, True)
    assert flags == 3
    s = int(c.new_slots[0])
    assert torch.equal(kc[s // c.BS, :, s % c.BS].view(torch.int16),
                       kc0[s // c.BS, :, s % c.BS].view(torch.int16))
