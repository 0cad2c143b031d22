"""Pins of the fp64 oracle against what the definitions fix (CPU only).

Each test checks the oracle against something other than itself: library
routines (numpy / torch number formats, torch softmax), the OFP8 code table,
closed forms, and invariants the attention definition implies.
"""
import math
import os

import numpy as np
import pytest
import torch

from oracle import oracle as O
from workloads import make_case, empty_cache
from tests.dense_ref import dense_attention, dense_decode, source_rows

GOLDEN = os.path.join(os.path.dirname(__file__), "golden")


def _read_golden(name):
    rows = []
    with open(os.path.join(GOLDEN, name)) as f:
        for line in f:
            line = line.split("#")[0].strip()
            if line:
                rows.append(line.split())
    return rows


# ---- number formats -------------------------------------------------------

def test_f16_decode_matches_numpy_all_codes():
    codes = np.arange(65536, dtype=np.uint32).astype(np.uint16)
    ref = codes.view(np.float16).astype(np.float64)
    mine = np.array([O.f16_value(int(c)) for c in codes])
    assert np.array_equal(np.isnan(ref), np.isnan(mine))
    ok = ~np.isnan(ref)
    assert np.array_equal(ref[ok], mine[ok])


def test_bf16_decode_matches_torch():
    codes = np.arange(0, 65536, 7, dtype=np.uint32).astype(np.uint16)
    ref = torch.from_numpy(codes.view(np.int16)).view(torch.bfloat16).double().numpy()
    mine = np.array([O.bf16_value(int(c)) for c in codes])
    ok = ~np.isnan(ref)
    assert np.array_equal(np.isnan(ref), np.isnan(mine))
    assert np.array_equal(ref[ok], mine[ok])


def test_e4m3_decode_matches_torch_all_codes():
    ref = torch.arange(256, dtype=torch.uint8).view(torch.float8_e4m3fn).double().numpy()
    mine = np.array([O.e4m3_value(c) for c in range(256)])
    assert np.array_equal(np.isnan(ref), np.isnan(mine))
    ok = ~np.isnan(ref)
    assert np.array_equal(ref[ok], mine[ok])
    assert np.array_equal(np.signbit(ref[ok]), np.signbit(mine[ok]))


def test_e4m3_golden_code_points():
    for code, val in _read_golden("e4m3_ofp8.txt"):
        c = int(code, 16)
        got = O.e4m3_value(c)
        if val == "nan":
            assert math.isnan(got)
        else:
            assert got == float(val) and math.copysign(1, got) == math.copysign(1, float(val))
            assert O.e4m3_encode(float(val)) == c


def test_e4m3_encode_round_trips_every_finite_code():
    for c in range(256):
        v = O.e4m3_value(c)
        if not math.isnan(v):
            assert O.e4m3_encode(v) == c, hex(c)


def test_e4m3_encode_ties_go_to_even_code():
    vals = sorted({O.e4m3_value(c) for c in range(0, 0x7F)})   # 0 .. 448
    for lo, hi in zip(vals[:-1], vals[1:]):
        mid = (lo + hi) / 2                                    # exact in fp32 here
        assert np.float32(mid) == mid
        c_lo, c_hi = O.e4m3_encode(lo), O.e4m3_encode(hi)
        want = c_lo if c_lo % 2 == 0 else c_hi
        assert O.e4m3_encode(mid) == want
        assert O.e4m3_encode(-mid) == (want | 0x80)
        below = float(np.nextafter(np.float32(mid), np.float32(0)))
        above = float(np.nextafter(np.float32(mid), np.float32(1e9)))
        assert O.e4m3_encode(below) == c_lo
        assert O.e4m3_encode(above) == c_hi


def test_e4m3_encode_saturates_and_keeps_nan():
    for y in (448.0, 449.0, 464.0, 1e6, float("inf"), 3.0e38):
        assert O.e4m3_encode(y) == 0x7E
        assert O.e4m3_encode(-y) == 0xFE
    assert (O.e4m3_encode(float("nan")) & 0x7F) == 0x7F
    assert O.e4m3_encode(-0.0) == 0x80 and O.e4m3_encode(0.0) == 0x00
    assert O.e4m3_encode(2.0 ** -11) == 0x00            # below half the smallest subnormal
    assert O.e4m3_encode(-(2.0 ** -10)) == 0x80         # tie with zero -> even (zero)


def test_e4m3_encode_matches_torch_in_range():
    g = torch.Generator().manual_seed(7)
    y = (torch.randn(200_000, generator=g) * torch.exp(torch.randn(200_000, generator=g) * 3)).float()
    y = y[(y.abs() < 440)]
    ref = y.to(torch.float8_e4m3fn).view(torch.uint8).numpy()
    mine = np.array([O.e4m3_encode(float(v)) for v in y.numpy()], dtype=np.uint8)
    assert np.array_equal(ref, mine)


# ---- cache write ----------------------------------------------------------

@pytest.mark.parametrize("fp8", [False, True])
def test_reshape_and_cache_places_rows_at_layout_offsets(fp8):
    nb, hkv, bs, d, T = 6, 3, 16, 64, 9
    g = torch.Generator().manual_seed(1)
    key = torch.randn((T, hkv, d), generator=g).to(torch.bfloat16)
    val = torch.randn((T, hkv, d), generator=g).to(torch.bfloat16)
    slots = np.array([5, 17, 95, -1, 0, 40, 63, -7, 33], np.int64)
    dt = torch.uint8 if fp8 else torch.bfloat16
    fillv = 0x55 if fp8 else 0
    kc = torch.full((nb, hkv, bs, d), fillv, dtype=dt) if fp8 else torch.zeros((nb, hkv, bs, d), dtype=dt)
    vc = kc.clone()
    ks = np.array([0.011, 0.02, 0.0155], np.float32) if fp8 else None
    vs = np.array([0.03, 0.0123, 0.02], np.float32) if fp8 else None
    assert O.reshape_and_cache(key, val, kc, vc, slots, ks, vs) == 0
    flat_k = kc.view(-1).numpy() if fp8 else kc.view(torch.int16).view(-1).numpy()
    written = np.zeros(flat_k.shape, bool)
    for t, s in enumerate(slots):
        if s < 0:
            continue
        for h in range(hkv):
            off = ((s // bs) * hkv + h) * bs * d + (s % bs) * d
            written[off:off + d] = True
            if fp8:
                want = (key[t, h].float() / torch.tensor(ks[h])).to(torch.float8_e4m3fn).view(torch.uint8).numpy()
            else:
                want = key[t, h].view(torch.int16).numpy()
            assert np.array_equal(flat_k[off:off + d], want)
    # nothing else changed (slots -1 / -7 wrote nothing)
    untouched = flat_k[~written]
    assert np.all(untouched == fillv)


def test_reshape_and_cache_rejects_slot_outside_pool():
    kc = torch.zeros((2, 1, 16, 64), dtype=torch.float16)
    vc = kc.clone()
    key = torch.ones((2, 1, 64), dtype=torch.float16)
    assert O.reshape_and_cache(key, key, kc, vc, np.array([32, 3], np.int64)) == -1
    assert kc.view(-1)[3 * 64:4 * 64].eq(1).all() and kc.sum() == 64


# ---- attention pins -------------------------------------------------------

def _oracle_case(case, **kw):
    k, v = O.fill_cache(case)
    return O.decode(case.q, k, v, case.block_tables, case.seq_lens, case.scale,
                    case.k_scales, case.v_scales, **kw), (k, v)


@pytest.mark.parametrize("fp8", [False, True])
def test_length_one_sequence_returns_its_v_row(fp8):
    c = make_case("tiny", 3, ctx=("fixed", [1, 1, 1, 1]), kv="fp8" if fp8 else "same")
    (out, lse), (kc, vc) = _oracle_case(c)
    K, V = source_rows(c)
    for b in range(c.B):
        row = c.logical_rows(c.block_tables[b], 1)[0]
        for h in range(c.Hq):
            g = h // c.G
            assert np.array_equal(out[b, h], V[row, g].numpy())
            s0 = float(c.scale) * float(torch.dot(c.q[b, h].double(), K[row, g]))
            assert lse[b, h] == pytest.approx(s0, abs=1e-12)


def test_identical_keys_give_mean_of_v():
    c = make_case("tiny", 4)
    kc, vc = O.fill_cache(c)
    for b in range(c.B):
        n = int(c.seq_lens[b])
        j = np.arange(n)
        blk = c.block_tables[b][j // 16]
        kc[blk, :, j % 16, :] = kc[c.block_tables[b][0], :, 0, :].clone()[None]
    out, lse = O.decode(c.q, kc, vc, c.block_tables, c.seq_lens, c.scale)
    for b in range(c.B):
        n = int(c.seq_lens[b])
        j = np.arange(n)
        blk = c.block_tables[b][j // 16]
        Vb = vc[blk, :, j % 16, :].double()              # [n, Hkv, D]
        mean = Vb.mean(dim=0).repeat_interleave(c.G, dim=0).numpy()
        assert np.abs(out[b] - mean).max() < 1e-13
        s0 = torch.einsum("hd,hd->h", c.q[b].double(),
                          kc[blk[0], :, 0, :].double().repeat_interleave(c.G, 0)) * float(c.scale)
        assert np.abs(lse[b] - (s0.numpy() + math.log(n))).max() < 1e-12


def _remap_blocks(case, kc, vc, seed):
    """The same logical cache with every owned block moved to another
    physical id: returns (tables', k', v')."""
    rng = np.random.default_rng(seed)
    perm = rng.permutation(case.num_blocks)
    k2, v2 = torch.empty_like(kc), torch.empty_like(vc)
    k2[perm] = kc
    v2[perm] = vc
    return perm[case.block_tables].astype(np.int32), k2, v2


@pytest.mark.parametrize("fp8", [False, True])
def test_block_placement_does_not_change_outputs(fp8):
    c = make_case("tiny", 5, kv="fp8" if fp8 else "same")
    (out, lse), (kc, vc) = _oracle_case(c)
    t2, k2, v2 = _remap_blocks(c, kc, vc, 11)
    out2, lse2 = O.decode(c.q, k2, v2, t2, c.seq_lens, c.scale, c.k_scales, c.v_scales)
    assert np.array_equal(out, out2) and np.array_equal(lse, lse2)


def test_shared_prefix_blocks_equal_copied_blocks():
    cfg = dict(B=6, Hq=4, Hkv=2, D=64, BS=16, dtype="bf16", kv="same",
               ctx=("uniform", 40, 120), pool=("scale", 2.0), partition_tokens=0,
               shared_prefix=(3, 32), prefill=None)
    c = make_case(cfg, 2)
    kc, vc = O.fill_cache(c)
    out, lse = O.decode(c.q, kc, vc, c.block_tables, c.seq_lens, c.scale)
    # give sequences 1 and 2 private copies of the shared blocks
    free = [i for i in range(c.num_blocks) if i not in set(c.block_tables.ravel().tolist())]
    t2 = c.block_tables.copy()
    k2, v2 = kc.clone(), vc.clone()
    for b in (1, 2):
        for i in range(2):
            nid = free.pop()
            k2[nid], v2[nid] = kc[t2[b, i]], vc[t2[b, i]]
            t2[b, i] = nid
    assert len(set(t2[:3, :2].ravel().tolist())) == 6
    out2, lse2 = O.decode(c.q, k2, v2, t2, c.seq_lens, c.scale)
    assert np.array_equal(out, out2) and np.array_equal(lse, lse2)


@pytest.mark.parametrize("part", [16, 48, 512])
@pytest.mark.parametrize("fp8", [False, True])
def test_split_merge_equals_unsplit(part, fp8):
    c = make_case("tiny", 6, kv="fp8" if fp8 else "same",
                  ctx=("fixed", [17, 64, 100, 600]), pool=("blocks", 128))
    (out, lse), (kc, vc) = _oracle_case(c)
    out2, lse2 = O.decode(c.q, kc, vc, c.block_tables, c.seq_lens, c.scale,
                          c.k_scales, c.v_scales, part_tokens=part)
    assert np.abs(out - out2).max() < 1e-12
    assert np.abs(lse - lse2).max() < 1e-12


@pytest.mark.parametrize("name,fp8,seed", [("tiny", False, 0), ("tiny", True, 1), ("gqa7", False, 2)])
def test_oracle_matches_dense_bruteforce(name, fp8, seed):
    if name == "gqa7":
        c = make_case("tiny", seed, Hq=14, Hkv=2, D=128, dtype="bf16",
                      ctx=("fixed", [1, 16, 33, 64]))
    else:
        c = make_case(name, seed, kv="fp8" if fp8 else "same")
    (out, lse), _ = _oracle_case(c)
    K, V = source_rows(c)
    for b in range(c.B):
        o_ref, l_ref = dense_decode(c, b, K, V)
        assert np.abs(out[b] - o_ref.numpy()).max() < 1e-12
        assert np.abs(lse[b] - l_ref.numpy()).max() < 1e-12


def test_empty_sequence_gives_zero_and_minus_inf():
    c = make_case("tiny", 0, ctx=("fixed", [0, 5, 0, 17]))
    (out, lse), _ = _oracle_case(c)
    for b in (0, 2):
        assert np.all(out[b] == 0) and np.all(np.isneginf(lse[b]))
    assert np.all(np.isfinite(out[1]))


def test_closed_form_golden_case():
    vals = {k: float(v) for k, v in _read_golden("closed_form_decode.txt")}
    D, BS = 64, 16
    q = torch.zeros((1, 1, D), dtype=torch.float16)
    q[0, 0, 0] = 8.0
    kc = torch.full((8, 1, BS, D), float("nan"), dtype=torch.float16)
    vc = kc.clone()
    kc[5, 0, :3] = 0
    vc[5, 0, :3] = 0
    for j in range(3):
        kc[5, 0, j, 0] = float(j)
        vc[5, 0, j, j] = 1.0
    tables = np.array([[5, 0]], np.int32)
    out, lse = O.decode(q, kc, vc, tables, np.array([3], np.int32), np.float32(1 / 8))
    for i in range(3):
        assert out[0, 0, i] == pytest.approx(vals[f"out{i}"], abs=1e-14)
    assert np.all(out[0, 0, 3:] == 0)
    assert lse[0, 0] == pytest.approx(vals["lse"], abs=1e-13)


# ---- prefill pins ---------------------------------------------------------

def _prefill_case(seed, L, P, fp8=False, Hq=4, Hkv=2, D=64):
    cfg = dict(B=2, Hq=Hq, Hkv=Hkv, D=D, BS=16, dtype="f16", kv="fp8" if fp8 else "same",
               ctx=("fixed", [20, 33]), pool=("scale", 2.0), partition_tokens=0,
               shared_prefix=None, prefill=(L, P))
    return make_case(cfg, seed)


@pytest.mark.parametrize("L,P,fp8", [(1, 40, False), (37, 0, False), (50, 29, False), (23, 17, True)])
def test_prefill_matches_dense_causal(L, P, fp8):
    c = _prefill_case(8, L, P, fp8)
    kc, vc = O.fill_cache(c)
    pf = c.prefill
    out, lse = O.prefill_chunk(pf.q, kc, vc, pf.block_tables, pf.seq_lens, pf.cu_q_lens,
                               c.scale, c.k_scales, c.v_scales)
    K, V = source_rows(c)
    rows = c.logical_rows(pf.block_tables[0], P + L)
    o_ref, l_ref = dense_attention(pf.q.double(), K[rows], V[rows], np.float64(c.scale),
                                   causal_offset=P)
    assert np.abs(out - o_ref.numpy()).max() < 1e-12
    assert np.abs(lse - l_ref.numpy()).max() < 1e-12


def test_prefill_chunk_of_one_equals_decode():
    c = _prefill_case(9, 1, 70)
    kc, vc = O.fill_cache(c)
    pf = c.prefill
    out, lse = O.prefill_chunk(pf.q, kc, vc, pf.block_tables, pf.seq_lens, pf.cu_q_lens, c.scale)
    out2, lse2 = O.decode(pf.q, kc, vc, pf.block_tables, pf.seq_lens, c.scale)
    assert np.array_equal(out, out2) and np.array_equal(lse, lse2)


def test_prefill_rejects_chunk_longer_than_context():
    c = _prefill_case(9, 5, 3)
    kc, vc = O.fill_cache(c)
    pf = c.prefill
    with pytest.raises(ValueError):
        O.prefill_chunk(pf.q, kc, vc, pf.block_tables, np.array([4], np.int32),
                        pf.cu_q_lens, c.scale)


# ---- generator recipe -----------------------------------------------------

def test_generator_is_seeded_and_poisons_unused_slots():
    a, b = make_case("tiny", 0), make_case("tiny", 0)
    assert np.array_equal(a.block_tables, b.block_tables)
    assert torch.equal(a.q, b.q) and torch.equal(a.fill_k, b.fill_k)
    assert not torch.equal(make_case("tiny", 1).q, a.q)
    assert list(a.seq_lens) == [17, 64, 100, 255]
    k, v = empty_cache(a)
    assert torch.isnan(k[a.poison_block]).all()
    blk = a.tail_slots // 16
    assert (k[blk, :, a.tail_slots % 16, :] == 60).all()
    used = set(a.block_tables.ravel().tolist())
    assert len(used) == 29 + 1                         # 29 owned blocks + poison


def test_shared_prefix_layout_and_mixed_counts():
    c = make_case("mixed", 0)
    assert c.B == 64 and c.prefill.L == 512 and c.prefill.P == 1500
    assert len(c.new_slots) == 576
    sh = c.block_tables[:16, :64]
    assert (sh == sh[0]).all() and (c.seq_lens[:16] >= 1025).all()
    assert len(set(c.fill_slots.tolist()) | set(c.new_slots.tolist())) == \
        len(c.fill_slots) + len(c.new_slots)
