"""GPU parity of rope_reshape_and_cache (rotary embedding fused with the cache
write) against the fp64 oracle: rotated queries and every cache byte must be
bit-identical, on the workloads' new tokens and on hand-made tables that
put exact results on and next to 16-bit rounding midpoints."""
import numpy as np
import pytest
import torch

import paged_kv_decode_11_gb300 as P
from oracle import oracle as O
from workloads import make_case, empty_cache, rope_cos_sin
from tests.gpu_helpers import check_device_ok, dev, scales

pytestmark = pytest.mark.gpu


@pytest.fixture(scope="module", autouse=True)
def _lib():
    from paged_kv_decode_11_gb300 import build
    build.build()
    P.load()
    O.build()
    torch.cuda.init()
    P.pkv_get_device_error()


def _queries(case, T, seed):
    g = torch.Generator().manual_seed(seed)
    return torch.randn((T, case.Hq, case.D), generator=g).to(case.torch_dtype)


def _run_both(case, q, cs, rot, neox, slots=None, positions=None):
    """The fused step on the GPU and in the oracle, each on its own empty
    pool. Returns (gpu q, oracle q, gpu caches, oracle caches, oracle flags)."""
    k, v = case.new_k.cpu().contiguous(), case.new_v.cpu().contiguous()
    slots = case.new_slots if slots is None else slots
    positions = case.new_positions if positions is None else positions
    ks, vs = scales(case)
    kc, vc = empty_cache(case, "cuda")
    qg = dev(q)
    P.rope_reshape_and_cache(qg, dev(k), dev(v), kc, vc, dev(np.asarray(slots, np.int64)),
                             dev(np.asarray(positions, np.int64)), dev(cs), rot, neox, ks, vs)
    torch.cuda.synchronize()
    ko, vo = empty_cache(case, "cpu")
    qo, flags = O.rope_reshape_and_cache(q, k, v, ko, vo, slots, positions, cs, rot, neox,
                                         case.k_scales, case.v_scales)
    return qg.cpu(), qo, (kc.cpu(), vc.cpu()), (ko, vo), flags


def _bits(t):
    return t.contiguous().view(torch.uint8)


CASES = [
    ("mixed", {}, 10000.0),
    ("llama3-8b-fp8", {"B": 48}, 500000.0),
    ("qwen2.5-7b", {}, 1000000.0),
    ("tiny", {}, 10000.0),
]


@pytest.mark.parametrize("neox", [True, False])
@pytest.mark.parametrize("name,over,base", CASES)
def test_rope_cache_bit_exact_on_workloads(name, over, base, neox):
    c = make_case(name, 0, device="cpu", **over)
    rot = c.D
    cs = rope_cos_sin(int(c.new_positions.max()) + 1, rot, base)
    q = _queries(c, len(c.new_slots), 3)
    qg, qo, (kc, vc), (ko, vo), flags = _run_both(c, q, cs, rot, neox)
    check_device_ok()
    assert flags == 0
    assert torch.equal(_bits(qg), _bits(qo)), "rotated queries differ"
    assert torch.equal(_bits(kc), _bits(ko)), "key cache differs"
    assert torch.equal(_bits(vc), _bits(vo)), "value cache differs"


@pytest.mark.parametrize("rot", [16, 32, 64])
@pytest.mark.parametrize("kv", ["same", "fp8"])
def test_rope_cache_partial_rotary(rot, kv):
    c = make_case("mixed", 1, device="cpu", kv=kv)
    cs = rope_cos_sin(int(c.new_positions.max()) + 1, rot, 10000.0)
    q = _queries(c, len(c.new_slots), 4)
    for neox in (True, False):
        qg, qo, (kc, vc), (ko, vo), flags = _run_both(c, q, cs, rot, neox)
        check_device_ok()
        assert flags == 0
        assert torch.equal(_bits(qg), _bits(qo))
        assert torch.equal(_bits(kc), _bits(ko)) and torch.equal(_bits(vc), _bits(vo))
        assert torch.equal(_bits(qg[..., rot:]), _bits(q[..., rot:]))


def test_rope_cache_f16_d64_fp8():
    c = make_case("tiny", 2, device="cpu", kv="fp8")
    cs = rope_cos_sin(300, 64, 10000.0)
    q = _queries(c, len(c.new_slots), 5)
    qg, qo, (kc, vc), (ko, vo), _ = _run_both(c, q, cs, 64, True)
    check_device_ok()
    assert torch.equal(_bits(qg), _bits(qo))
    assert torch.equal(_bits(kc), _bits(ko)) and torch.equal(_bits(vc), _bits(vo))


@pytest.mark.parametrize("dtype", ["bf16", "f16"])
def test_rope_results_on_and_next_to_rounding_midpoints(dtype):
    """Table rows that make x1 c an exact 16-bit midpoint and x2 s a tiny
    term of either sign, down to below the double's resolution: the result
    then hangs on the last rounding steps (the fp32 path cannot decide and
    the double path takes over), and must still equal the oracle's."""
    c = make_case("tiny", 0, device="cpu", dtype=dtype)
    rot, T = 16, 12
    half = rot // 2
    ulp16 = 2.0 ** -7 if dtype == "bf16" else 2.0 ** -10
    mid = np.float32(1.0 + ulp16 / 2)                 # halfway between 1 and the next value
    tiny = [2.0 ** -30, -(2.0 ** -30), 2.0 ** -60, -(2.0 ** -60), 0.0, 2.0 ** -24,
            -(2.0 ** -24), 2.0 ** -100, 3 * 2.0 ** -25, -(2.0 ** -80), 2.0 ** -126, 2.0 ** -149]
    cs = np.zeros((T, rot), np.float32)
    for p in range(T):
        cs[p, :half] = mid
        cs[p, half:] = np.float32(tiny[p])
    c.new_k = torch.ones((T, c.Hkv, c.D)).to(c.torch_dtype)
    c.new_k[:, :, half:rot] = torch.tensor([1.0, -1.0] * (half // 2)).to(c.torch_dtype)
    c.new_v = torch.zeros((T, c.Hkv, c.D)).to(c.torch_dtype)
    c.new_slots = np.arange(T, dtype=np.int64) * 3
    c.new_positions = np.arange(T, dtype=np.int64)
    q = torch.ones((T, c.Hq, c.D)).to(c.torch_dtype)
    q[:, :, half:rot] = torch.tensor([-1.0, 1.0] * (half // 2)).to(c.torch_dtype)
    for neox in (True, False):
        qg, qo, (kc, vc), (ko, vo), flags = _run_both(c, q.clone(), cs, rot, neox)
        check_device_ok()
        assert flags == 0
        assert torch.equal(_bits(qg), _bits(qo)), f"queries differ (neox={neox})"
        assert torch.equal(_bits(kc), _bits(ko)), f"key cache differs (neox={neox})"
    # the double-rounding tie: x1 c at the midpoint -+ 2^-60 rounds (in
    # double) to the midpoint itself, which ties to the even value 1.0
    assert qo[2, 0, 0].item() == 1.0 and qg[2, 0, 0].item() == 1.0


def test_rope_cache_skips_and_flags():
    c = make_case("tiny", 3, device="cpu")
    T = len(c.new_slots)
    cs = rope_cos_sin(256, c.D, 10000.0)
    q = _queries(c, T, 6)
    pos = c.new_positions.copy()
    slots = c.new_slots.copy()
    slots[0] = -1                                     # not cached, query still rotated
    pos[1] = 256                                      # outside the table
    qg, qo, (kc, vc), (ko, vo), flags = _run_both(c, q, cs, c.D, True, slots, pos)
    assert P.pkv_get_device_error() == 0x20
    assert flags == 2
    assert torch.equal(_bits(qg), _bits(qo))
    assert torch.equal(_bits(qg[1]), _bits(q[1]))     # left as it was
    assert not torch.equal(_bits(qg[0]), _bits(q[0]))
    assert torch.equal(_bits(kc), _bits(ko)) and torch.equal(_bits(vc), _bits(vo))
    # a slot outside the pool
    slots = c.new_slots.copy()
    slots[2] = c.num_blocks * c.BS
    qg, qo, (kc, vc), (ko, vo), flags = _run_both(c, q, cs, c.D, True, slots)
    assert P.pkv_get_device_error() == 0x2
    assert flags == 1
    assert torch.equal(_bits(kc), _bits(ko)) and torch.equal(_bits(vc), _bits(vo))


def test_rope_cache_then_decode_matches_oracle_attention():
    """The fused step feeding decode: attention over the rotated cache with
    the rotated queries equals the oracle's attention over its own."""
    from tests.gpu_helpers import assert_close, tol
    c = make_case("qwen2.5-7b", 4, device="cpu")
    cs = rope_cos_sin(int(c.new_positions.max()) + 1, c.D, 1000000.0)
    ks, vs = scales(c)
    kc, vc = empty_cache(c, "cuda")
    P.reshape_and_cache(dev(c.fill_k), dev(c.fill_v), kc, vc, dev(c.fill_slots), ks, vs)
    qg = dev(c.q)
    P.rope_reshape_and_cache(qg, dev(c.new_k), dev(c.new_v), kc, vc, dev(c.new_slots),
                             dev(c.new_positions), dev(cs), c.D, True, ks, vs)
    out = torch.empty_like(qg)
    P.paged_attn_decode(out, qg, kc, vc, dev(c.block_tables), dev(c.seq_lens), float(c.scale),
                        c.max_seq_len, ks, vs)
    torch.cuda.synchronize()
    check_device_ok()
    ko, vo = empty_cache(c, "cpu")
    assert O.reshape_and_cache(c.fill_k.cpu().contiguous(), c.fill_v.cpu().contiguous(), ko, vo,
                               c.fill_slots, c.k_scales, c.v_scales) == 0
    qo, flags = O.rope_reshape_and_cache(c.q.cpu().contiguous(), c.new_k.cpu().contiguous(),
                                         c.new_v.cpu().contiguous(), ko, vo, c.new_slots,
                                         c.new_positions, cs, c.D, True)
    assert flags == 0
    sel = [0, 9, 31]
    want, _ = O.decode(qo, ko, vo, c.block_tables, c.seq_lens, c.scale, sel=sel)
    assert_close(out[torch.as_tensor(sel)], want, tol(c), "decode after fused rotary write")
