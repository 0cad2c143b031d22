"""head_dim 256 (rows of 512 bytes for 16-bit caches, 256 for E4M3: two or four
TMA boxes per page row) against the oracle: cache writes and rotary writes bit
for bit, decode, prefill and the whole-step varlen call within tolerance.
Blocks below 16 tokens are refused at this head size."""
import numpy as np
import pytest
import torch

import paged_kv_decode_11_gb300 as P
from oracle import oracle as O
from workloads import make_case, empty_cache, rope_cos_sin
from tests.gpu_helpers import (LSE_TOL, assert_close, check_device_ok, dev, oracle_cache,
                               oracle_decode, product_cache, run_decode, run_prefill, scales,
                               tol)

pytestmark = pytest.mark.gpu


@pytest.fixture(scope="module", autouse=True)
def _lib():
    from paged_kv_decode_11_gb300 import build
    build.build()
    P.load()
    O.build()
    torch.cuda.init()
    P.pkv_get_device_error()


CTX = [1, 16, 17, 40, 129, 333, 900]


def _case(kv, dtype, Hq, Hkv, BS=16, seed=40, ctx=CTX, **kw):
    return make_case("tiny", seed, B=len(ctx), BS=BS, Hq=Hq, Hkv=Hkv, D=256, dtype=dtype, kv=kv,
                     ctx=("fixed", ctx), pool=("scale", 1.4), **kw)


@pytest.mark.parametrize("kv,dtype,Hq,Hkv", [("same", "bf16", 8, 1), ("same", "f16", 16, 8),
                                             ("fp8", "bf16", 8, 8), ("fp8", "f16", 16, 2)])
@pytest.mark.parametrize("BS", [16, 32, 64])
@pytest.mark.parametrize("part", [0, 48])
def test_decode_vs_oracle(kv, dtype, Hq, Hkv, BS, part):
    c = _case(kv, dtype, Hq, Hkv, BS)
    kc, vc = product_cache(c)
    out, lse = run_decode(c, kc, vc, partition_tokens=part)
    check_device_ok()
    ko, vo = oracle_cache(c)
    want, wlse = oracle_decode(c, ko, vo)
    assert_close(out, want, tol(c), "D256 decode")
    assert_close(lse, wlse, LSE_TOL, "D256 lse")


@pytest.mark.parametrize("kv", ["same", "fp8"])
def test_cache_write_bit_exact(kv):
    c = _case(kv, "bf16", 8, 2)
    kc, vc = product_cache(c)
    torch.cuda.synchronize()
    check_device_ok()
    ko, vo = oracle_cache(c)
    assert torch.equal(kc.cpu().view(torch.uint8), ko.view(torch.uint8))
    assert torch.equal(vc.cpu().view(torch.uint8), vo.view(torch.uint8))


@pytest.mark.parametrize("rot", [256, 64])
def test_rope_cache_bit_exact(rot):
    c = _case("fp8", "bf16", 8, 2)
    cs = rope_cos_sin(int(c.new_positions.max()) + 1, rot, 10000.0)
    g = torch.Generator().manual_seed(6)
    q = torch.randn((len(c.new_slots), c.Hq, c.D), generator=g).to(c.torch_dtype)
    ks, vs = scales(c)
    kc, vc = empty_cache(c, "cuda")
    qg = dev(q)
    P.rope_reshape_and_cache(qg, dev(c.new_k), dev(c.new_v), kc, vc, dev(c.new_slots),
                             dev(c.new_positions), dev(cs), rot, True, ks, vs)
    torch.cuda.synchronize()
    check_device_ok()
    ko, vo = empty_cache(c, "cpu")
    qo, flags = O.rope_reshape_and_cache(q, c.new_k.cpu().contiguous(), c.new_v.cpu().contiguous(),
                                         ko, vo, c.new_slots, c.new_positions, cs, rot, True,
                                         c.k_scales, c.v_scales)
    assert flags == 0
    assert torch.equal(qg.cpu().view(torch.int16), qo.view(torch.int16))
    assert torch.equal(kc.cpu(), ko) and torch.equal(vc.cpu(), vo)


@pytest.mark.parametrize("L,P_,kv,Hq,Hkv", [(1, 50, "same", 8, 1), (70, 0, "same", 8, 8),
                                            (100, 150, "fp8", 16, 2), (33, 47, "same", 16, 2),
                                            (600, 40, "same", 16, 8),   # 80 tiles: no key split
                                            (200, 330, "same", 4, 4)])  # G = 1, 2-CTA clusters
def test_prefill_vs_oracle(L, P_, kv, Hq, Hkv):
    c = _case(kv, "bf16", Hq, Hkv, ctx=[30, 60], seed=41, prefill=(L, P_))
    kc, vc = product_cache(c)
    out, lse = run_prefill(c, kc, vc)
    check_device_ok()
    ko, vo = oracle_cache(c)
    pf = c.prefill
    want, wlse = O.prefill_chunk(pf.q, ko, vo, pf.block_tables, pf.seq_lens, pf.cu_q_lens,
                                 c.scale, c.k_scales, c.v_scales)
    assert_close(out, want, tol(c), "D256 prefill")
    assert_close(lse, wlse, LSE_TOL, "D256 prefill lse")


def test_varlen_step_vs_oracle():
    from paged_kv_decode_11_gb300.step import MixedStep
    c = _case("same", "bf16", 8, 2, ctx=[90, 300, 17, 1000], seed=42, prefill=(64, 200))
    kc, vc = product_cache(c, write_new=False)
    step = MixedStep.from_case(c, kc, vc, mode="varlen")
    step.run()
    torch.cuda.synchronize()
    check_device_ok()
    ko, vo = oracle_cache(c)
    want, _ = oracle_decode(c, ko, vo)
    assert_close(step.out, want, tol(c), "D256 varlen decode rows")
    pf = c.prefill
    pw, _ = O.prefill_chunk(pf.q.cpu(), ko, vo, pf.block_tables, pf.seq_lens, pf.cu_q_lens,
                            c.scale)
    assert_close(step.prefill_out, pw, tol(c), "D256 varlen chunk rows")


@pytest.mark.parametrize("BS", [1, 8])
def test_token_blocks_are_refused_at_256(BS):
    c = _case("same", "bf16", 8, 2, BS=BS)
    kc, vc = product_cache(c)
    with pytest.raises(P.PkvError):
        run_decode(c, kc, vc)


def test_group_above_8_is_refused_at_256():
    c = _case("same", "bf16", 32, 2)
    kc, vc = product_cache(c)
    with pytest.raises(P.PkvError):
        run_decode(c, kc, vc)
