"""Block sizes 32 and 64 (a block holds 2 or 4 pages of 16 tokens per KV
head): cache writes bit-exact against the oracle, decode and prefill within
tolerance of it, and decode bit-identical across block sizes on the same
logical workload (the kernels walk the same 16-token pages in the same
order whatever the block size)."""
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


CTX = [1, 15, 16, 17, 31, 32, 33, 63, 64, 65, 130, 300, 700]


def _case(BS, kv="same", dtype="bf16", Hq=8, Hkv=2, D=128, seed=21, ctx=CTX):
    return make_case("tiny", seed, B=len(ctx), BS=BS, Hq=Hq, Hkv=Hkv, D=D, dtype=dtype, kv=kv,
                     ctx=("fixed", ctx), pool=("scale", 1.5))


@pytest.mark.parametrize("BS", [32, 64])
@pytest.mark.parametrize("kv", ["same", "fp8"])
def test_cache_write_bit_exact(BS, kv):
    c = _case(BS, kv)
    kc, vc = product_cache(c)
    torch.cuda.synchronize()
    check_device_ok()
    ko, vo = oracle_cache(c)
    assert torch.equal(kc.cpu().view(torch.uint8), ko.view(torch.uint8))
    assert torch.equal(vc.cpu().view(torch.uint8), vo.view(torch.uint8))


@pytest.mark.parametrize("BS", [32, 64])
@pytest.mark.parametrize("kv,dtype,Hq,Hkv,D", [("same", "bf16", 8, 2, 128),
                                               ("fp8", "bf16", 32, 8, 128),
                                               ("same", "f16", 7, 7, 64),
                                               ("fp8", "f16", 14, 2, 64)])
@pytest.mark.parametrize("part", [0, 16, 48])
def test_decode_vs_oracle(BS, kv, dtype, Hq, Hkv, D, part):
    c = _case(BS, kv, dtype, Hq, Hkv, D)
    kc, vc = product_cache(c)
    out, lse = run_decode(c, kc, vc, partition_tokens=part)
    check_device_ok()
    ko, vo = oracle_cache(c)
    want, wlse = oracle_decode(c, ko, vo)
    assert_close(out, want, tol(c), f"BS{BS} decode")
    assert_close(lse, wlse, LSE_TOL, f"BS{BS} lse")


@pytest.mark.parametrize("kv", ["same", "fp8"])
@pytest.mark.parametrize("part", [0, 32])
def test_decode_bit_identical_across_block_sizes(kv, part):
    outs = []
    for BS in (16, 32, 64):
        c = _case(BS, kv, seed=22)
        kc, vc = product_cache(c)
        out, lse = run_decode(c, kc, vc, partition_tokens=part)
        check_device_ok()
        outs.append((out.cpu(), lse.cpu()))
    for o, l in outs[1:]:
        assert torch.equal(o, outs[0][0]) and torch.equal(l, outs[0][1])


@pytest.mark.parametrize("BS", [32, 64])
@pytest.mark.parametrize("L,P_,kv", [(1, 40, "same"), (45, 0, "same"), (100, 77, "fp8"),
                                     (129, 130, "same")])
def test_prefill_vs_oracle(BS, L, P_, kv):
    c = make_case("tiny", 23, B=2, BS=BS, Hq=8, Hkv=2, D=128, dtype="bf16", kv=kv,
                  ctx=("fixed", [40, 70]), pool=("scale", 1.5), prefill=(L, P_))
    kc, vc = product_cache(c)
    out, lse = run_prefill(c, kc, vc)
    check_device_ok()
    ko, vo = oracle_cache(c)
    pf = c.prefill
    want, wlse = O.prefill_chunk(pf.q, ko, vo, pf.block_tables, pf.seq_lens, pf.cu_q_lens,
                                 c.scale, c.k_scales, c.v_scales)
    assert_close(out, want, tol(c), f"BS{BS} prefill")
    assert_close(lse, wlse, LSE_TOL, f"BS{BS} prefill lse")


@pytest.mark.parametrize("BS", [1, 32, 64])
def test_rope_cache_bit_exact(BS):
    c = _case(BS, "fp8")
    cs = rope_cos_sin(int(c.new_positions.max()) + 1, c.D, 10000.0)
    g = torch.Generator().manual_seed(5)
    q = torch.randn((len(c.new_slots), c.Hq, c.D), generator=g).to(c.torch_dtype)
    ks, vs = scales(c)
    kc, vc = empty_cache(c, "cuda")
    qg = dev(q)
    P.rope_reshape_and_cache(qg, dev(c.new_k), dev(c.new_v), kc, vc, dev(c.new_slots),
                             dev(c.new_positions), dev(cs), c.D, True, ks, vs)
    torch.cuda.synchronize()
    check_device_ok()
    ko, vo = empty_cache(c, "cpu")
    qo, flags = O.rope_reshape_and_cache(q, c.new_k.cpu().contiguous(), c.new_v.cpu().contiguous(),
                                         ko, vo, c.new_slots, c.new_positions, cs, c.D, True,
                                         c.k_scales, c.v_scales)
    assert flags == 0
    assert torch.equal(qg.cpu().view(torch.int16), qo.view(torch.int16))
    assert torch.equal(kc.cpu(), ko) and torch.equal(vc.cpu(), vo)


def test_decode_flags_block_id_past_pool_with_block_size_32():
    c = _case(32)
    kc, vc = product_cache(c)
    bt = c.block_tables.copy()
    bt[5, 0] = c.num_blocks                            # one past the pool
    out, _ = run_decode(c, kc, vc, block_tables=bt)
    assert P.pkv_get_device_error() & 0x1


# ---- blocks smaller than a page: rows gathered per token ------------------------------

@pytest.mark.parametrize("BS", [1, 2, 8])
@pytest.mark.parametrize("kv,dtype,Hq,Hkv,D", [("same", "bf16", 8, 2, 128),
                                               ("fp8", "bf16", 32, 8, 128),
                                               ("same", "f16", 12, 4, 64),
                                               ("fp8", "f16", 16, 1, 64)])
@pytest.mark.parametrize("part", [0, 48])
def test_gather_decode_vs_oracle(BS, kv, dtype, Hq, Hkv, D, part):
    c = _case(BS, kv, dtype, Hq, Hkv, D)
    kc, vc = product_cache(c)
    out, lse = run_decode(c, kc, vc, partition_tokens=part)
    check_device_ok()
    ko, vo = oracle_cache(c)
    want, wlse = oracle_decode(c, ko, vo)
    assert_close(out, want, tol(c), f"BS{BS} decode")
    assert_close(lse, wlse, LSE_TOL, f"BS{BS} lse")


@pytest.mark.parametrize("BS", [1, 8])
@pytest.mark.parametrize("kv", ["same", "fp8"])
def test_gather_cache_write_bit_exact(BS, kv):
    c = _case(BS, kv)
    kc, vc = product_cache(c)
    torch.cuda.synchronize()
    check_device_ok()
    ko, vo = oracle_cache(c)
    assert torch.equal(kc.cpu().view(torch.uint8), ko.view(torch.uint8))
    assert torch.equal(vc.cpu().view(torch.uint8), vo.view(torch.uint8))


@pytest.mark.parametrize("kv", ["same", "fp8"])
def test_decode_bit_identical_within_each_page_path(kv):
    # blocks below a page are gathered row by row (the warps of a CTA take
    # its partition's pages in turn), blocks of a page or more are read page
    # by page by TMA (each warp reduces a partition of its own): each path
    # walks the same 16-token pages in the same order for every block size,
    # so within a path the results are bit-identical; both paths agree with
    # the oracle
    outs = {}
    for BS in (1, 4, 16, 32, 64):
        c = _case(BS, kv)
        kc, vc = product_cache(c)
        out, lse = run_decode(c, kc, vc, partition_tokens=64)
        check_device_ok()
        outs[BS] = (out.cpu(), lse.cpu())
        ko, vo = oracle_cache(c)
        want, wlse = oracle_decode(c, ko, vo)
        assert_close(out, want, tol(c), f"BS {BS} out")
        assert_close(lse, wlse, LSE_TOL, f"BS {BS} lse")
    for fam in ((1, 4), (16, 32, 64)):
        for bs in fam[1:]:
            assert torch.equal(outs[bs][0], outs[fam[0]][0]), f"BS {bs} vs {fam[0]}"
            assert torch.equal(outs[bs][1], outs[fam[0]][1])


def test_gather_decode_flags_bad_block_id():
    c = _case(1)
    kc, vc = product_cache(c)
    bt = c.block_tables.copy()
    bt[7, 3] = -2
    run_decode(c, kc, vc, block_tables=bt)
    assert P.pkv_get_device_error() & 0x1


def test_prefill_refuses_blocks_below_a_page():
    c = make_case("tiny", 25, B=2, BS=8, Hq=8, Hkv=2, D=128, dtype="bf16", kv="same",
                  ctx=("fixed", [40, 70]), pool=("scale", 1.5), prefill=(20, 30))
    kc, vc = product_cache(c)
    with pytest.raises(P.PkvError):
        run_prefill(c, kc, vc)


# ---- slots past a context hold garbage: weight 0 must stay 0 ------------------------

def _poison_tails(c, kc, vc):
    ts = torch.as_tensor(c.tail_slots)
    blk, off = (ts // c.BS).cuda(), (ts % c.BS).cuda()
    if c.kv_fp8:
        kc[blk, :, off, :] = 0x7F                       # E4M3 NaN
        vc[blk, :, off, :] = 0x7F
    else:
        kc[blk, :, off, :] = float("nan")
        vc[blk, :, off, :] = float("inf")
    return len(c.tail_slots)


@pytest.mark.parametrize("BS", [16, 32])
@pytest.mark.parametrize("kv", ["same", "fp8"])
def test_decode_ignores_nan_past_the_context(BS, kv):
    c = _case(BS, kv, seed=26)
    kc, vc = product_cache(c)
    assert _poison_tails(c, kc, vc) > 0
    for part in (0, 16, 48):
        out, lse = run_decode(c, kc, vc, partition_tokens=part)
        check_device_ok()
        assert torch.isfinite(out.float()).all()
    ko, vo = oracle_cache(c)
    want, _ = oracle_decode(c, ko, vo)
    assert_close(out, want, tol(c), f"BS{BS} decode with poisoned tails")


@pytest.mark.parametrize("kv", ["same", "fp8"])
def test_prefill_ignores_nan_past_the_context(kv):
    c = make_case("tiny", 27, B=2, BS=16, Hq=8, Hkv=2, D=128, dtype="bf16", kv=kv,
                  ctx=("fixed", [40, 70]), pool=("scale", 1.5), prefill=(37, 50))
    kc, vc = product_cache(c)
    assert _poison_tails(c, kc, vc) > 0
    out, lse = run_prefill(c, kc, vc)
    check_device_ok()
    assert torch.isfinite(out.float()).all()
    ko, vo = oracle_cache(c)
    pf = c.prefill
    want, _ = O.prefill_chunk(pf.q, ko, vo, pf.block_tables, pf.seq_lens, pf.cu_q_lens,
                              c.scale, c.k_scales, c.v_scales)
    assert_close(out, want, tol(c), "prefill with poisoned tails")
