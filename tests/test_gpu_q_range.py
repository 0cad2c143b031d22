"""bf16 queries beyond the f16 range on E4M3 caches.

An E4M3 cache runs f16 MMAs, so a bf16 query is converted to f16 on the way
in. The kernels scale the query by a power of two first (its largest
magnitude into [2^14, 2^15)) and scale the scores back, which is exact. Two
identities check it, for decode and for both prefill kernels:
  * q * 2^17 with scale * 2^-17, and q * 2^-30 with scale * 2^30, define the
    same scores as (q, scale); the outputs must be bit-identical to the
    unscaled call's (without the prescale the first overflows f16 to inf and
    gives NaN, the second flushes the query to zero and averages V);
  * the same calls agree with the fp64 oracle within the FP8-KV tolerance.
"""
import pytest
import torch

import paged_kv_decode_11_gb300 as P
from oracle import oracle as O
from workloads import make_case
from tests.gpu_helpers import (assert_close, check_device_ok, dev, oracle_cache, oracle_decode,
                               product_cache, scales, tol)

pytestmark = pytest.mark.gpu

FACTORS = [(2.0 ** 17, 2.0 ** -17), (2.0 ** -30, 2.0 ** 30)]


@pytest.fixture(scope="module", autouse=True)
def _lib():
    from paged_kv_decode_11_gb300 import build
    build.build()
    P.load()
    O.build()
    torch.cuda.init()
    P.pkv_get_device_error()


def _decode(c, kc, vc, q, scale, part):
    out = torch.empty_like(q)
    lse = torch.empty(q.shape[:2], dtype=torch.float32, device="cuda")
    ks, vs = scales(c)
    P.paged_attn_decode(out, q, kc, vc, dev(c.block_tables), dev(c.seq_lens), scale,
                        c.max_seq_len, ks, vs, partition_tokens=part, out_lse=lse)
    return out, lse


@pytest.mark.parametrize("Hq,Hkv,D,part", [(32, 8, 128, 0), (8, 2, 64, 64), (16, 1, 128, 32),
                                           (16, 8, 256, 0)])
def test_decode_bf16_q_outside_f16_range_on_e4m3(Hq, Hkv, D, part):
    # contexts of 17 or more: a bf16 output that is a single V row can sit
    # above 4, where bf16's spacing alone exceeds the comparison's 1e-2
    ctx = [17, 33, 100, 300]
    c = make_case("tiny", 21, B=len(ctx), Hq=Hq, Hkv=Hkv, D=D, dtype="bf16", kv="fp8",
                  ctx=("fixed", ctx), pool=("scale", 1.5))
    kc, vc = product_cache(c)
    q = dev(c.q)
    base, base_lse = _decode(c, kc, vc, q, float(c.scale), part)
    check_device_ok()
    ko, vo = oracle_cache(c)
    for fq, fs in FACTORS:
        qs = (q.float() * fq).to(torch.bfloat16)
        assert torch.equal(qs.float(), q.float() * fq)          # the scaling is exact in bf16
        out, lse = _decode(c, kc, vc, qs, float(c.scale) * fs, part)
        check_device_ok()
        assert torch.equal(out, base), f"x{fq}: output differs from the unscaled call"
        assert torch.equal(lse, base_lse)
        want, wlse = O.decode(qs.cpu(), ko, vo, c.block_tables, c.seq_lens, float(c.scale) * fs,
                              c.k_scales, c.v_scales)
        assert_close(out, want, tol(c), f"x{fq} vs oracle")


def _prefill(c, kc, vc, q, scale):
    pf = c.prefill
    out = torch.empty_like(q)
    lse = torch.empty(q.shape[:2], dtype=torch.float32, device="cuda")
    ks, vs = scales(c)
    P.paged_attn_prefill_chunk(out, q, kc, vc, dev(pf.block_tables), dev(pf.seq_lens),
                               dev(pf.cu_q_lens), scale, pf.L, ks, vs, out_lse=lse)
    return out, lse


# D = 128: the tensor-core kernel (one CTA per tile, and the 2-CTA key split);
# D = 256: the warp-MMA kernel, which takes E4M3 caches at that size
@pytest.mark.parametrize("L,P_,Hq,Hkv,D", [(70, 45, 8, 2, 128), (640, 100, 16, 8, 128),
                                           (40, 60, 8, 4, 256)])
def test_prefill_bf16_q_outside_f16_range_on_e4m3(L, P_, Hq, Hkv, D):
    cfg = dict(B=2, Hq=Hq, Hkv=Hkv, D=D, BS=16, dtype="bf16", kv="fp8", ctx=("fixed", [20, 33]),
               pool=("scale", 2.0), partition_tokens=0, shared_prefix=None, prefill=(L, P_))
    c = make_case(cfg, 23)
    kc, vc = product_cache(c)
    q = dev(c.prefill.q)
    base, base_lse = _prefill(c, kc, vc, q, float(c.scale))
    check_device_ok()
    ko, vo = oracle_cache(c)
    pf = c.prefill
    for fq, fs in FACTORS:
        qs = (q.float() * fq).to(torch.bfloat16)
        assert torch.equal(qs.float(), q.float() * fq)
        out, lse = _prefill(c, kc, vc, qs, float(c.scale) * fs)
        check_device_ok()
        assert torch.equal(out, base), f"x{fq}: output differs from the unscaled call"
        assert torch.equal(lse, base_lse)
        want, _ = O.prefill_chunk(qs.cpu(), ko, vo, pf.block_tables, pf.seq_lens, pf.cu_q_lens,
                                  float(c.scale) * fs, c.k_scales, c.v_scales)
        assert_close(out, want, tol(c), f"x{fq} vs oracle")
