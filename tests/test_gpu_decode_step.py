"""paged_attn_decode_step: the cache write of each sequence's new token and
decode attention in one call, the attention kernel starting before the write
has finished. Through the C ABI: the cache it leaves and the outputs are
bit-identical to reshape_and_cache followed by paged_attn_decode, and agree
with the fp64 oracle."""
import numpy as np
import pytest
import torch

import paged_kv_decode_11_gb300 as P
from oracle import oracle as O
from workloads import make_case
from tests.gpu_helpers import (LSE_TOL, assert_close, check_device_ok, dev, oracle_cache,
                               oracle_decode, product_cache, scales, tol)

pytestmark = pytest.mark.gpu


@pytest.fixture(scope="module", autouse=True)
def _lib():
    from paged_kv_decode_11_gb300 import build
    build.build()
    P.load()
    O.build()
    torch.cuda.init()
    P.pkv_get_device_error()


def _both(c, part=0):
    """(cache, out, lse) after the one-call step, and after the two calls."""
    ks, vs = scales(c)
    q = dev(c.q)
    bt, sl = dev(c.block_tables), dev(c.seq_lens)
    nk, nv, ns = dev(c.new_k[:c.B]), dev(c.new_v[:c.B]), dev(c.new_slots[:c.B])
    res = []
    for one_call in (True, False):
        kc, vc = product_cache(c, write_new=False)
        out = torch.empty_like(q)
        lse = torch.empty(q.shape[:2], dtype=torch.float32, device="cuda")
        if one_call:
            P.paged_attn_decode_step(nk, nv, ns, out, q, kc, vc, bt, sl, float(c.scale),
                                     c.max_seq_len, ks, vs, partition_tokens=part, out_lse=lse)
        else:
            P.reshape_and_cache(nk, nv, kc, vc, ns, ks, vs)
            P.paged_attn_decode(out, q, kc, vc, bt, sl, float(c.scale), c.max_seq_len, ks, vs,
                                partition_tokens=part, out_lse=lse)
        torch.cuda.synchronize()
        check_device_ok()
        res.append((kc, vc, out, lse))
    return res


@pytest.mark.parametrize("name,over,part", [
    ("tiny", {}, 0),
    ("tiny", dict(kv="fp8", dtype="bf16", D=128, Hq=32, Hkv=8,
                  ctx=("fixed", [17, 2048, 333, 4100])), 0),
    ("tiny", dict(dtype="bf16", D=128, Hq=28, Hkv=4, ctx=("fixed", [16, 1500, 700, 33])), 0),
    ("tiny", dict(kv="fp8", dtype="bf16", D=128, Hq=32, Hkv=8,
                  ctx=("fixed", [17, 2048, 333, 4100])), 512),
])
def test_decode_step_equals_write_then_decode(name, over, part):
    c = make_case(name, 31, pool=("scale", 1.5), **over)
    (k1, v1, o1, l1), (k2, v2, o2, l2) = _both(c, part)
    # byte for byte (the pools hold NaN poison blocks)
    assert torch.equal(k1.view(torch.uint8), k2.view(torch.uint8))
    assert torch.equal(v1.view(torch.uint8), v2.view(torch.uint8))
    assert torch.equal(o1, o2) and torch.equal(l1, l2)
    ko, vo = oracle_cache(c)
    want, wlse = oracle_decode(c, ko, vo)
    assert_close(o1, want, tol(c), "step out")
    assert_close(l1, wlse, LSE_TOL, "step lse")


def test_decode_step_full_size_llama_sampled():
    c = make_case("llama3-8b-fp8", 0, device="cuda")
    (k1, v1, o1, l1), (_, _, o2, l2) = _both(c)
    assert torch.equal(o1, o2) and torch.equal(l1, l2)
    sel = [0, 9, 64, 127]
    ko, vo = oracle_cache(c, seqs=sel)
    want, wlse = oracle_decode(c, ko, vo, sel=sel)
    idx = torch.as_tensor(sel)
    assert_close(o1[idx], want, tol(c), "llama step out")
    assert_close(l1[idx], wlse, LSE_TOL, "llama step lse")
