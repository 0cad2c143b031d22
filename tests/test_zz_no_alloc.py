"""paged_attn_decode_noalloc: decode attention for callers that cannot
allocate device memory (an engine whose planner owns all of HBM, a loop that
cannot afford cudaMalloc's device synchronisation, a C host without an
allocator). Its scratch is the library's fixed device array, so these tests
check, through the C ABI, that it returns what paged_attn_decode returns with
a caller workspace, and what the fp64 oracle returns, on two calls in a row
with different shapes (the shared array keeps the previous call's contents);
that paged_attn_decode_noalloc_reset gives the array back clean; and that
sizes needing more scratch than the array holds are refused before any
launch.

This file is collected last on purpose, and works alone in a fresh process."""
import pytest
import torch

import paged_kv_decode_11_gb300 as P
from oracle import oracle as O
from workloads import make_case
from tests.gpu_helpers import (LSE_TOL, assert_close, dev, oracle_cache, oracle_decode,
                               product_cache, scales, tol)

pytestmark = pytest.mark.gpu


@pytest.fixture(scope="module", autouse=True)
def _lib():
    from paged_kv_decode_11_gb300 import build
    build.build()
    P.load()
    O.build()
    torch.cuda.init()
    P.pkv_get_device_error()


def _both(case, partition_tokens):
    kc, vc = product_cache(case)
    ks, vs = scales(case)
    q = dev(case.q)
    bt, sl = dev(case.block_tables), dev(case.seq_lens)
    ref, ref_lse = torch.empty_like(q), torch.empty(q.shape[:2], device="cuda")
    P.paged_attn_decode(ref, q, kc, vc, bt, sl, float(case.scale), case.max_seq_len, ks, vs,
                        partition_tokens=partition_tokens, out_lse=ref_lse)
    got, got_lse = torch.full_like(q, float("nan")), torch.full_like(ref_lse, float("nan"))
    P.paged_attn_decode_noalloc(got, q, kc, vc, bt, sl, float(case.scale), case.max_seq_len, ks,
                                vs, partition_tokens=partition_tokens, out_lse=got_lse)
    torch.cuda.synchronize()
    assert P.pkv_get_device_error() == 0
    return ref, ref_lse, got, got_lse


def _vs_oracle(case, got, got_lse):
    ko, vo = oracle_cache(case)
    want, wlse = oracle_decode(case, ko, vo)
    assert_close(got, want, tol(case), f"{case.name} noalloc vs oracle")
    assert_close(got_lse, wlse, LSE_TOL, f"{case.name} noalloc lse vs oracle")


def test_noalloc_matches_workspace_decode_on_two_calls_in_a_row():
    first = make_case("tiny", 11, kv="fp8", ctx=("fixed", [17, 300, 1, 700]),
                      pool=("blocks", 128))
    second = make_case("tiny", 12, Hq=28, Hkv=4, D=128, dtype="bf16", B=6,
                       ctx=("fixed", [40, 513, 0, 129, 1000, 16]), pool=("scale", 1.5))
    for case, part in ((first, 64), (second, 0)):
        ref, ref_lse, got, got_lse = _both(case, part)
        err = (got.double() - ref.double()).abs().max().item()
        assert err <= tol(case), f"{case.name}: max abs diff {err:.2e}"
        fin = torch.isfinite(ref_lse)
        assert torch.equal(fin, torch.isfinite(got_lse))
        assert (got_lse[fin] - ref_lse[fin]).abs().max().item() <= 1e-3
        _vs_oracle(case, got, got_lse)


def test_noalloc_reset_then_decode_matches_the_oracle():
    # the reset clears the whole array (counters and partials); a decode right
    # after it starts from zero counters and returns the oracle's result
    case = make_case("tiny", 13, kv="fp8", dtype="bf16", D=128, Hq=32, Hkv=8,
                     ctx=("fixed", [17, 64, 2000, 333]), pool=("scale", 1.5))
    kc, vc = product_cache(case)
    ks, vs = scales(case)
    q = dev(case.q)
    P.paged_attn_decode_noalloc_reset()
    for part in (0, 32):
        got = torch.full_like(q, float("nan"))
        got_lse = torch.full(q.shape[:2], float("nan"), device="cuda")
        P.paged_attn_decode_noalloc(got, q, kc, vc, dev(case.block_tables), dev(case.seq_lens),
                                    float(case.scale), case.max_seq_len, ks, vs,
                                    partition_tokens=part, out_lse=got_lse)
        torch.cuda.synchronize()
        assert P.pkv_get_device_error() == 0
        _vs_oracle(case, got, got_lse)
        P.paged_attn_decode_noalloc_reset()


def test_noalloc_refuses_sizes_beyond_its_scratch():
    need = P.paged_attn_decode_workspace_size(4096, 32, 8, 128, 65536, 256)
    assert need > (32 << 20)
    st = P.load().paged_attn_decode_noalloc(None, None, 1, None, None, 1, None, None, 4096, 32, 8,
                                            128, 16, 4096, 1 << 20, 65536, 0.1, None, None, 256,
                                            None, None)
    assert st == 3   # PKV_ERR_WORKSPACE, nothing launched
