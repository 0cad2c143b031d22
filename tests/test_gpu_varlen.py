"""paged_attn_varlen: one call over a whole continuous-batching step (decode
sequences first, then prefill chunks) against the oracle, against the two
separate entry points, and under CUDA-graph capture. Decode rows: bit for bit
with an explicit partition size (the same kernel and plan compute them);
with automatic partitions the varlen call plans longer ones (the prefill grid
holds SMs beside it), so they agree within tolerance. Chunk rows within
tolerance: alone, a chunk runs the 128-key-tile kernel and a small chunk's
keys may be split over a cluster of two CTAs, which sums in another order."""
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


def _bits(t):
    return t.contiguous().view(torch.uint8)


@pytest.mark.parametrize("kv,part", [("same", 0), ("fp8", 0), ("same", 512), ("fp8", 1024)])
def test_mixed_step_varlen_vs_oracle_and_two_streams(kv, part):
    from paged_kv_decode_11_gb300.step import MixedStep
    c = make_case("mixed", 0, device="cuda", kv=kv, partition_tokens=part)
    kc, vc = product_cache(c, write_new=False)
    one = MixedStep.from_case(c, kc, vc, mode="varlen")
    one.run()
    torch.cuda.synchronize()
    check_device_ok()
    two = MixedStep.from_case(c, kc, vc, mode="streams")
    two.run()
    torch.cuda.synchronize()
    check_device_ok()
    if part:
        assert torch.equal(_bits(one.out), _bits(two.out)), "decode rows differ between modes"
    else:
        assert_close(one.out, two.out.double().cpu().numpy(), tol(c), "decode rows between modes")
    assert_close(one.prefill_out, two.prefill_out.double().cpu().numpy(), tol(c),
                 "chunk rows between modes")
    sel = [0, 7, 16, 40, 63]
    ko, vo = oracle_cache(c)
    want, wlse = oracle_decode(c, ko, vo, sel=sel)
    assert_close(one.out[torch.as_tensor(sel)], want, tol(c), "varlen decode rows")
    assert_close(one.lse_all[torch.as_tensor(sel)], wlse, LSE_TOL, "varlen decode lse")
    pf = c.prefill
    pw, plse = O.prefill_chunk(pf.q.cpu(), ko, vo, pf.block_tables, pf.seq_lens, pf.cu_q_lens,
                               c.scale, c.k_scales, c.v_scales)
    assert_close(one.prefill_out, pw, tol(c), "varlen chunk rows")
    assert_close(one.prefill_lse, plse, LSE_TOL, "varlen chunk lse")


def _batch(seed, n_dec, chunks, kv="same", BS=16, ctx_dec=None):
    """A batch of n_dec decode sequences and one chunk sequence per (L, P)."""
    rng = np.random.default_rng(seed)
    ctx_dec = list(rng.integers(1, 900, n_dec)) if ctx_dec is None else list(ctx_dec)
    c = make_case("tiny", seed, B=n_dec + len(chunks), BS=BS, Hq=16, Hkv=4, D=128,
                  dtype="bf16", kv=kv, ctx=("fixed", ctx_dec + [L + Pp for L, Pp in chunks]),
                  pool=("scale", 1.3))
    Ls = [1] * n_dec + [L for L, _ in chunks]
    qsl = np.concatenate([[0], np.cumsum(Ls)]).astype(np.int32)
    g = torch.Generator().manual_seed(seed + 1)
    q = torch.randn((int(qsl[-1]), c.Hq, c.D), generator=g).to(torch.bfloat16)
    return c, q, qsl


@pytest.mark.parametrize("n_dec,chunks,kv", [
    (5, [(64, 100), (1, 10), (200, 0)], "same"),
    (0, [(37, 20), (90, 300)], "fp8"),
    (9, [], "fp8"),
    (3, [(16, 16)], "same"),
])
def test_varlen_batch_vs_oracle(n_dec, chunks, kv):
    c, q, qsl = _batch(30 + n_dec, n_dec, chunks, kv)
    kc, vc = product_cache(c)                       # every context token cached
    ks, vs = scales(c)
    out = torch.empty_like(q).cuda()
    lse = torch.empty(q.shape[:2], dtype=torch.float32, device="cuda")
    max_q = max([L for L, _ in chunks], default=1)
    P.paged_attn_varlen(out, dev(q), kc, vc, dev(c.block_tables), dev(c.seq_lens), dev(qsl),
                        n_dec, float(c.scale), max_q, int(c.seq_lens.max()), ks, vs,
                        out_lse=lse)
    torch.cuda.synchronize()
    check_device_ok()
    ko, vo = oracle_cache(c)
    # every row of the batch is causal attention of its token over its own context
    want, wlse = O.prefill_chunk(q, ko, vo, c.block_tables, c.seq_lens, qsl, c.scale,
                                 c.k_scales, c.v_scales)
    assert_close(out, want, tol(c), "varlen rows")
    assert_close(lse, wlse, LSE_TOL, "varlen lse")


@pytest.mark.parametrize("kv", ["same", "fp8"])
def test_varlen_decode_contexts_on_partition_boundaries(kv):
    # beside a chunk the decode CTAs take their work in full-first order:
    # every full partition, then the shorter last ones by decreasing length;
    # contexts that end exactly on a partition boundary have no short one
    ctx_dec = [512, 1024, 1, 513, 1535, 1536, 2048, 700, 16, 17]
    c, q, qsl = _batch(41, len(ctx_dec), [(64, 200)], kv, ctx_dec=ctx_dec)
    kc, vc = product_cache(c)
    ks, vs = scales(c)
    out = torch.empty_like(q).cuda()
    lse = torch.empty(q.shape[:2], dtype=torch.float32, device="cuda")
    P.paged_attn_varlen(out, dev(q), kc, vc, dev(c.block_tables), dev(c.seq_lens), dev(qsl),
                        len(ctx_dec), float(c.scale), 64, int(max(ctx_dec)), ks, vs, out_lse=lse)
    torch.cuda.synchronize()
    check_device_ok()
    ko, vo = oracle_cache(c)
    want, wlse = O.prefill_chunk(q, ko, vo, c.block_tables, c.seq_lens, qsl, c.scale,
                                 c.k_scales, c.v_scales)
    assert_close(out, want, tol(c), "varlen rows")
    assert_close(lse, wlse, LSE_TOL, "varlen lse")


def test_varlen_graph_capture_replays_bit_identically():
    from paged_kv_decode_11_gb300.step import MixedStep
    c = make_case("mixed", 2, device="cuda")
    kc, vc = product_cache(c, write_new=False)
    step = MixedStep.from_case(c, kc, vc, mode="varlen")
    side = torch.cuda.Stream()
    side.wait_stream(torch.cuda.current_stream())
    with torch.cuda.stream(side):
        step.run()
    torch.cuda.current_stream().wait_stream(side)
    torch.cuda.synchronize()
    eager = step.out_all.clone()
    g = torch.cuda.CUDAGraph()
    with torch.cuda.graph(g):
        step.run()
    for _ in range(3):
        g.replay()
        torch.cuda.synchronize()
        assert torch.equal(_bits(step.out_all), _bits(eager))
    check_device_ok()
