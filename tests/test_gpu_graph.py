"""CUDA-graph capture of a whole step. A decode step (cache write + decode
attention, whose split-KV counters reset themselves) and a mixed step (cache
write, then one varlen call, or prefill on a second stream beside decode)
are captured once and replayed with new inputs copied into the captured
buffers. Each replay must
equal an eager run on the same inputs bit for bit, and a sample of the
replayed output must match the oracle."""
import numpy as np
import pytest
import torch

import paged_kv_decode_11_gb300 as P
from oracle import oracle as O
from workloads import make_case
from tests.gpu_helpers import (assert_close, check_device_ok, oracle_cache, oracle_decode,
                               product_cache, tol)

pytestmark = pytest.mark.gpu


@pytest.fixture(scope="module", autouse=True)
def _lib():
    from paged_kv_decode_11_gb300 import build
    build.build()
    P.load()
    O.build()
    torch.cuda.init()
    P.pkv_get_device_error()


def capture(step):
    """Warm the step up on a side stream, then capture one run of it."""
    side = torch.cuda.Stream()
    side.wait_stream(torch.cuda.current_stream())
    with torch.cuda.stream(side):
        step.run()
    torch.cuda.current_stream().wait_stream(side)
    torch.cuda.synchronize()
    g = torch.cuda.CUDAGraph()
    with torch.cuda.graph(g):
        step.run()
    torch.cuda.synchronize()
    return g


def fresh_q(like, seed):
    gen = torch.Generator().manual_seed(seed)
    return torch.randn(like.shape, generator=gen, dtype=torch.float32).to(like.dtype)


@pytest.mark.parametrize("name", ["qwen2.5-7b", "llama3-8b-fp8"])
def test_decode_step_graph_replay_matches_eager(name):
    from paged_kv_decode_11_gb300.step import DecodeStep
    over = {"B": 24} if name == "llama3-8b-fp8" else {}
    c = make_case(name, 0, device="cuda", **over)
    kc, vc = product_cache(c, write_new=False)
    step = DecodeStep.from_case(c, kc, vc)
    g = capture(step)
    for seed in (11, 12):
        q_new = fresh_q(step.q, seed)
        step.q.copy_(q_new.cuda())
        g.replay()
        torch.cuda.synchronize()
        replayed, replayed_lse = step.out.clone(), step.lse.clone()
        step.run()
        torch.cuda.synchronize()
        check_device_ok()
        assert torch.equal(replayed, step.out), "graph replay differs from the eager step"
        assert torch.equal(replayed_lse, step.lse)
    # the replayed output against the oracle on the last q
    sel = [0, c.B // 2, c.B - 1]
    ko, vo = oracle_cache(c, sel)
    c.q = step.q.cpu()
    want, _ = oracle_decode(c, ko, vo, sel=sel)
    assert_close(replayed[torch.as_tensor(sel)], want, tol(c), f"{name} graph replay")


@pytest.mark.parametrize("mode", ["varlen", "streams"])
def test_mixed_step_graph_replay_matches_eager(mode):
    from paged_kv_decode_11_gb300.step import MixedStep
    c = make_case("mixed", 0, device="cuda")
    kc, vc = product_cache(c, write_new=False)
    step = MixedStep.from_case(c, kc, vc, mode=mode)
    g = capture(step)
    d = step.decode
    nd = d.q.shape[0]
    q_new, pq_new = fresh_q(d.q, 21).cuda(), fresh_q(step.pf_q, 22).cuda()
    if mode == "varlen":                       # the step reads its own batched copy
        step.q_all[:nd].copy_(q_new)
        step.q_all[nd:].copy_(pq_new)
    else:
        d.q.copy_(q_new)
        step.pf_q.copy_(pq_new)
    g.replay()
    torch.cuda.synchronize()
    rd, rp = step.out.clone(), step.prefill_out.clone()
    step.run()
    torch.cuda.synchronize()
    check_device_ok()
    as_bytes = lambda t: t.contiguous().view(torch.uint8)
    assert torch.equal(as_bytes(rd), as_bytes(step.out)), "decode rows of the replay differ"
    assert torch.equal(as_bytes(rp), as_bytes(step.prefill_out)), "chunk rows of the replay differ"
    # prefill of the replayed step against the oracle
    ko, vo = oracle_cache(c)
    pf = c.prefill
    pw, _ = O.prefill_chunk(pq_new.cpu(), ko, vo, pf.block_tables, pf.seq_lens, pf.cu_q_lens,
                            c.scale)
    assert_close(rp, pw, tol(c), f"mixed prefill (graph replay, {mode})")


def test_graph_replays_are_deterministic():
    from paged_kv_decode_11_gb300.step import DecodeStep
    c = make_case("long-ctx", 0, device="cuda")
    kc, vc = product_cache(c, write_new=False)
    step = DecodeStep.from_case(c, kc, vc)
    g = capture(step)
    outs = []
    for _ in range(3):
        g.replay()
        torch.cuda.synchronize()
        outs.append(step.out.clone())
    check_device_ok()
    assert all(torch.equal(outs[0], o) for o in outs[1:]), "replays differ"
    assert np.isfinite(outs[0].float().cpu().numpy()).all()
