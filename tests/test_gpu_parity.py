"""GPU parity: the CUDA path (through the C ABI) against the fp64 oracle on the
same seeded inputs. Cache writes are compared byte for byte; attention
outputs within the stated max-abs tolerances."""
import numpy as np
import pytest
import torch

import paged_kv_decode_11_gb300 as P
from oracle import oracle as O
from workloads import make_case, empty_cache
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
    P.pkv_get_device_error()          # start from a clear error word


# ---- reshape_and_cache: bit exact ------------------------------------------

@pytest.mark.parametrize("dtype,kv,D", [("f16", "same", 64), ("bf16", "same", 128),
                                        ("bf16", "fp8", 128), ("f16", "fp8", 64),
                                        ("bf16", "fp8", 64)])
def test_reshape_and_cache_bit_exact(dtype, kv, D):
    c = make_case("tiny", 1, dtype=dtype, kv=kv, D=D, ctx=("fixed", [1, 16, 17, 255]))
    kc, vc = product_cache(c)
    ko, vo = oracle_cache(c)
    check_device_ok()
    for g, o in ((kc, ko), (vc, vo)):
        gb = g.cpu().view(torch.uint8).numpy()
        ob = o.view(torch.uint8).numpy()
        assert np.array_equal(gb, ob), f"{(gb != ob).sum()} bytes differ"


def test_reshape_and_cache_skips_negative_slots_and_flags_bad_ones():
    c = make_case("tiny", 2, kv="fp8", dtype="bf16", D=128)
    kc, vc = empty_cache(c, "cuda")
    before = kc.clone()
    ks, vs = scales(c)
    slots = torch.tensor([-1, -5, c.num_blocks * 16, c.num_blocks * 16 + 3], dtype=torch.int64)
    k = dev(c.new_k[:4])
    P.reshape_and_cache(k, k, kc, vc, dev(slots), ks, vs)
    bits = P.pkv_get_device_error()
    assert bits == 0x2
    assert torch.equal(kc, before)


def test_fp8_encode_edge_values_bit_exact():
    # saturation, ties, subnormals, signed zero: every E4M3 code value, the
    # midpoints between neighbours, and values beyond +-448
    codes = torch.arange(0, 256, dtype=torch.int32)
    vals = np.array([O.e4m3_value(int(x)) for x in codes])
    fin = np.sort(np.unique(vals[np.isfinite(vals)]))
    mids = (fin[1:] + fin[:-1]) / 2
    extra = np.array([449.0, 464.0, 500.0, 1e6, -1e6, 2.0 ** -11, -2.0 ** -11, 2.0 ** -10,
                      -0.0, 0.0, 3.0e-8])
    x = np.concatenate([fin, mids, extra]).astype(np.float32)
    D, Hkv = 64, 1
    T = -(-len(x) // D)
    xs = np.zeros(T * D, np.float32)
    xs[:len(x)] = x
    # the values pass through bf16 sources exactly only if representable; use
    # f16, which holds every E4M3 value and midpoint in range
    src = torch.from_numpy(xs).to(torch.float16).view(T, Hkv, D)
    nb = -(-T // 16) + 1
    kc = torch.zeros((nb, Hkv, 16, D), dtype=torch.uint8)
    vc = kc.clone()
    ks = np.array([1.0], np.float32)
    slots = np.arange(T, dtype=np.int64)
    O.reshape_and_cache(src, src, kc, vc, slots, ks, ks)
    kg = torch.zeros_like(kc).cuda()
    vg = torch.zeros_like(kg)
    P.reshape_and_cache(dev(src), dev(src), kg, vg, dev(slots), dev(ks), dev(ks))
    check_device_ok()
    assert torch.equal(kg.cpu(), kc)


# ---- decode -------------------------------------------------------------------

def _decode_vs_oracle(c, partition_tokens=None, sel=None):
    kc, vc = product_cache(c)
    out, lse = run_decode(c, kc, vc, partition_tokens=partition_tokens)
    check_device_ok()
    ko, vo = oracle_cache(c, seqs=sel)
    want, wlse = oracle_decode(c, ko, vo, sel=sel)
    idx = slice(None) if sel is None else torch.as_tensor(sel)
    e = assert_close(out[idx], want, tol(c), f"{c.name} out")
    assert_close(lse[idx], wlse, LSE_TOL, f"{c.name} lse")
    return e


@pytest.mark.parametrize("seed", [0, 1, 2])
def test_decode_tiny(seed):
    _decode_vs_oracle(make_case("tiny", seed))


@pytest.mark.parametrize("part", [16, 48, 64, 256])
@pytest.mark.parametrize("kv", ["same", "fp8"])
def test_decode_forced_partitions(part, kv):
    c = make_case("tiny", 3, kv=kv, ctx=("fixed", [17, 64, 100, 700]), pool=("blocks", 128))
    _decode_vs_oracle(c, partition_tokens=part)


SHAPES = [
    # (D, Hq, Hkv, dtype, kv)
    (64, 8, 2, "f16", "same"), (128, 8, 8, "bf16", "same"), (128, 28, 4, "bf16", "same"),
    (128, 32, 8, "bf16", "fp8"), (128, 16, 1, "f16", "fp8"), (64, 16, 2, "bf16", "fp8"),
    (128, 32, 2, "f16", "same"), (64, 12, 12, "bf16", "same"), (128, 14, 2, "bf16", "fp8"),
    (64, 32, 2, "bf16", "fp8"),
]


@pytest.mark.parametrize("D,Hq,Hkv,dtype,kv", SHAPES)
@pytest.mark.parametrize("part", [0, 32])
def test_decode_shape_sweep(D, Hq, Hkv, dtype, kv, part):
    ctx = [1, 15, 16, 17, 31, 33, 130, 300]
    c = make_case("tiny", 4, B=len(ctx), Hq=Hq, Hkv=Hkv, D=D, dtype=dtype, kv=kv,
                  ctx=("fixed", ctx), pool=("scale", 1.5))
    _decode_vs_oracle(c, partition_tokens=part)


@pytest.mark.parametrize("extra", [0, 1])
@pytest.mark.parametrize("kv", ["same", "fp8"])
def test_decode_automatic_plan_either_side_of_one_cta_per_sm(extra, kv):
    # automatic partitions: with (sequence, KV head) units at most one per SM
    # (and contexts up to 4096 tokens) the planner takes the whole-context
    # 8-warp CTAs; one sequence more and it splits contexts into partitions
    # merged across CTAs
    sms = torch.cuda.get_device_properties(0).multi_processor_count
    Hkv = 8
    B = sms // Hkv + extra
    rng = np.random.default_rng(11)
    ctx = [int(x) for x in rng.integers(1, 1500, size=B)]
    ctx[:4] = [1, 16, 17, 1499]
    c = make_case("tiny", 5, B=B, Hq=16, Hkv=Hkv, D=128, dtype="bf16", kv=kv,
                  ctx=("fixed", ctx), pool=("scale", 1.25))
    _decode_vs_oracle(c, partition_tokens=0)


@pytest.mark.parametrize("kv", ["same", "fp8"])
def test_decode_merge_in_several_chunks(kv):
    # G = 16 at D = 128: one partition's partial is 16 rows of 128 fp32, so the
    # merging CTA's shared memory holds a few partitions at a time and a head's
    # 16 CTA partials (16-token partitions, 4 per CTA, 1000-token contexts)
    # arrive in several bulk-copy rounds
    ctx = [1000, 999, 1, 64, 65, 700]
    c = make_case("tiny", 6, B=len(ctx), Hq=32, Hkv=2, D=128, dtype="bf16", kv=kv,
                  ctx=("fixed", ctx), pool=("scale", 1.5))
    _decode_vs_oracle(c, partition_tokens=16)


def test_decode_empty_sequences():
    c = make_case("tiny", 5, ctx=("fixed", [0, 40, 0, 1]))
    kc, vc = product_cache(c)
    out, lse = run_decode(c, kc, vc, partition_tokens=16)
    check_device_ok()
    for b in (0, 2):
        assert torch.all(out[b] == 0) and torch.all(torch.isneginf(lse[b]))
    ko, vo = oracle_cache(c)
    want, wlse = oracle_decode(c, ko, vo)
    assert_close(out, want, tol(c), "out")


@pytest.mark.parametrize("kv", ["same", "fp8"])
def test_decode_length_one_is_v_row_bit_exact(kv):
    c = make_case("tiny", 6, ctx=("fixed", [1, 1, 1, 1]), kv=kv)
    kc, vc = product_cache(c)
    out, _ = run_decode(c, kc, vc)
    ko, vo = oracle_cache(c)
    want, _ = oracle_decode(c, ko, vo)
    # one token: p = 1 exactly, so out is the (dequantised) V row, rounded once
    ref = torch.from_numpy(want).to(c.torch_dtype)
    assert torch.equal(out.cpu(), ref)


def test_decode_block_permutation_and_shared_prefix_bit_identical():
    cfg = dict(B=6, Hq=8, Hkv=2, D=128, BS=16, dtype="bf16", kv="same",
               ctx=("uniform", 40, 400), pool=("scale", 2.0), partition_tokens=0,
               shared_prefix=(3, 32), prefill=None)
    c = make_case(cfg, 7)
    kc, vc = product_cache(c)
    out, lse = run_decode(c, kc, vc, partition_tokens=64)
    perm = torch.from_numpy(np.random.default_rng(3).permutation(c.num_blocks)).cuda()
    k2, v2 = torch.empty_like(kc), torch.empty_like(vc)
    k2[perm], v2[perm] = kc, vc
    t2 = perm.cpu().numpy()[c.block_tables].astype(np.int32)
    out2, lse2 = run_decode(c, k2, v2, partition_tokens=64, block_tables=t2)
    assert torch.equal(out, out2) and torch.equal(lse, lse2)
    # private copies of the shared prefix blocks
    used = set(c.block_tables.ravel().tolist())
    free = [i for i in range(c.num_blocks) if i not in used]
    t3 = c.block_tables.copy()
    k3, v3 = kc.clone(), vc.clone()
    for b in (1, 2):
        for i in range(2):
            nid = free.pop()
            k3[nid], v3[nid] = kc[t3[b, i]], vc[t3[b, i]]
            t3[b, i] = nid
    out3, lse3 = run_decode(c, k3, v3, partition_tokens=64, block_tables=t3)
    check_device_ok()
    assert torch.equal(out, out3) and torch.equal(lse, lse3)


def test_decode_flags_bad_block_id_and_seq_len():
    c = make_case("tiny", 8)
    kc, vc = product_cache(c)
    bt = c.block_tables.copy()
    bt[1, 0] = c.num_blocks + 5
    run_decode(c, kc, vc, block_tables=bt)
    assert P.pkv_get_device_error() & 0x1
    sl = c.seq_lens.copy()
    sl[2] = c.max_seq_len + 40
    run_decode(c, kc, vc, seq_lens=sl)
    assert P.pkv_get_device_error() & 0x4


def test_decode_rejects_missing_workspace():
    c = make_case("tiny", 0)
    kc, vc = product_cache(c)
    q = dev(c.q)
    with pytest.raises(P.PkvError) as ei:
        P.paged_attn_decode(torch.empty_like(q), q, kc, vc, dev(c.block_tables),
                            dev(c.seq_lens), float(c.scale), c.max_seq_len, partition_tokens=16,
                            workspace=torch.empty(16, dtype=torch.uint8, device="cuda"))
    assert ei.value.status == 3


# ---- full-size workloads, sampled outputs ----------------------------------------

def test_decode_workspace_counters_reset_themselves():
    """Many calls on one zero-filled workspace, with sequences split into many
    partitions: every call merges the same way (the counters come back to
    zero each time) and no device error is raised."""
    c = make_case("tiny", 8, kv="fp8", ctx=("fixed", [700, 33, 520, 1]), pool=("blocks", 128))
    kc, vc = product_cache(c)
    ks, vs = scales(c)
    q = dev(c.q)
    bt, sl = dev(c.block_tables), dev(c.seq_lens)
    ws = torch.zeros(P.paged_attn_decode_workspace_size(c.B, c.Hq, c.Hkv, c.D, c.max_seq_len, 32),
                     dtype=torch.uint8, device="cuda")
    outs = []
    for _ in range(6):
        out = torch.empty_like(q)
        P.paged_attn_decode(out, q, kc, vc, bt, sl, float(c.scale), c.max_seq_len, ks, vs,
                            partition_tokens=32, workspace=ws)
        outs.append(out)
    torch.cuda.synchronize()
    check_device_ok()
    assert all(torch.equal(outs[0], o) for o in outs[1:])
    assert int(ws[:c.B * c.Hkv * 8].view(torch.int64).abs().sum()) == 0
    ko, vo = oracle_cache(c)
    want, _ = oracle_decode(c, ko, vo)
    assert_close(outs[-1], want, tol(c), "after repeated calls")


def test_decode_reports_counters_left_nonzero():
    c = make_case("tiny", 9, ctx=("fixed", [700, 33, 520, 1]), pool=("blocks", 128))
    kc, vc = product_cache(c)
    q = dev(c.q)
    ws = torch.zeros(P.paged_attn_decode_workspace_size(c.B, c.Hq, c.Hkv, c.D, c.max_seq_len, 32),
                     dtype=torch.uint8, device="cuda")
    # a (sequence, KV head) counter a failed call could have left: the
    # counters open the workspace
    ws[0:8].view(torch.int64)[0] = 1000
    out = torch.empty_like(q)
    P.paged_attn_decode(out, q, kc, vc, dev(c.block_tables), dev(c.seq_lens), float(c.scale),
                        c.max_seq_len, partition_tokens=32, workspace=ws)
    assert P.pkv_get_device_error() & 0x40


@pytest.mark.parametrize("name,sel", [("qwen2.5-7b", [0, 5, 17, 31]),
                                      ("llama3-8b-fp8", [0, 9, 64, 127]),
                                      ("long-ctx", [0, 3])])
def test_decode_full_size_sampled(name, sel):
    c = make_case(name, 0, device="cuda")
    # the launch configuration the bench times (automatic partitions unless
    # the workload fixes them)
    _decode_vs_oracle(c, sel=sel)


# ---- prefill -------------------------------------------------------------------

def _prefill_case(seed, L, P_, dtype="f16", kv="same", Hq=4, Hkv=2, D=64):
    cfg = dict(B=2, Hq=Hq, Hkv=Hkv, D=D, BS=16, dtype=dtype, kv=kv, ctx=("fixed", [20, 33]),
               pool=("scale", 2.0), partition_tokens=0, shared_prefix=None, prefill=(L, P_))
    return make_case(cfg, seed)


@pytest.mark.parametrize("L,P_,dtype,kv,Hq,Hkv,D", [
    (1, 40, "f16", "same", 4, 2, 64), (37, 0, "f16", "same", 4, 2, 64),
    (50, 29, "bf16", "same", 8, 2, 128), (23, 17, "bf16", "fp8", 8, 2, 128),
    (100, 300, "bf16", "same", 16, 8, 128), (65, 7, "f16", "fp8", 14, 2, 64),
    (129, 130, "bf16", "same", 7, 7, 128),
    (70, 45, "bf16", "same", 28, 4, 128),      # G = 7: 18 tokens, 126 of 128 rows per tile
    (40, 100, "f16", "same", 16, 1, 64)])      # G = 16: 8 tokens per tile
def test_prefill_vs_oracle(L, P_, dtype, kv, Hq, Hkv, D):
    c = _prefill_case(9, L, P_, dtype, kv, Hq, Hkv, D)
    kc, vc = product_cache(c)
    out, lse = run_prefill(c, kc, vc)
    check_device_ok()
    ko, vo = oracle_cache(c)
    pf = c.prefill
    want, wlse = O.prefill_chunk(pf.q, ko, vo, pf.block_tables, pf.seq_lens, pf.cu_q_lens,
                                 c.scale, c.k_scales, c.v_scales)
    assert_close(out, want, tol(c), "prefill out")
    assert_close(lse, wlse, LSE_TOL, "prefill lse")


@pytest.mark.parametrize("L,P_,dtype,Hq,Hkv,D,split,kv", [
    (640, 100, "f16", 16, 8, 64, False, "same"),    # 80 query tiles: one CTA each
    (300, 500, "bf16", 16, 8, 128, True, "same"),   # 40 query tiles: a cluster of two each
    (200, 0, "bf16", 8, 8, 128, True, "same"),      # odd key-tile counts per row
    (640, 100, "bf16", 16, 8, 128, False, "fp8"),   # E4M3 tiles converted on chip
    (300, 500, "f16", 16, 8, 64, True, "fp8"),
])
def test_prefill_one_cta_and_cluster_key_split(L, P_, dtype, Hq, Hkv, D, split, kv):
    # the tensor-core prefill splits each query tile's keys over a cluster of
    # two CTAs when the tiles alone would fill at most half of the SMs
    sms = torch.cuda.get_device_properties(0).multi_processor_count
    ctas = -(-L // (128 // (Hq // Hkv))) * Hkv
    assert (2 * ctas <= sms) == split, "case does not take the intended path"
    c = _prefill_case(12, L, P_, dtype, kv, Hq, Hkv, D)
    kc, vc = product_cache(c)
    out, lse = run_prefill(c, kc, vc)
    check_device_ok()
    ko, vo = oracle_cache(c)
    pf = c.prefill
    want, wlse = O.prefill_chunk(pf.q, ko, vo, pf.block_tables, pf.seq_lens, pf.cu_q_lens,
                                 c.scale, c.k_scales, c.v_scales)
    assert_close(out, want, tol(c), "prefill out")
    assert_close(lse, wlse, LSE_TOL, "prefill lse")


@pytest.mark.parametrize("Hq,Hkv", [(8, 2), (28, 4)])
def test_prefill_several_sequences_in_one_call(Hq, Hkv):
    # three sequences with different chunk lengths and histories; a query
    # tile of one sequence spans the next sequence's rows of q (G = 4: 32
    # tokens a tile; G = 7: 18 tokens, 126 of 128 rows), which its output
    # must leave alone
    c = _prefill_case(10, 10, 10, "bf16", "same", Hq, Hkv, 128)
    kc, vc = product_cache(c)
    ko, vo = oracle_cache(c)
    # reuse the two decode sequences as extra prefill sequences: their chunk
    # is their last few tokens
    tables = np.zeros((3, max(c.block_tables.shape[1], c.prefill.block_tables.shape[1])), np.int32)
    tables[:2, :c.block_tables.shape[1]] = c.block_tables
    tables[2, :c.prefill.block_tables.shape[1]] = c.prefill.block_tables[0]
    seq_lens = np.array([c.seq_lens[0], c.seq_lens[1], c.prefill.seq_lens[0]], np.int32)
    Ls = [5, 33, 10]
    cu = np.array([0, 5, 38, 48], np.int32)
    g = torch.Generator().manual_seed(4)
    q = torch.randn((48, c.Hq, c.D), generator=g).to(torch.bfloat16)
    out = torch.empty_like(q).cuda()
    P.paged_attn_prefill_chunk(out, dev(q), kc, vc, dev(tables), dev(seq_lens), dev(cu),
                               float(c.scale), max(Ls))
    check_device_ok()
    want, _ = O.prefill_chunk(q, ko, vo, tables, seq_lens, cu, c.scale)
    assert_close(out, want, 1e-2, "multi-seq prefill")


@pytest.mark.parametrize("kv", ["same", "fp8"])
def test_prefill_flags_bad_block_id(kv):
    # an id past the pool is flagged and read as block 0: the call completes
    c = _prefill_case(13, 100, 60, "bf16", kv, 8, 2, 128)
    kc, vc = product_cache(c)
    pf = c.prefill
    bt = pf.block_tables.copy()
    bt[0, 3] = c.num_blocks
    q = dev(pf.q)
    out = torch.zeros_like(q)
    ks, vs = scales(c)
    P.paged_attn_prefill_chunk(out, q, kc, vc, dev(bt), dev(pf.seq_lens), dev(pf.cu_q_lens),
                               float(c.scale), pf.L, ks, vs)
    torch.cuda.synchronize()
    assert P.pkv_get_device_error() & 0x1


def test_prefill_flags_chunk_longer_than_context():
    c = _prefill_case(11, 8, 4)
    kc, vc = product_cache(c)
    pf = c.prefill
    q = dev(pf.q)
    out = torch.zeros_like(q)
    P.paged_attn_prefill_chunk(out, q, kc, vc, dev(pf.block_tables), dev(np.array([5], np.int32)),
                               dev(pf.cu_q_lens), float(c.scale), pf.L)
    assert P.pkv_get_device_error() & 0x10


def test_prefill_flags_chunk_outside_q_rows():
    # the second sequence's chunk claims rows 5 .. 44 of a 30-row q and out:
    # flagged and skipped, nothing read or written past the rows; the first
    # sequence's chunk (rows 0 .. 4) is computed as usual
    c = _prefill_case(13, 40, 30, "bf16", "same", 8, 2, 128)
    kc, vc = product_cache(c)
    ko, vo = oracle_cache(c)
    width = max(c.block_tables.shape[1], c.prefill.block_tables.shape[1])
    tables = np.zeros((2, width), np.int32)
    tables[0, :c.block_tables.shape[1]] = c.block_tables[0]
    tables[1, :c.prefill.block_tables.shape[1]] = c.prefill.block_tables[0]
    seq_lens = np.array([c.seq_lens[0], c.prefill.seq_lens[0]], np.int32)
    assert seq_lens[1] >= 40                              # the chunk fits its context
    cu = np.array([0, 5, 45], np.int32)
    g = torch.Generator().manual_seed(5)
    q = torch.randn((30, c.Hq, c.D), generator=g).to(torch.bfloat16)
    out = torch.zeros_like(q).cuda()
    P.paged_attn_prefill_chunk(out, dev(q), kc, vc, dev(tables), dev(seq_lens), dev(cu),
                               float(c.scale), 40)
    assert P.pkv_get_device_error() & 0x10
    want, _ = O.prefill_chunk(q[:5], ko, vo, tables[:1], seq_lens[:1], cu[:2], c.scale)
    assert_close(out[:5], want, 1e-2, "the chunk inside q's rows")
    assert not out[5:].any(), "rows of the flagged chunk were written"


# ---- the mixed continuous-batching step ----------------------------------------------

def test_mixed_step_vs_oracle():
    from paged_kv_decode_11_gb300.step import MixedStep
    c = make_case("mixed", 0, device="cuda")
    kc, vc = product_cache(c, write_new=False)
    step = MixedStep.from_case(c, kc, vc)
    step.run()
    torch.cuda.synchronize()
    check_device_ok()
    sel = [0, 7, 15, 16, 40, 63]                       # 0..15 share the prefix
    ko, vo = oracle_cache(c)
    want, wlse = oracle_decode(c, ko, vo, sel=sel)
    assert_close(step.out[torch.as_tensor(sel)], want, tol(c), "mixed decode")
    pf = c.prefill
    pw, _ = O.prefill_chunk(pf.q.cpu(), ko, vo, pf.block_tables, pf.seq_lens, pf.cu_q_lens,
                            c.scale)
    assert_close(step.prefill_out, pw, tol(c), "mixed prefill")
    # the step wrote the same cache bytes as the oracle
    assert torch.equal(kc.cpu().view(torch.uint8), ko.view(torch.uint8))


# ---- failure path of the bounded waits ---------------------------------------------------

@pytest.mark.parametrize("polls", [1, 64, 4096])
def test_bounded_wait_gives_up_reports_timeout_and_leaves_the_context_usable(polls):
    P.pkv_get_device_error()                           # start clear
    P.pkv_selftest_bounded_wait(polls)
    assert P.pkv_get_device_error() == 0x8             # PKV_DEVERR_TIMEOUT, nothing else
    # the next real call runs normally on the same context
    c = make_case("tiny", 0)
    kc, vc = product_cache(c)
    out, lse = run_decode(c, kc, vc)
    check_device_ok()
    ko, vo = oracle_cache(c)
    want, _ = oracle_decode(c, ko, vo)
    assert_close(out, want, tol(c), "decode after a timed-out wait")
