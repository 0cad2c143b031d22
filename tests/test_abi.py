"""The C-ABI library builds, loads and exports every symbol include/pkv.h
declares; argument checks that need no GPU return their status codes. No
compute call is made here (no GPU needed)."""
import ctypes
import os
import re

import pytest

import paged_kv_decode_11_gb300 as P
from paged_kv_decode_11_gb300 import _binding, build

ROOT = os.path.dirname(os.path.dirname(os.path.abspath(__file__)))
HEADER = os.path.join(ROOT, "include", "pkv.h")

OK, INVALID, UNSUPPORTED, WORKSPACE = 0, 1, 2, 3
F16, BF16, FP8 = 0, 1, 2
FAKE = 0x10000          # never dereferenced: every call below fails its checks first


@pytest.fixture(scope="module")
def lib():
    build.build()
    return P.load()


def header_functions():
    txt = open(HEADER).read()
    txt = re.sub(r"/\*.*?\*/", "", txt, flags=re.S)
    return sorted(set(re.findall(r"\b([a-z_][a-z0-9_]*)\s*\(", txt)) -
                  {"if", "sizeof", "defined"})


def test_header_declares_the_abi():
    assert header_functions() == sorted(_binding.EXPORTS)


def header_param_counts():
    """Number of parameters of every function the header declares."""
    txt = re.sub(r"/\*.*?\*/", "", open(HEADER).read(), flags=re.S)
    counts = {}
    for m in re.finditer(r"\b([a-z_][a-z0-9_]*)\s*\(([^;{]*?)\)\s*;", txt):
        params = m.group(2).strip()
        counts[m.group(1)] = 0 if params in ("", "void") else params.count(",") + 1
    return counts


def test_binding_signatures_match_the_header(lib):
    counts = header_param_counts()
    for name in _binding.EXPORTS:
        fn = getattr(lib, name)
        assert fn.argtypes is not None, name
        assert len(fn.argtypes) == counts[name], (name, len(fn.argtypes), counts[name])


def test_library_exports_every_declared_symbol(lib):
    for name in header_functions():
        assert hasattr(lib, name), name


def test_library_exports_nothing_else():
    out = os.popen(f"nm -D --defined-only {_binding.LIB_PATH}").read()
    syms = {l.split()[-1] for l in out.splitlines() if " T " in l}
    assert syms == set(header_functions())


def test_status_strings(lib):
    for s in range(6):
        assert P.pkv_status_string(s) == _binding.STATUS[s]
    assert P.pkv_status_string(99) == "unknown status"


def _decode(lib, **kw):
    a = dict(out=FAKE, q=FAKE, q_dtype=BF16, k=FAKE, v=FAKE, kv_dtype=BF16, bt=FAKE, sl=FAKE,
             B=4, Hq=8, Hkv=2, D=128, BS=16, maxb=8, nb=64, msl=128, scale=0.1, ks=None,
             vs=None, part=0, lse=None, ws=None, wsb=0, stream=None)
    a.update(kw)
    return lib.paged_attn_decode(a["out"], a["q"], a["q_dtype"], a["k"], a["v"], a["kv_dtype"],
                                 a["bt"], a["sl"], a["B"], a["Hq"], a["Hkv"], a["D"], a["BS"],
                                 a["maxb"], a["nb"], a["msl"], a["scale"], a["ks"], a["vs"],
                                 a["part"], a["lse"], a["ws"], a["wsb"], a["stream"])


@pytest.mark.parametrize("kw,want", [
    (dict(D=96), UNSUPPORTED), (dict(D=512), UNSUPPORTED), (dict(D=256, Hq=32, Hkv=2), UNSUPPORTED),
    (dict(BS=3), UNSUPPORTED), (dict(BS=48), UNSUPPORTED), (dict(D=256, B=0, out=None), OK),
    (dict(D=256, BS=8), UNSUPPORTED),
    (dict(BS=1, B=0, out=None), OK), (dict(BS=8, B=0, out=None), OK),
    (dict(BS=1, part=4096), UNSUPPORTED), (dict(BS=16, part=4096, B=0, out=None), OK),
    (dict(BS=128), UNSUPPORTED), (dict(BS=32, B=0, out=None), OK),
    (dict(BS=64, B=0, out=None), OK), (dict(Hq=34, Hkv=2), UNSUPPORTED),
    (dict(Hq=9, Hkv=2), INVALID), (dict(q_dtype=FP8, kv_dtype=FP8), UNSUPPORTED),
    (dict(q_dtype=F16, kv_dtype=BF16), UNSUPPORTED), (dict(part=24), INVALID),
    (dict(part=8192 + 16), INVALID), (dict(out=None), INVALID), (dict(bt=None), INVALID),
    (dict(kv_dtype=FP8), INVALID), (dict(q=FAKE + 8), INVALID), (dict(B=-1), INVALID),
    (dict(nb=0), INVALID), (dict(B=0, out=None), OK), (dict(B=70000), UNSUPPORTED),
])
def test_decode_argument_checks(lib, kw, want):
    assert _decode(lib, **kw) == want


def test_decode_workspace_check(lib):
    # the workspace (work counters + partials) is always required, 256-aligned
    assert _decode(lib, part=64, msl=128, ws=None) == WORKSPACE
    need = P.paged_attn_decode_workspace_size(4, 8, 2, 128, 128, 64)
    assert _decode(lib, part=64, msl=128, ws=FAKE, wsb=need - 1) == WORKSPACE
    assert _decode(lib, part=64, msl=128, ws=FAKE + 16, wsb=need) == WORKSPACE


def test_workspace_size_formula(lib):
    # [done counters: B*Hkv words | partition outputs: B*Hq*parts rows of D
    # fp32 | partition log2-sum-exps: B*Hq*parts fp32], each region
    # 256-aligned, parts = ceil(max_seq_len / partition)
    def a256(x):
        return (x + 255) // 256 * 256

    def want(B, Hq, Hkv, D, parts):
        rows = B * Hq * parts
        return a256(B * Hkv * 8) + a256(rows * D * 4) + a256(rows * 4)
    assert P.paged_attn_decode_workspace_size(128, 32, 8, 128, 8192, 1024) == \
        want(128, 32, 8, 128, 8)
    assert P.paged_attn_decode_workspace_size(4, 8, 2, 64, 100, 256) == want(4, 8, 2, 64, 1)
    assert P.paged_attn_decode_workspace_size(4, 8, 2, 64, 100, 24) == 0      # invalid


def _prefill(lib, **kw):
    a = dict(out=FAKE, q=FAKE, q_dtype=BF16, k=FAKE, v=FAKE, kv_dtype=BF16, bt=FAKE, sl=FAKE,
             cu=FAKE, n=1, T=10, maxq=10, Hq=8, Hkv=2, D=128, BS=16, maxb=8, nb=64, scale=0.1,
             ks=None, vs=None, lse=None, stream=None)
    a.update(kw)
    return lib.paged_attn_prefill_chunk(a["out"], a["q"], a["q_dtype"], a["k"], a["v"],
                                        a["kv_dtype"], a["bt"], a["sl"], a["cu"], a["n"], a["T"],
                                        a["maxq"], a["Hq"], a["Hkv"], a["D"], a["BS"], a["maxb"],
                                        a["nb"], a["scale"], a["ks"], a["vs"], a["lse"],
                                        a["stream"])


@pytest.mark.parametrize("kw,want", [
    (dict(D=320), UNSUPPORTED), (dict(cu=None), INVALID), (dict(kv_dtype=FP8), INVALID),
    (dict(BS=1), UNSUPPORTED), (dict(T=0, out=None), OK), (dict(Hq=7, Hkv=2), INVALID),
])
def test_prefill_argument_checks(lib, kw, want):
    assert _prefill(lib, **kw) == want


def _cache(lib, **kw):
    a = dict(k=FAKE, v=FAKE, src=BF16, kc=FAKE, vc=FAKE, kv=FP8, slots=FAKE, T=4, Hkv=2, D=128,
             BS=16, nb=8, ks=FAKE, vs=FAKE, stream=None)
    a.update(kw)
    return lib.reshape_and_cache(a["k"], a["v"], a["src"], a["kc"], a["vc"], a["kv"], a["slots"],
                                 a["T"], a["Hkv"], a["D"], a["BS"], a["nb"], a["ks"], a["vs"],
                                 a["stream"])


@pytest.mark.parametrize("kw,want", [
    (dict(ks=None), INVALID), (dict(src=FP8), UNSUPPORTED), (dict(D=80), UNSUPPORTED),
    (dict(slots=None), INVALID), (dict(T=0, k=None), OK), (dict(kc=FAKE + 4), INVALID),
    (dict(src=F16, kv=BF16), UNSUPPORTED),
])
def test_cache_write_argument_checks(lib, kw, want):
    assert _cache(lib, **kw) == want


def _rope(lib, **kw):
    a = dict(q=FAKE, k=FAKE, v=FAKE, src=BF16, kc=FAKE, vc=FAKE, kv=FP8, slots=FAKE, pos=FAKE,
             cs=FAKE, maxpos=4096, rot=128, neox=1, T=4, Hq=8, Hkv=2, D=128, BS=16, nb=8,
             ks=FAKE, vs=FAKE, stream=None)
    a.update(kw)
    return lib.rope_reshape_and_cache(a["q"], a["k"], a["v"], a["src"], a["kc"], a["vc"], a["kv"],
                                      a["slots"], a["pos"], a["cs"], a["maxpos"], a["rot"],
                                      a["neox"], a["T"], a["Hq"], a["Hkv"], a["D"], a["BS"],
                                      a["nb"], a["ks"], a["vs"], a["stream"])


@pytest.mark.parametrize("kw,want", [
    (dict(rot=0), INVALID), (dict(rot=24), INVALID), (dict(rot=144), INVALID),
    (dict(D=64, rot=128), INVALID), (dict(maxpos=0), INVALID), (dict(pos=None), INVALID),
    (dict(cs=None), INVALID), (dict(cs=FAKE + 8), INVALID), (dict(q=None), INVALID),
    (dict(ks=None), INVALID), (dict(src=FP8), UNSUPPORTED), (dict(BS=24), UNSUPPORTED),
    (dict(T=0, q=None, k=None), OK), (dict(Hq=0), INVALID),
])
def test_rope_cache_argument_checks(lib, kw, want):
    assert _rope(lib, **kw) == want


@pytest.mark.parametrize("polls", [0, (1 << 20) + 1])
def test_selftest_wait_argument_check(lib, polls):
    assert lib.pkv_selftest_bounded_wait(polls, None) == INVALID
