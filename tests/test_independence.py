"""The oracle and the CUDA path share no code, and nothing on the product path
reaches the oracle (the checks read source text only)."""
import glob
import os
import re

ROOT = os.path.dirname(os.path.dirname(os.path.abspath(__file__)))


def _read(path):
    with open(path, encoding="utf-8") as f:
        return f.read()


def test_oracle_does_not_import_the_cuda_path():
    for p in glob.glob(os.path.join(ROOT, "oracle", "*")):
        if p.endswith((".py", ".c", ".h")):
            t = _read(p)
            assert "paged_kv_decode_11_gb300" not in t, p
            assert "csrc" not in t and "pkv.h" not in t, p


def test_product_path_does_not_reach_the_oracle():
    pkg = os.path.join(ROOT, "paged_kv_decode_11_gb300")
    for p in glob.glob(os.path.join(pkg, "**", "*"), recursive=True):
        if p.endswith((".py", ".cu", ".cuh", ".h")):
            t = _read(p)
            assert "import oracle" not in t and "from oracle" not in t, p
            assert "pkvo_" not in t and "liboracle" not in t, p


def test_generator_holds_no_method_arithmetic():
    gen = _read(os.path.join(ROOT, "workloads", "gen.py"))
    for word in ("softmax", "exp(", "log(", "encode", "einsum", "matmul"):
        assert word not in gen, word


def test_bench_uses_oracle_only_in_baseline_legs():
    t = _read(os.path.join(ROOT, "bench.py"))
    # every oracle import sits inside a CPU-baseline / reference function
    for m in re.finditer(r"from oracle import oracle", t):
        head = t[:m.start()]
        fn = re.findall(r"\ndef (\w+)\(", head)[-1]
        assert fn in {"oracle_setup", "oracle_units", "cpu_baseline", "run_reference"}, fn
