"""Host-side arithmetic of bench.py that its JSON lines rest on, checked
against closed forms (no GPU)."""
import sys

import pytest

from workloads import make_case


def test_prefill_flops_closed_form():
    import bench
    c = make_case("mixed", 0, device="cpu")
    L, P = c.prefill.L, c.prefill.P
    keys = L * P + L * (L + 1) // 2            # row i sees P + i + 1 keys
    assert bench.prefill_flops(c) == 4.0 * c.Hq * c.D * keys
    assert bench.prefill_flops(c) == 7_367_294_976.0   # the mixed chunk: 7.37 GFLOP


def test_step_kv_bytes_counts_every_context_token_once():
    import bench
    for name in ("tiny", "qwen2.5-7b", "llama3-8b-fp8"):
        c = make_case(name, 0, device="cpu")
        metric, logical = bench.step_kv_bytes(c)
        want = int(c.seq_lens.sum()) * c.Hkv * c.D * 2 * c.kv_elem_bytes
        assert metric == logical == want


def test_mixed_step_counts_shared_prefix_blocks_once():
    import bench
    c = make_case("mixed", 0, device="cpu")
    metric, logical = bench.step_kv_bytes(c)
    assert logical == int(c.seq_lens.sum()) * c.Hkv * c.D * 2 * c.kv_elem_bytes
    # 15 of the 16 prefix sharers reuse the first one's 1024 cached tokens
    assert logical - metric == 15 * 1024 * c.Hkv * c.D * 2 * c.kv_elem_bytes


def test_prefill_only_flag_parses(monkeypatch):
    import bench
    monkeypatch.setattr(sys, "argv", ["bench.py", "--config", "mixed", "--prefill-only"])
    args = bench.parse_args()
    assert args.prefill_only and args.config == "mixed"


def test_cpu_baseline_leg_runs_the_oracle_on_a_bounded_sample():
    import bench
    c = make_case("tiny", 0, device="cpu")
    r = bench.cpu_baseline(c, 1.0, 0, 2)
    assert r["kind"] == "oracle" and r["unit"] == "GB/s" and r["value"] > 0
    assert r["cores"] == 2
    assert "units of the same workload" in r["sample"]
