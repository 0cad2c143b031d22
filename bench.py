#!/usr/bin/env python
"""Benchmark of one attention-layer pass of a continuous-batching decode step
over a paged KV cache: reshape_and_cache of the step's new tokens, then decode
attention (split-KV partitions + log-sum-exp merge), on synthetic inputs.

Metric: KV-read GB/s = algorithmic K+V bytes of the step (every context token
of every sequence, per KV head, K and V) / device time of the step; also
reported as seqs/s per layer and as a fraction of the HBM roofline.

  python bench.py [--gpus N] [--steps K] [--warmup W] [--config NAME]
  python bench.py --impl reference ...    # the fp64 CPU oracle, bounded sample

Prints one JSON line (rank 0). Under torchrun each rank runs its own replica
(weak scaling: one independent batch per GPU, no collective on the data path);
the timed region is bracketed by a barrier and device syncs and the slowest
rank's time is reported.
"""
from __future__ import annotations

import argparse
import hashlib
import json
import os
import statistics
import subprocess
import sys
import tempfile
import time

ROOT = os.path.dirname(os.path.abspath(__file__))
sys.path.insert(0, ROOT)

import numpy as np  # noqa: E402
import torch  # noqa: E402

from workloads import BENCH_CONFIG, CONFIGS, empty_cache, make_case  # noqa: E402

NOMINAL_HBM_GBS = 8000.0
FALLBACK_HBM_GBS = 6800.0
FALLBACK_BF16_TFLOPS = 1900.0
L2_FLUSH_BYTES = 256 << 20
CLOCK_QUERY = ("index,clocks.sm,clocks.max.sm,power.draw,clocks_event_reasons.active,"
               "clocks_event_reasons.hw_slowdown,clocks_event_reasons.hw_thermal_slowdown,"
               "clocks_event_reasons.sw_thermal_slowdown,clocks_event_reasons.sw_power_cap")
REASON_NAMES = ["hw_slowdown", "hw_thermal_slowdown", "sw_thermal_slowdown", "sw_power_cap"]


def parse_args():
    ap = argparse.ArgumentParser()
    ap.add_argument("--gpus", type=int, default=1)
    ap.add_argument("--steps", type=int, default=2000)
    ap.add_argument("--warmup", type=int, default=20)
    ap.add_argument("--impl", choices=["ours", "reference"], default="ours")
    ap.add_argument("--config", default=BENCH_CONFIG, choices=sorted(CONFIGS))
    ap.add_argument("--seed", type=int, default=0)
    ap.add_argument("--batch", type=int, default=0,
                    help="override the workload's batch size (profiling on a smaller case)")
    ap.add_argument("--no-e2e", action="store_true")
    ap.add_argument("--no-graph", action="store_true",
                    help="skip the CUDA-graph replay timing of the same step")
    ap.add_argument("--no-cpu-baseline", action="store_true")
    ap.add_argument("--cpu-seconds", type=float, default=10.0,
                    help="CPU work budget of the oracle baseline sample")
    ap.add_argument("--cpu-threads", type=int, default=0,
                    help="host threads for the oracle legs (0: all cores)")
    ap.add_argument("--record-traffic", metavar="NCU_CSV", default=None,
                    help="store the DRAM bytes of the last decode launch in this ncu --csv "
                         "capture (dram__bytes_read.sum, dram__bytes_write.sum) as the "
                         "workload's traffic, keyed by the current decode source hash")
    ap.add_argument("--capture-command", default="",
                    help="with --record-traffic: the command the capture ran, kept with it")
    ap.add_argument("--prefill-only", action="store_true",
                    help="time the workload's prefill chunk alone (paged_attn_prefill_chunk); "
                         "prints a TFLOP/s line instead of the step line")
    return ap.parse_args()


# ---- distributed plumbing ---------------------------------------------------------

def dist_setup():
    world = int(os.environ.get("WORLD_SIZE", "1"))
    rank = int(os.environ.get("RANK", "0"))
    local = int(os.environ.get("LOCAL_RANK", "0"))
    if world > 1:
        import torch.distributed as dist
        backend = "nccl" if torch.cuda.is_available() else "gloo"
        if backend == "nccl":
            torch.cuda.set_device(local)
        dist.init_process_group(backend=backend)
    return rank, world, local


def barrier(world):
    if world > 1:
        import torch.distributed as dist
        dist.barrier()


def allreduce(x: float, op: str, world: int) -> float:
    if world == 1:
        return x
    import torch.distributed as dist
    dev = "cuda" if torch.cuda.is_available() else "cpu"
    t = torch.tensor([x], dtype=torch.float64, device=dev)
    dist.all_reduce(t, op=dist.ReduceOp.MAX if op == "max" else dist.ReduceOp.SUM)
    return float(t.item())


# ---- clocks -----------------------------------------------------------------------

class ClockSampler:
    """nvidia-smi clock / throttle-reason samples of this GPU while running."""

    def __init__(self, device_index: int):
        self.proc = None
        self.path = None
        sel = None
        try:
            uuid = str(torch.cuda.get_device_properties(device_index).uuid)
            sel = uuid if uuid.startswith("GPU-") else "GPU-" + uuid
        except Exception:
            vis = os.environ.get("CUDA_VISIBLE_DEVICES")
            sel = vis.split(",")[device_index] if vis else str(device_index)
        self.sel = sel

    def start(self):
        fd, self.path = tempfile.mkstemp(suffix=".csv")
        os.close(fd)
        try:
            self.proc = subprocess.Popen(
                ["nvidia-smi", f"--query-gpu=timestamp,{CLOCK_QUERY}", "--format=csv,noheader,nounits",
                 "-lms", "100", "-i", self.sel], stdout=open(self.path, "w"),
                stderr=subprocess.DEVNULL)
        except Exception:
            self.proc = None
        time.sleep(0.3)

    def stop(self):
        if self.proc is not None:
            time.sleep(0.25)
            self.proc.terminate()
            try:
                self.proc.wait(timeout=5)
            except Exception:
                self.proc.kill()
        rows = []
        if self.path and os.path.exists(self.path):
            with open(self.path) as f:
                for line in f:
                    parts = [x.strip() for x in line.split(",")]
                    if len(parts) >= 10:
                        rows.append(parts)
            os.unlink(self.path)
        return rows

    @staticmethod
    def summarise(rows, t0_wall, t1_wall):
        if not rows:
            return {"sm_mhz": None, "sm_max_mhz": None, "reasons": [], "samples": 0}
        sm, smax, reasons, n = [], None, set(), 0
        for r in rows:
            try:
                sm.append(float(r[2]))
                smax = float(r[3])
            except ValueError:
                continue
            n += 1
            for name, val in zip(REASON_NAMES, r[6:10]):
                if val.strip().lower() == "active":
                    reasons.add(name)
        # samples under load: clocks above the idle floor
        load = [x for x in sm if smax and x > 0.5 * smax] or sm
        return {"sm_mhz": statistics.median(load) if load else None, "sm_max_mhz": smax,
                "reasons": sorted(reasons), "samples": n}


# ---- profile-derived traffic ----------------------------------------------------

# The device code the decode kernels are built from and their partition
# planner: a traffic figure ncu took stays valid while none of these changes.
DECODE_SOURCES = ("common.cuh", "decode.cu", "decode_frags.cuh", "decode_full_first.cu",
                  "decode_kernel.cuh", "decode_wide.cu", "launch.h", "plan.h", "ptx.cuh")
TRAFFIC_FILE = os.path.join(ROOT, "profiles", "decode_traffic.json")


def source_hash() -> str:
    h = hashlib.sha256()
    csrc = os.path.join(ROOT, "paged_kv_decode_11_gb300", "csrc")
    for name in DECODE_SOURCES:
        with open(os.path.join(csrc, name), "rb") as f:
            h.update(name.encode())
            h.update(f.read())
    return h.hexdigest()[:16]


def profile_traffic(config: str):
    """DRAM bytes per decode call of this workload, as ncu measured them
    (profiles/decode_traffic.json, written by `bench.py --record-traffic`),
    if they were taken on the current decode sources; else None."""
    try:
        with open(TRAFFIC_FILE) as f:
            rec = json.load(f).get(config)
    except (OSError, ValueError):
        return None
    if not rec or rec.get("source_hash") != source_hash():
        return None
    return int(rec["dram_bytes_per_call"])


_BYTE_UNITS = {"byte": 1, "kbyte": 1e3, "mbyte": 1e6, "gbyte": 1e9, "tbyte": 1e12}


def record_traffic(args):
    """Reads an ncu --csv capture of this workload's bench run and stores the
    DRAM bytes (read + write) of its last decode launch in the traffic file."""
    import csv
    launches = {}
    with open(args.record_traffic, newline="") as f:
        rows = [r for r in csv.reader(f) if r]
    hdr_i = next(i for i, r in enumerate(rows) if "Metric Name" in r)
    hdr = rows[hdr_i]
    col = {name: hdr.index(name) for name in ("ID", "Kernel Name", "Metric Name", "Metric Unit",
                                              "Metric Value")}
    for r in rows[hdr_i + 1:]:
        if len(r) < len(hdr):
            continue
        name = r[col["Kernel Name"]]
        if "decode_kernel" not in name:
            continue
        metric = r[col["Metric Name"]]
        if metric not in ("dram__bytes_read.sum", "dram__bytes_write.sum"):
            continue
        unit = _BYTE_UNITS[r[col["Metric Unit"]].lower()]
        val = float(r[col["Metric Value"]].replace(",", "")) * unit
        launches.setdefault(int(r[col["ID"]]), {})[metric] = val
    last = max(i for i, m in launches.items() if len(m) == 2)
    m = launches[last]
    try:
        with open(TRAFFIC_FILE) as f:
            data = json.load(f)
    except (OSError, ValueError):
        data = {}
    data[args.config] = {
        "source_hash": source_hash(),
        "dram_bytes_per_call": int(round(m["dram__bytes_read.sum"] + m["dram__bytes_write.sum"])),
        "dram_bytes_read": int(round(m["dram__bytes_read.sum"])),
        "dram_bytes_write": int(round(m["dram__bytes_write.sum"])),
        "launch_id": last,
        "command": args.capture_command,
    }
    with open(TRAFFIC_FILE, "w") as f:
        json.dump(data, f, indent=1, sort_keys=True)
        f.write("\n")
    print(json.dumps({args.config: data[args.config]}))


class L2Flush:
    """Evicts everything from L2 between timed iterations (untimed): a write
    of a buffer twice the L2's size, then a read of a second one, so the
    write's dirty lines go back to HBM here and the L2 is left holding clean
    lines that the next iteration can drop for free."""

    def __init__(self):
        self.w = torch.empty(L2_FLUSH_BYTES, dtype=torch.uint8, device="cuda")
        self.r = torch.zeros(L2_FLUSH_BYTES // 4, dtype=torch.float32, device="cuda")
        self.acc = torch.zeros((), dtype=torch.float32, device="cuda")

    def __call__(self, i: int):
        self.w.fill_(i & 0xFF)
        self.acc.copy_(self.r.sum())

    @staticmethod
    def describe(what: str) -> str:
        return (f"flushed between timed {what}: a {L2_FLUSH_BYTES >> 20} MiB write, then a "
                f"{L2_FLUSH_BYTES >> 20} MiB read, so no dirty lines remain (untimed)")


def decode_kernel_name(case) -> str:
    """The kernel a decode call of this workload launches (decode.cu's routing)."""
    if case.BS < 16:
        return "decode_kernel, cp.async gather instantiation (one launch per decode call)"
    return "decode_kernel (one launch per decode call)"


def measured_hbm_peak():
    path = os.path.join(ROOT, "MEASURED_PEAKS.json")
    try:
        with open(path) as f:
            return float(json.load(f)["hbm_gbs"]), "measured"
    except Exception:
        return FALLBACK_HBM_GBS, "fallback"


# ---- workload helpers ---------------------------------------------------------------

def workload_desc(case) -> str:
    cfg = case.cfg
    ctx = cfg["ctx"]
    ctxs = (f"ctx U[{ctx[1]},{ctx[2]}]" if ctx[0] == "uniform" else
            "ctx {" + ",".join(str(x) for x in ctx[1]) + "}")
    kv = "E4M3 KV + per-head fp32 scales" if case.kv_fp8 else f"{case.dtype} KV"
    s = (f"{case.name} decode step: reshape_and_cache of {len(case.new_slots)} new tokens + "
         f"paged decode attention, B{case.B} Hq{case.Hq} Hkv{case.Hkv} D{case.D} block 16, "
         f"{ctxs}, {case.dtype} q, {kv}, pool {case.num_blocks} blocks")
    if case.prefill is not None:
        s += (f" + prefill chunk L{case.prefill.L} on P{case.prefill.P} (one paged_attn_varlen "
              f"call with the decode rows)")
    if cfg.get("shared_prefix"):
        s += f"; {cfg['shared_prefix'][0]} seqs share a {cfg['shared_prefix'][1]}-token prefix"
    return s


def step_kv_bytes(case):
    """(bytes counted for the metric, logical bytes) of one step."""
    if case.cfg.get("shared_prefix"):
        return case.kv_bytes_unique(), case.kv_bytes_logical()
    return case.kv_bytes_logical(), case.kv_bytes_logical()


def sample_units(case, n_units, rng):
    """n (sequence, KV head) units of the workload, drawn without replacement."""
    all_units = [(b, h) for b in range(case.B) for h in range(case.Hkv)]
    idx = rng.choice(len(all_units), size=min(n_units, len(all_units)), replace=False)
    return [all_units[i] for i in idx]


def oracle_setup(case, units):
    """The oracle's cache holding the rows the sampled sequences read."""
    from oracle import oracle as O
    seqs = sorted({b for b, _ in units})
    kc, vc = empty_cache(case, "cpu")
    slots_all = np.concatenate([case.fill_slots, case.new_slots])
    rows = np.unique(np.concatenate(
        [case.logical_rows(case.block_tables[b], int(case.seq_lens[b])) for b in seqs]))
    nf = len(case.fill_slots)
    rt = torch.as_tensor(rows)
    fr, nr = rt[rt < nf], rt[rt >= nf] - nf
    k = torch.cat([case.fill_k[fr.to(case.fill_k.device)].cpu(),
                   case.new_k[nr.to(case.new_k.device)].cpu()]).contiguous()
    v = torch.cat([case.fill_v[fr.to(case.fill_v.device)].cpu(),
                   case.new_v[nr.to(case.new_v.device)].cpu()]).contiguous()
    sl = np.concatenate([slots_all[fr.numpy()], slots_all[nf + nr.numpy()]])
    assert O.reshape_and_cache(k, v, kc, vc, sl, case.k_scales, case.v_scales) == 0
    return kc, vc


def oracle_seconds_per_unit(case, units, q_cpu, threads):
    """Calibration: one batch of as many units as the oracle has threads."""
    c = units[:max(1, min(len(units), threads))]
    kc, vc = oracle_setup(case, c)
    t = time.perf_counter()
    oracle_units(case, kc, vc, c, q_cpu)
    return max(time.perf_counter() - t, 1e-4) / len(c)


ORACLE_THREADS = 0          # host threads of the oracle legs (0: all cores)


def oracle_units(case, kc, vc, units, q_cpu):
    """Several (sequence, KV head) units in one oracle call per KV head, so the
    oracle's OpenMP loop over (sequence, query head) has work for every core."""
    from oracle import oracle as O
    # set before every call: torch's own OpenMP set-up can run in between and,
    # when both share one OpenMP runtime, reset the thread count
    O.set_threads(ORACLE_THREADS)
    G = case.G
    nbytes = 0
    for h in sorted({h for _, h in units}):
        seqs = [b for b, hh in units if hh == h]
        O.decode(q_cpu, kc, vc, case.block_tables, case.seq_lens, case.scale, case.k_scales,
                 case.v_scales, sel=seqs, heads=(h * G, (h + 1) * G))
        nbytes += sum(int(case.seq_lens[b]) for b in seqs) * case.D * 2 * case.kv_elem_bytes
    return nbytes


def cpu_baseline(case, seconds: float, seed: int, threads: int = 0):
    """The oracle as it stands, on a bounded sample of (sequence, KV head)
    units of this workload, on the host cores; KV-read GB/s."""
    from oracle import oracle as O
    global ORACLE_THREADS
    O.build()
    ORACLE_THREADS = threads
    O.set_threads(threads)
    rng = np.random.default_rng(seed + 99)
    units = sample_units(case, case.B * case.Hkv, rng)
    q_cpu = case.q.cpu().contiguous()
    # size the sample: time one batch, then take what fits the budget
    t1 = oracle_seconds_per_unit(case, units, q_cpu, O.threads())
    n = int(max(1, min(len(units), seconds / t1)))
    units = units[:n]
    kc, vc = oracle_setup(case, units)
    t = time.perf_counter()
    nbytes = oracle_units(case, kc, vc, units, q_cpu)
    dt = time.perf_counter() - t
    return {"value": nbytes / dt / 1e9, "unit": "GB/s", "cores": O.threads(), "kind": "oracle",
            "sample": f"{n} of {case.B * case.Hkv} (sequence, KV head) units of the same "
                      f"workload, all {case.G} query heads of each, fp64 oracle (one call per "
                      f"KV head over the sampled sequences, OpenMP over (sequence, query "
                      f"head)), {nbytes / 1e6:.1f} MB of KV in {dt:.2f} s"}


# ---- our arm -------------------------------------------------------------------------------

def run_ours(args):
    rank, world, local = dist_setup()
    torch.cuda.set_device(local)
    from paged_kv_decode_11_gb300 import build as pkv_build
    pkv_build.build()
    import paged_kv_decode_11_gb300 as P
    from paged_kv_decode_11_gb300.step import DecodeStep, MixedStep
    P.load()

    over = {"B": args.batch} if args.batch else {}
    case = make_case(args.config, args.seed + rank, device="cuda", **over)
    kc, vc = empty_cache(case, "cuda")
    ks = vs = None
    if case.kv_fp8:
        ks = torch.from_numpy(case.k_scales).cuda()
        vs = torch.from_numpy(case.v_scales).cuda()
    # the cache as the previous steps left it (every context token but the new ones)
    P.reshape_and_cache(case.fill_k, case.fill_v, kc, vc,
                        torch.from_numpy(case.fill_slots).cuda(), ks, vs)
    torch.cuda.synchronize()
    step = (MixedStep if case.prefill is not None else DecodeStep).from_case(case, kc, vc)
    dstep = step.decode if isinstance(step, MixedStep) else step
    # reshape_and_cache + one decode launch (+ one prefill launch)
    launches_per_step = 2 + (1 if case.prefill is not None else 0)
    kv_bytes, kv_logical = step_kv_bytes(case)
    flush = L2Flush()
    stream = torch.cuda.current_stream()

    def one_step():
        step.run(stream)

    for _ in range(args.warmup):
        one_step()
    torch.cuda.synchronize()
    assert P.pkv_get_device_error() == 0

    sampler = ClockSampler(local)
    if rank == 0:
        sampler.start()
    K = args.steps
    ev = [(torch.cuda.Event(enable_timing=True), torch.cuda.Event(enable_timing=True))
          for _ in range(K)]
    barrier(world)
    torch.cuda.synchronize()
    t0 = time.time()
    for i in range(K):
        flush(i)                                    # evict the previous step from L2
        ev[i][0].record(stream)
        one_step()                                  # the step's own call(s)
        ev[i][1].record(stream)
    torch.cuda.synchronize()
    barrier(world)
    t1 = time.time()
    # the decode kernel alone, for its roofline: the cache write, then an event,
    # then the attention call (which then cannot start before the write ends)
    attn_ms = None
    if not isinstance(step, MixedStep):
        ev2 = [(torch.cuda.Event(enable_timing=True), torch.cuda.Event(enable_timing=True))
               for _ in range(K)]
        for i in range(K):
            flush(i)
            step.write_cache(stream)
            ev2[i][0].record(stream)
            step.attend(stream)
            ev2[i][1].record(stream)
        torch.cuda.synchronize()
        attn_ms = [a.elapsed_time(b) for a, b in ev2]
    rows = sampler.stop() if rank == 0 else []
    step_ms = [a.elapsed_time(b) for a, b in ev]
    ms_local = float(np.mean(step_ms))
    ms = allreduce(ms_local, "max", world)
    total_bytes = allreduce(float(kv_bytes), "sum", world)
    value = total_bytes / (ms / 1e3) / 1e9
    total_seqs = allreduce(float(case.B), "sum", world)

    # dominant kernel: the decode attention call (split kernel + merge) on this stream
    peak, peak_kind = measured_hbm_peak()
    if attn_ms is not None:
        attn_mean = float(np.mean(attn_ms))
        achieved = kv_bytes / (attn_mean / 1e3) / 1e9
    else:
        attn_mean, achieved = None, None
    traffic = profile_traffic(args.config)

    graph = None
    if not args.no_graph:
        graph = measure_graph(step, stream, args, world, kv_bytes, flush, launches_per_step)

    e2e = None
    if not args.no_e2e:
        e2e = measure_e2e(step, stream, args, world, kv_bytes, flush)

    cpu = None
    if rank == 0 and world == 1 and not args.no_cpu_baseline:
        cpu = cpu_baseline(case, args.cpu_seconds, args.seed, args.cpu_threads)

    clocks = ClockSampler.summarise(rows, t0, t1)
    if rank == 0:
        line = {
            "metric": "paged-KV decode attn: KV-read GB/s (% of GB300 HBM peak); seqs/s per layer",
            "value": round(value, 2),
            "unit": "GB/s",
            "n_gpus": world,
            "steps": K,
            "warmup": args.warmup,
            "ms_per_step": round(ms, 5),
            "higher_is_better": True,
            "scaling": "weak",
            "vs_baseline": None,
            "dtype": (("e4m3 KV dequantised to f16 for m16n8k16 MMA, fp32 accumulate"
                       if case.kv_fp8 else f"{case.dtype} m16n8k16 MMA, fp32 accumulate")
                      + ("; prefill chunk on tcgen05 MMA (TMEM fp32 accumulators)"
                         if case.prefill is not None else "")),
            "data": "synthetic (seeded N(0,1) values, random block placement)",
            "config": {
                "workload": workload_desc(case),
                "global_batch": int(total_seqs),
                "kv_bytes_per_step": int(kv_bytes),
                "kv_bytes_logical_per_step": int(kv_logical),
                "l2": L2Flush.describe("steps") +
                      f"; the step reads {kv_bytes / 1e6:.0f} MB of KV",
                "parallelism": f"replicas x{world} (independent batch per GPU)",
            },
            "seqs_per_s_per_layer": round(total_seqs / (ms / 1e3), 1),
            "pct_of_nominal_hbm": round(100 * value / world / NOMINAL_HBM_GBS, 2),
            "roofline": {
                "kernel": decode_kernel_name(case),
                "bound": "hbm",
                "achieved": round(achieved, 2) if achieved else None,
                "peak": peak,
                "peak_kind": peak_kind,
                "unit": "GB/s",
                "frac": round(achieved / peak, 4) if achieved else None,
                "traffic": traffic,
                "algorithmic_bytes_per_launch": int(kv_bytes),
                "mean_call_us": round(attn_mean * 1e3, 2) if attn_mean else None,
            },
            "cpu_baseline": cpu,
            "e2e": e2e,
            "cuda_graph": graph,
            "clocks": clocks,
            "gpu_launches": launches_per_step * K,
        }
        print(json.dumps(line), flush=True)
    if world > 1:
        import torch.distributed as dist
        dist.destroy_process_group()


def measure_graph(step, stream, args, world, kv_bytes, flush, launches):
    """The same step captured once into a CUDA graph (cache write, counter
    reset, decode and, for the mixed step, the prefill on its second stream)
    and replayed; the L2 flush runs outside the graph, untimed."""
    side = torch.cuda.Stream()
    side.wait_stream(stream)
    with torch.cuda.stream(side):
        step.run()
    stream.wait_stream(side)
    torch.cuda.synchronize()
    g = torch.cuda.CUDAGraph()
    with torch.cuda.graph(g):
        step.run()
    torch.cuda.synchronize()
    for _ in range(args.warmup):
        g.replay()
    torch.cuda.synchronize()
    K = args.steps
    ev = [(torch.cuda.Event(enable_timing=True), torch.cuda.Event(enable_timing=True))
          for _ in range(K)]
    barrier(world)
    torch.cuda.synchronize()
    cur = torch.cuda.current_stream()
    for i in range(K):
        flush(i)
        ev[i][0].record(cur)
        g.replay()
        ev[i][1].record(cur)
    torch.cuda.synchronize()
    barrier(world)
    ms = allreduce(float(np.mean([a.elapsed_time(b) for a, b in ev])), "max", world)
    total = allreduce(float(kv_bytes), "sum", world)
    return {"value": round(total / (ms / 1e3) / 1e9, 2), "unit": "GB/s",
            "ms_per_step": round(ms, 5), "kernels_per_replay": launches}


def measure_e2e(step, stream, args, world, kv_bytes, flush):
    """The same step through the public API with inputs copied from pinned
    host memory and outputs read back, every step, inside the timed region."""
    dev_in = step.inputs()
    dev_out = step.outputs()
    host_in = [t.cpu().pin_memory() for t in dev_in]
    host_out = [torch.empty(t.shape, dtype=t.dtype).pin_memory() for t in dev_out]
    h2d = sum(t.numel() * t.element_size() for t in host_in)
    d2h = sum(t.numel() * t.element_size() for t in host_out)

    def e2e_step():
        for d, h in zip(dev_in, host_in):
            d.copy_(h, non_blocking=True)
        step.run(stream)
        for d, h in zip(dev_out, host_out):
            h.copy_(d, non_blocking=True)

    for _ in range(args.warmup):
        e2e_step()
    torch.cuda.synchronize()
    K = args.steps
    ev = [(torch.cuda.Event(enable_timing=True), torch.cuda.Event(enable_timing=True))
          for _ in range(K)]
    barrier(world)
    torch.cuda.synchronize()
    for i in range(K):
        flush(i)
        ev[i][0].record(stream)
        e2e_step()
        ev[i][1].record(stream)
    torch.cuda.synchronize()
    barrier(world)
    ms = allreduce(float(np.mean([a.elapsed_time(b) for a, b in ev])), "max", world)
    total = allreduce(float(kv_bytes), "sum", world)
    return {"value": round(total / (ms / 1e3) / 1e9, 2), "unit": "GB/s",
            "h2d_bytes_per_step": int(h2d), "d2h_bytes_per_step": int(d2h),
            "ms_per_step": round(ms, 5)}


# ---- reference arm: the fp64 oracle on the host cores ------------------------------------

def run_reference(args):
    rank = int(os.environ.get("RANK", "0"))
    if rank != 0:
        return
    from oracle import oracle as O
    global ORACLE_THREADS
    O.build()
    ORACLE_THREADS = args.cpu_threads
    O.set_threads(args.cpu_threads)
    dev = "cuda" if torch.cuda.is_available() else "cpu"
    case = make_case(args.config, args.seed, device=dev)
    rng = np.random.default_rng(args.seed + 7)
    units = sample_units(case, case.B * case.Hkv, rng)
    q_cpu = case.q.cpu().contiguous()
    # calibrate: units per step so the whole warmup + timed run stays within ~2 minutes
    t1 = oracle_seconds_per_unit(case, units, q_cpu, O.threads())
    budget = 120.0 / max(1, args.steps + args.warmup)
    per_step = int(max(1, min(len(units), budget / t1)))
    need = min(len(units), per_step * (args.steps + args.warmup))
    kc, vc = oracle_setup(case, units[:need])
    cursor = 0

    def ref_step():
        nonlocal cursor
        batch = [units[(cursor + i) % need] for i in range(per_step)]
        cursor += per_step
        return oracle_units(case, kc, vc, batch, q_cpu)

    for _ in range(args.warmup):
        ref_step()
    nbytes = 0
    t = time.perf_counter()
    for _ in range(args.steps):
        nbytes += ref_step()
    dt = time.perf_counter() - t
    value = nbytes / dt / 1e9
    kv_bytes, _ = step_kv_bytes(case)
    sample = (f"each step: {per_step} (sequence, KV head) unit(s) of the workload, all "
              f"{case.G} query heads each, fp64 oracle ({nbytes / max(1, args.steps) / 1e6:.2f} MB "
              f"of KV per step vs {kv_bytes / 1e6:.0f} MB for the whole step)")
    line = {
        "impl": "reference",
        "metric": "paged-KV decode attn: KV-read GB/s (% of GB300 HBM peak); seqs/s per layer",
        "value": round(value, 4),
        "unit": "GB/s",
        "n_gpus": int(os.environ.get("WORLD_SIZE", "1")),
        "steps": args.steps,
        "warmup": args.warmup,
        "ms_per_step": round(dt / args.steps * 1e3, 4),
        "higher_is_better": True,
        "scaling": "weak",
        "vs_baseline": None,
        "dtype": "f64",
        "data": "synthetic (seeded N(0,1) values, random block placement)",
        "config": {"workload": workload_desc(case), "global_batch": case.B,
                   "parallelism": "host cores (OpenMP)"},
        "cpu_baseline": {"value": round(value, 4), "unit": "GB/s", "cores": O.threads(),
                         "kind": "oracle", "sample": sample},
        "e2e": {"value": round(value, 4), "unit": "GB/s", "h2d_bytes_per_step": 0,
                "d2h_bytes_per_step": 0},
    }
    print(json.dumps(line), flush=True)


# ---- the prefill chunk alone ----------------------------------------------------------

def prefill_flops(case) -> float:
    """Causal attention flops of the chunk: row i of L sees P + i + 1 keys; QK^T and PV
    each take 2 flops per multiply-add."""
    pf = case.prefill
    keys = sum(pf.P + i + 1 for i in range(pf.L))
    return 4.0 * case.Hq * case.D * keys


def measured_bf16_peak():
    path = os.path.join(ROOT, "MEASURED_PEAKS.json")
    try:
        with open(path) as f:
            return float(json.load(f)["bf16_tflops"]), "measured (bf16 burst)"
    except Exception:
        return FALLBACK_BF16_TFLOPS, "fallback"


def run_prefill_only(args):
    """paged_attn_prefill_chunk on the workload's chunk, timed alone with CUDA events on
    its stream (L2 flushed between calls, untimed); tensor-core roofline."""
    rank, world, local = dist_setup()
    torch.cuda.set_device(local)
    from paged_kv_decode_11_gb300 import build as pkv_build
    pkv_build.build()
    import paged_kv_decode_11_gb300 as P
    from paged_kv_decode_11_gb300.step import MixedStep
    P.load()
    case = make_case(args.config, args.seed + rank, device="cuda")
    if case.prefill is None:
        raise SystemExit(f"--prefill-only: workload {args.config} has no prefill chunk")
    kc, vc = empty_cache(case, "cuda")
    ks = vs = None
    if case.kv_fp8:
        ks = torch.from_numpy(case.k_scales).cuda()
        vs = torch.from_numpy(case.v_scales).cuda()
    P.reshape_and_cache(case.fill_k, case.fill_v, kc, vc,
                        torch.from_numpy(case.fill_slots).cuda(), ks, vs)
    P.reshape_and_cache(case.new_k, case.new_v, kc, vc,
                        torch.from_numpy(case.new_slots).cuda(), ks, vs)
    step = MixedStep.from_case(case, kc, vc, mode="streams")
    stream = torch.cuda.current_stream()
    flush = L2Flush()
    for _ in range(args.warmup):
        step.prefill(stream)
    torch.cuda.synchronize()
    assert P.pkv_get_device_error() == 0
    sampler = ClockSampler(local)
    if rank == 0:
        sampler.start()
    K = args.steps
    ev = [(torch.cuda.Event(enable_timing=True), torch.cuda.Event(enable_timing=True))
          for _ in range(K)]
    barrier(world)
    torch.cuda.synchronize()
    t0 = time.time()
    for i in range(K):
        flush(i)
        ev[i][0].record(stream)
        step.prefill(stream)
        ev[i][1].record(stream)
    torch.cuda.synchronize()
    barrier(world)
    t1 = time.time()
    rows = sampler.stop() if rank == 0 else []
    assert P.pkv_get_device_error() == 0
    ms = allreduce(float(np.mean([a.elapsed_time(b) for a, b in ev])), "max", world)
    flops = prefill_flops(case)
    value = allreduce(flops, "sum", world) / (ms / 1e3) / 1e12
    peak, peak_kind = measured_bf16_peak()
    achieved = flops / (ms / 1e3) / 1e12
    if rank == 0:
        pf = case.prefill
        print(json.dumps({
            "metric": "causal chunked prefill: TFLOP/s (attention flops of the chunk)",
            "value": round(value, 2), "unit": "TFLOP/s", "n_gpus": world, "steps": K,
            "warmup": args.warmup, "ms_per_step": round(ms, 5), "higher_is_better": True,
            "scaling": "weak", "vs_baseline": None,
            "dtype": ("f16" if case.kv_fp8 or case.dtype == "f16" else "bf16")
                     + " tcgen05 MMA operands, fp32 TMEM accumulators",
            "data": "synthetic (seeded N(0,1) values, random block placement)",
            "config": {"workload": f"{case.name} prefill chunk alone: L{pf.L} on P{pf.P}, "
                                   f"Hq{case.Hq} Hkv{case.Hkv} D{case.D}, "
                                   f"{'E4M3' if case.kv_fp8 else case.dtype} KV, "
                                   f"{case.dtype} q, block 16",
                       "flops_per_call": flops,
                       "l2": L2Flush.describe("calls")},
            "roofline": {"kernel": "prefill_tc_kernel (one launch per call)", "bound": "tensor",
                         "achieved": round(achieved, 2), "peak": peak, "peak_kind": peak_kind,
                         "unit": "TFLOP/s", "frac": round(achieved / peak, 4), "traffic": None},
            "clocks": ClockSampler.summarise(rows, t0, t1),
            "gpu_launches": K,
        }), flush=True)
    if world > 1:
        import torch.distributed as dist
        dist.destroy_process_group()


def main():
    args = parse_args()
    if args.record_traffic:
        record_traffic(args)
    elif args.impl == "reference":
        run_reference(args)
    elif args.prefill_only:
        run_prefill_only(args)
    else:
        run_ours(args)


if __name__ == "__main__":
    main()
