#!/usr/bin/env python3
"""Benchmark of the predicate -> scan -> scatter hot path on one GB300 (or N, as replicas).

One step runs every operation of the path over one batch of seeded synthetic
input of n = 2^28 elements (the stable even/odd partition and selectivity
sweep workload, 1 GiB per int32 array):

    scan_i32      exclusive scan, int32 uniform random
    scan_f32      exclusive scan, float32 uniform on [0, 1)
    select_p01    stable select-if NONZERO, 1 % kept
    select_p50    stable select-if NONZERO, 50 % kept
    select_p99    stable select-if NONZERO, 99 % kept
    partition     stable partition, EVEN first (count pre-pass + one pass)
    radix32       LSD radix sort, 32 one-bit splits, uint32 keys + uint32 index payload
    atomic_tile_p50  atomic-counter select-if with one atomic per tile (the unordered
                  comparison path), 50 % kept; the page's one-atomic-per-survivor form is
                  timed beside the stable select at 1/50/99 % in the line's `comparator`

Every call goes through the C ABI (libgc.so) via partition_pass_tile_gb300.gc.
Inputs are 1 GiB each, larger than the 129 MB L2, so no L2 flush is needed
between timed steps.  Timing: W warm-up steps, then K timed steps between
CUDA events on the launching stream, with a barrier and synchronize on both
sides, max over ranks.  `value` counts n elements per operation and step
(radix counts its n keys once).

--impl reference times the CPU oracle (single-threaded C) on a bounded
sample of the same workload instead.
"""

from __future__ import annotations

import argparse
import hashlib
import json
import os
import platform
import statistics
import subprocess
import sys
import tempfile
import time

import numpy as np

ROOT = os.path.dirname(os.path.abspath(__file__))
if ROOT not in sys.path:
    sys.path.insert(0, ROOT)

from partition_pass_tile_gb300 import synth  # noqa: E402

METRIC = "compaction/scan Gelem/s and achieved HBM GB/s (% of GB300 peak) at n=2^28"
def workload_name(n: int) -> str:
    size = f"2^{n.bit_length() - 1}" if n & (n - 1) == 0 else str(n)
    return (f"stable even/odd partition + select-if sweep (1/50/99 %) at n={size} int32, "
            "with exclusive scan (int32, float32), 32-bit one-bit-split LSD radix sort "
            "(uint32 keys + index payload) and the atomic select comparator on the same batch")
OPS = ["scan_i32", "scan_f32", "select_p01", "select_p50", "select_p99", "partition",
       "radix32", "atomic_tile_p50"]
LAUNCHES_PER_OP = {"scan_i32": 1, "scan_f32": 1, "select_p01": 1, "select_p50": 1,
                   "select_p99": 1, "partition": 2, "radix32": 33, "atomic_tile_p50": 1}
FALLBACK_HBM_GBS = 6800.0
NOMINAL_HBM_GBS = 7900.0  # GB300 HBM3e, NVIDIA's nominal figure: a secondary denominator


def parse_args(argv=None):
    p = argparse.ArgumentParser(description=__doc__.split("\n\n")[0])
    p.add_argument("--gpus", type=int, default=1)
    p.add_argument("--steps", type=int, default=10)
    p.add_argument("--warmup", type=int, default=3)
    p.add_argument("--impl", choices=["gc", "reference"], default="gc")
    p.add_argument("--n", type=int, default=1 << 28, help="elements per array (default 2^28)")
    p.add_argument("--cpu-sample", type=int, default=1 << 24,
                   help="elements per array in the timed CPU-oracle sample")
    p.add_argument("--configs", action="store_true",
                   help="instead of the step: one line per benchmark configuration at its own size")
    p.add_argument("--kernels", action="store_true",
                   help="instead of the step: every entry point once at n elements (a workload for "
                        "an ncu launch list of every kernel), then one line per call with its bytes")
    return p.parse_args(argv)


# ---------------------------------------------------------------- ranks

def dist_env():
    return (int(os.environ.get("RANK", "0")), int(os.environ.get("LOCAL_RANK", "0")),
            int(os.environ.get("WORLD_SIZE", "1")))


def init_dist(world: int, backend: str):
    if world > 1:
        import torch.distributed as dist
        if not dist.is_initialized():
            dist.init_process_group(backend)


def barrier(world: int):
    if world > 1:
        import torch.distributed as dist
        dist.barrier()


def max_over_ranks(value: float, world: int, device=None) -> float:
    """Largest value over all ranks (the slowest rank sets the job's time)."""
    if world <= 1:
        return value
    import torch
    import torch.distributed as dist
    t = torch.tensor([value], dtype=torch.float64, device=device)
    dist.all_reduce(t, op=dist.ReduceOp.MAX)
    return float(t.item())


def sum_over_ranks(value: float, world: int, device=None) -> float:
    if world <= 1:
        return value
    import torch
    import torch.distributed as dist
    t = torch.tensor([value], dtype=torch.float64, device=device)
    dist.all_reduce(t, op=dist.ReduceOp.SUM)
    return float(t.item())


# ---------------------------------------------------------------- inputs

def rank_seed(seed: int, rank: int) -> int:
    """Rank 0 uses the recipe's seed; replicas get their own independent batch."""
    return seed + 1000 * rank


def host_inputs(n: int, rank: int = 0) -> dict:
    S = synth.SEEDS
    x = synth.uniform_i32(n, rank_seed(S["partition"], rank))
    return {
        "x": x,
        "f": synth.scan_unit_f32(n, rank_seed(S["scan_f32"], rank)),
        "s01": synth.keep_fraction(n, 0.01, rank_seed(S["keep_0.01"], rank)),
        "s50": synth.keep_fraction(n, 0.50, rank_seed(S["keep_0.50"], rank)),
        "s99": synth.keep_fraction(n, 0.99, rank_seed(S["keep_0.99"], rank)),
        "payload": np.arange(n, dtype=np.uint32),
    }


def alg_bytes(op: str, n: int, kept: dict) -> float:
    """Algorithmic bytes of one call: every input element read once, every
    output element written once (scan 8 B/elem; select 4 B + 4 B per survivor
    + the count; partition 8 B; radix 16 B per split x 32 + a 4 B histogram
    read; status words excluded)."""
    if op in ("scan_i32", "scan_f32"):
        return 8.0 * n
    if op.startswith("select_") or op.startswith("atomic_"):
        return 4.0 * n + 4.0 * kept[op] + 4
    if op == "partition":
        return 8.0 * n + 4
    if op == "radix32":
        return 16.0 * n * 32 + 4.0 * n
    raise KeyError(op)


def read_peaks() -> tuple[float, str]:
    path = os.path.join(ROOT, "MEASURED_PEAKS.json")
    try:
        with open(path) as f:
            return float(json.load(f)["hbm_gbs"]), "measured"
    except (OSError, KeyError, ValueError):
        return FALLBACK_HBM_GBS, "fallback"


# Sources that build the kernels profiles/dram_traffic.json records (the
# persistent scan, select and partition kernels and their launchers); the
# digit sort and the workspace-free entry point build none of them.
TRAFFIC_SOURCES_EXCLUDED = {"radix.cu", "noalloc.cu"}


def kernel_source_hash() -> str:
    h = hashlib.sha256()
    csrc = os.path.join(ROOT, "partition_pass_tile_gb300", "csrc")
    for name in sorted(os.listdir(csrc)):
        if name in TRAFFIC_SOURCES_EXCLUDED:
            continue
        with open(os.path.join(csrc, name), "rb") as f:
            h.update(name.encode() + b"\0" + f.read())
    return h.hexdigest()[:16]


def recorded_traffic(kernel: str, n: int):
    """DRAM bytes per launch of `kernel` from the committed ncu summary, scaled
    to n elements, or None if there is none or the kernels changed since."""
    path = os.path.join(ROOT, "profiles", "dram_traffic.json")
    try:
        with open(path) as f:
            rec = json.load(f)[kernel]
    except (OSError, KeyError, ValueError):
        return None
    if rec.get("source_hash") != kernel_source_hash():
        return None
    return float(rec["dram_bytes_per_launch"]) * n / float(rec["n"])


# ---------------------------------------------------------------- clocks

class ClockSampler:
    """nvidia-smi sampled every 200 ms while the timed region runs."""

    FIELDS = ("index,clocks.sm,clocks.max.sm,power.draw,clocks_event_reasons.active,"
              "clocks_event_reasons.hw_slowdown,clocks_event_reasons.hw_thermal_slowdown,"
              "clocks_event_reasons.sw_thermal_slowdown,clocks_event_reasons.sw_power_cap")

    def __init__(self, gpu_index: int):
        self.gpu = gpu_index
        self.proc = None
        self.tmp = None

    def __enter__(self):
        self.tmp = tempfile.NamedTemporaryFile("w+", suffix=".csv", delete=False)
        try:
            self.proc = subprocess.Popen(
                ["nvidia-smi", f"--id={self.gpu}", f"--query-gpu={self.FIELDS}",
                 "--format=csv,noheader,nounits", "-lms", "200"],
                stdout=self.tmp, stderr=subprocess.DEVNULL)
        except OSError:
            self.proc = None
        time.sleep(0.3)
        return self

    def __exit__(self, *exc):
        time.sleep(0.25)
        if self.proc is not None:
            self.proc.terminate()
            try:
                self.proc.wait(timeout=5)
            except subprocess.TimeoutExpired:
                self.proc.kill()

    def summary(self) -> dict:
        rows = []
        try:
            with open(self.tmp.name) as f:
                for line in f:
                    parts = [p.strip() for p in line.split(",")]
                    if len(parts) >= 9 and parts[1].replace(".", "").isdigit():
                        rows.append(parts)
            os.unlink(self.tmp.name)
        except OSError:
            pass
        if not rows:
            return {"sm_mhz": None, "sm_max_mhz": None, "reasons": ["clock sampling unavailable"],
                    "samples": 0}
        sm = [float(r[1]) for r in rows]
        names = ["hw_slowdown", "hw_thermal_slowdown", "sw_thermal_slowdown", "sw_power_cap"]
        reasons = sorted({names[i] for r in rows for i in range(4) if r[5 + i] == "Active"})
        loaded = [s for s in sm if s >= 0.5 * max(sm)] or sm
        return {"sm_mhz": statistics.median(loaded), "sm_max_mhz": float(rows[0][2]),
                "reasons": reasons, "samples": len(rows),
                "power_w_max": max(float(r[3]) for r in rows if r[3].replace(".", "").isdigit())
                if any(r[3].replace(".", "").isdigit() for r in rows) else None}


# ---------------------------------------------------------------- CPU oracle

def oracle_step(orc, h: dict, n: int) -> dict:
    """One pass of every operation of the step through the CPU oracle, on the
    first n elements of each input.  Returns seconds per operation."""
    import oracle as O
    t = {}
    x, f = h["x"][:n], h["f"][:n]
    calls = [
        ("scan_i32", lambda: orc.exclusive_scan(x)),
        ("scan_f32", lambda: orc.exclusive_scan(f)),
        ("select_p01", lambda: orc.select_if(h["s01"][:n], O.NONZERO)),
        ("select_p50", lambda: orc.select_if(h["s50"][:n], O.NONZERO)),
        ("select_p99", lambda: orc.select_if(h["s99"][:n], O.NONZERO)),
        ("partition", lambda: orc.partition(x, O.EVEN)),
        ("radix32", lambda: orc.split_radix(x.view(np.uint32), h["payload"][:n])),
        ("atomic_tile_p50", lambda: orc.select_if(h["s50"][:n], O.NONZERO)),
    ]
    for name, fn in calls:
        t0 = time.perf_counter()
        fn()
        t[name] = time.perf_counter() - t0
    return t


def host_cpu() -> dict:
    """The host's core count and CPU model, for the CPU-baseline record."""
    model = ""
    try:
        with open("/proc/cpuinfo") as f:
            for line in f:
                key = line.split(":")[0].strip().lower()
                if key in ("model name", "cpu part", "hardware") and ":" in line:
                    model = line.split(":", 1)[1].strip()
                    if key == "model name":
                        break
    except OSError:
        pass
    arm_parts = {"0xd4f": "Arm Neoverse V2", "0xd40": "Arm Neoverse V1", "0xd0c": "Arm Neoverse N1",
                 "0xd8e": "Arm Neoverse N3", "0xd84": "Arm Neoverse V3"}
    model = arm_parts.get(model.lower(), model)
    return {"nproc": os.cpu_count(), "cpu": model or platform.machine()}


class OneCore:
    """Pins the calling process to one core (the first it may use) while the
    single-threaded oracle is timed, then restores the affinity."""

    def __enter__(self):
        self.saved = None
        if hasattr(os, "sched_getaffinity"):
            self.saved = os.sched_getaffinity(0)
            os.sched_setaffinity(0, {min(self.saved)})
        return self

    def __exit__(self, *exc):
        if self.saved is not None:
            os.sched_setaffinity(0, self.saved)
        return False


def cpu_baseline(h: dict, sample: int) -> dict:
    import oracle
    oracle.build()
    orc = oracle.default()
    sample = min(sample, h["x"].shape[0])
    with OneCore():
        t = oracle_step(orc, h, sample)
    total = sum(t.values())
    return {"value": len(OPS) * sample / total / 1e9, "unit": "Gelem/s", "cores": 1,
            "kind": "oracle", **host_cpu(),
            "sample": f"first {sample} elements of every input array, one pass of all "
                      f"{len(OPS)} operations, single-threaded C pinned to one core, {total:.2f} s",
            "ms_per_op": {k: round(v * 1e3, 3) for k, v in t.items()}}


# ---------------------------------------------------------------- GPU arm

def run_gc(args):
    import torch

    from partition_pass_tile_gb300 import gc

    rank, local_rank, world = dist_env()
    torch.cuda.set_device(local_rank)
    init_dist(world, "nccl")
    dev = torch.device("cuda", local_rank)
    n = args.n
    gc.load()

    h = host_inputs(n, rank)

    def to_dev(a):
        t = torch.from_numpy(a.view(np.int32) if a.dtype == np.uint32 else a).to(dev)
        return t.view(torch.uint32) if a.dtype == np.uint32 else t

    d = {k: to_dev(v) for k, v in h.items()}
    out_a = torch.empty(n, dtype=torch.int32, device=dev)
    out_b = torch.empty(n, dtype=torch.int32, device=dev)
    counts = torch.zeros(8, dtype=torch.uint32, device=dev)
    ws = gc.workspace(gc.OP_SPLIT_RADIX, n, gc.F32, dev)
    assert ws.numel() >= max(gc.workspace_bytes(op, n, gc.F32) for op in range(5))
    stream = torch.cuda.Stream(device=dev)
    outf = out_a.view(torch.float32)

    def op_calls(e2e_copy=None):
        """The step's operations in order; e2e_copy(name) runs after each one."""
        xk = d["x"].view(torch.uint32)
        calls = [
            ("scan_i32", lambda: gc.exclusive_scan(d["x"], out=out_a, total=counts[0:1].view(torch.int32), ws=ws, stream=stream)),
            ("scan_f32", lambda: gc.exclusive_scan(d["f"], out=outf, total=counts[1:2].view(torch.float32), ws=ws, stream=stream)),
            ("select_p01", lambda: gc.select_if(d["s01"], "nonzero", out=out_a, count=counts[2:3], ws=ws, stream=stream)),
            ("select_p50", lambda: gc.select_if(d["s50"], "nonzero", out=out_a, count=counts[3:4], ws=ws, stream=stream)),
            ("select_p99", lambda: gc.select_if(d["s99"], "nonzero", out=out_a, count=counts[4:5], ws=ws, stream=stream)),
            ("partition", lambda: gc.partition(d["x"], "even", out=out_a, count_true=counts[5:6], ws=ws, stream=stream)),
            ("radix32", lambda: gc.split_radix(xk, d["payload"], 0, 32, keys_out=out_a.view(torch.uint32),
                                               vals_out=out_b.view(torch.uint32), ws=ws, stream=stream)),
            ("atomic_tile_p50", lambda: gc.select_if_atomic(d["s50"], "nonzero", out=out_a, count=counts[7:8], ws=ws, stream=stream, per_tile=True)),
        ]
        return calls

    def device_step(ev=None):
        for i, (name, fn) in enumerate(op_calls()):
            if ev is not None:
                ev[name][0].record(stream)
            fn()
            if ev is not None:
                ev[name][1].record(stream)

    # warm-up (also loads every kernel)
    for _ in range(max(args.warmup, 0)):
        device_step()
    stream.synchronize()
    kept_h = counts.view(torch.int32).cpu().numpy().view(np.uint32)
    kept = {"select_p01": int(kept_h[2]), "select_p50": int(kept_h[3]),
            "select_p99": int(kept_h[4]), "atomic_tile_p50": int(kept_h[7])}
    # the counts must be the true counts of the inputs (cheap host check)
    for k, key in (("select_p01", "s01"), ("select_p50", "s50"), ("select_p99", "s99")):
        assert kept[k] == int(np.count_nonzero(h[key])), k
    assert kept["atomic_tile_p50"] == kept["select_p50"]
    assert int(kept_h[5]) == int(np.count_nonzero((h["x"] & 1) == 0))

    # timed region: every event recorded on the launching stream, read after
    # the last step (no host synchronisation between steps)
    def new_ev():
        return torch.cuda.Event(enable_timing=True)
    evs = [{name: (new_ev(), new_ev()) for name in OPS} for _ in range(args.steps)]
    t_start, t_end = new_ev(), new_ev()
    barrier(world)
    torch.cuda.synchronize(dev)
    with ClockSampler(local_rank) as clocks:
        t_start.record(stream)
        for k in range(args.steps):
            device_step(evs[k])
        t_end.record(stream)
        torch.cuda.synchronize(dev)
    barrier(world)
    total_ms = max_over_ranks(t_start.elapsed_time(t_end), world, dev)
    ms_step = total_ms / args.steps
    op_ms = {name: sum(e[name][0].elapsed_time(e[name][1]) for e in evs) / args.steps
             for name in OPS}

    # The widened entry points (not part of the step): inclusive scans, the
    # parameterised-predicate select / partition and the float32-key radix sort
    # (four 8-bit digit passes over the order-preserving key, payload carried;
    # algorithmic bytes: keys and payloads read and written once per pass) on
    # the same 2^28 arrays.
    ws_sort = gc.workspace(gc.OP_RADIX_SORT, n, gc.F32, dev)
    pf = gc.predicate(d["f"], ">", 0.75)
    pi = gc.predicate(d["x"], "<", 0)
    next_calls = {
        "inclusive_scan_i32": (lambda: gc.inclusive_scan(d["x"], out=out_a, total=counts[0:1].view(torch.int32), ws=ws, stream=stream), 8.0 * n),
        "inclusive_scan_f32": (lambda: gc.inclusive_scan(d["f"], out=outf, total=counts[1:2].view(torch.float32), ws=ws, stream=stream), 8.0 * n),
        "select_pred_f32_gt_0.75": (lambda: gc.select_if_pred(d["f"], pf, out=out_a, count=counts[2:3], ws=ws, stream=stream), None),
        "partition_pred_i32_lt_0": (lambda: gc.partition_pred(d["x"], pi, out=out_a, count_true=counts[5:6], ws=ws, stream=stream), 8.0 * n + 4),
        "radix_sort_f32": (lambda: gc.radix_sort(d["f"], d["payload"], keys_out=outf, vals_out=out_b.view(torch.uint32), ws=ws_sort, stream=stream), 64.0 * n),
    }
    next_ops = {}
    for name, (fn, nbytes) in next_calls.items():
        for _ in range(max(args.warmup, 1)):
            fn()
        evn = [(new_ev(), new_ev()) for _ in range(args.steps)]
        for a_, b_ in evn:
            a_.record(stream)
            fn()
            b_.record(stream)
        torch.cuda.synchronize(dev)
        ms = sum(a_.elapsed_time(b_) for a_, b_ in evn) / args.steps
        if nbytes is None:  # select: read n, write the survivors
            kept_n = int(counts[2:3].view(torch.int32).item())
            assert kept_n == int(np.count_nonzero(h["f"] > np.float32(0.75)))
            nbytes = 4.0 * n + 4.0 * kept_n + 4
        next_ops[name] = {"ms": round(ms, 4), "gelem_s": round(n / ms / 1e6, 2),
                          "alg_gbs": round(nbytes / ms / 1e6, 1)}

    # The comparison the atomic-counter path exists for ("compaction.cu -- Day
    # 33": its cost should move with the survival rate, the scanned one's
    # should not): stable select-if against the page's comparator (one atomic
    # per survivor) and the per-tile variant, at 1 / 50 / 99 % kept, on the
    # step's arrays.  misplaced = output positions whose element differs from
    # the stable answer's, reported and never gated (the page's
    # countOutOfOrder).
    comparator = {}
    out_s = torch.empty(n, dtype=torch.int32, device=dev)
    for key, pname in (("s01", "p01"), ("s50", "p50"), ("s99", "p99")):
        xs = d[key]
        m = int(np.count_nonzero(h[key]))
        variants = {
            "select_if": lambda: gc.select_if(xs, "nonzero", out=out_s, count=counts[2:3], ws=ws, stream=stream),
            "atomic_per_survivor": lambda: gc.select_if_atomic(xs, "nonzero", out=out_a, count=counts[3:4], ws=ws, stream=stream),
            "atomic_per_tile": lambda: gc.select_if_atomic(xs, "nonzero", out=out_b, count=counts[4:5], ws=ws, stream=stream, per_tile=True),
        }
        row = {}
        for vname, fn in variants.items():
            for _ in range(max(args.warmup, 1)):
                fn()
            evn = [(new_ev(), new_ev()) for _ in range(args.steps)]
            for a_, b_ in evn:
                a_.record(stream)
                fn()
                b_.record(stream)
            torch.cuda.synchronize(dev)
            ms = sum(a_.elapsed_time(b_) for a_, b_ in evn) / args.steps
            nbytes = 4.0 * n + 4.0 * m + 4
            row[vname] = {"ms": round(ms, 4), "alg_gbs": round(nbytes / ms / 1e6, 1),
                          "frac_of_peak": round(nbytes / ms / 1e6 / read_peaks()[0], 4)}
        got_c = counts[2:5].view(torch.int32).cpu().numpy()
        assert all(int(c) == m for c in got_c), (pname, got_c, m)
        ref = out_s[:m]
        row["atomic_per_survivor"]["misplaced"] = int((out_a[:m] != ref).sum().item())
        row["atomic_per_tile"]["misplaced"] = int((out_b[:m] != ref).sum().item())
        row["kept"] = m
        comparator[pname] = row
    del out_s

    # End to end: every step copies its inputs in from pinned host memory and
    # its results back, through the C ABI.  Three streams: host-to-device
    # copies, the kernels, device-to-host copies, ordered by events.  Device
    # inputs are double-buffered by step parity, so the copies of step k + 1
    # run while step k computes.  An op with a fixed-size result (the scans,
    # the partition, the sort's keys and payloads) is copied back whole as
    # soon as it is done.  A select's result is its first `count` elements:
    # the host reads step k's counts (copied to pinned memory on the kernel
    # stream) while step k + 1 is already queued, then copies back exactly
    # those elements; select outputs are double-buffered by step parity so
    # step k + 1 does not overwrite them first.  The sort's outputs are
    # double-buffered too: otherwise each step's 22 ms sort would wait for the
    # previous step's 2 GB of keys and payloads to be copied back, and the
    # step would become that chain.
    pinned = {k: torch.from_numpy(v.view(np.int32) if v.dtype == np.uint32 else v).pin_memory()
              for k, v in h.items()}
    d_in = [d, {k: torch.empty_like(v) for k, v in d.items()}]
    SELECTS = ("select_p01", "select_p50", "select_p99", "atomic_tile_p50")
    COUNT_SLOT = {"select_p01": 2, "select_p50": 3, "select_p99": 4, "atomic_tile_p50": 7}
    DOUBLE = SELECTS + ("radix32",)
    outs = [{name: torch.empty(n, dtype=torch.int32, device=dev) for name in OPS}, {}]
    outs[1] = {name: (torch.empty(n, dtype=torch.int32, device=dev) if name in DOUBLE else outs[0][name])
               for name in OPS}
    out_vals = [torch.empty(n, dtype=torch.int32, device=dev) for _ in range(2)]
    host_outs = {name: torch.empty(n, dtype=torch.int32).pin_memory() for name in OPS}
    host_vals = torch.empty(n, dtype=torch.int32).pin_memory()
    host_counts = [torch.empty(8, dtype=torch.int32).pin_memory() for _ in range(2)]
    h2d = sum(v.numel() * v.element_size() for v in pinned.values())
    s_h2d = torch.cuda.Stream(device=dev)
    s_d2h = torch.cuda.Stream(device=dev)
    s_sel = torch.cuda.Stream(device=dev)  # survivors: not queued behind the next step's copies
    inputs_of = {"scan_i32": ["x"], "scan_f32": ["f"], "select_p01": ["s01"],
                 "select_p50": ["s50"], "select_p99": ["s99"], "partition": ["x"],
                 "radix32": ["x", "payload"], "atomic_tile_p50": ["s50"]}
    set_free = [None, None]  # event: the compute stream is done with an input set
    out_free = [{name: None for name in OPS}, {name: None for name in OPS}]  # copied back
    pending = []             # (parity, counts-copied event) of steps whose selects await copy-back
    d2h_total = [0]

    def e2e_ops(dd, o, ov):
        xk = dd["x"].view(torch.uint32)
        return {
            "scan_i32": lambda: gc.exclusive_scan(dd["x"], out=o["scan_i32"], total=counts[0:1].view(torch.int32), ws=ws, stream=stream),
            "scan_f32": lambda: gc.exclusive_scan(dd["f"], out=o["scan_f32"].view(torch.float32), total=counts[1:2].view(torch.float32), ws=ws, stream=stream),
            "select_p01": lambda: gc.select_if(dd["s01"], "nonzero", out=o["select_p01"], count=counts[2:3], ws=ws, stream=stream),
            "select_p50": lambda: gc.select_if(dd["s50"], "nonzero", out=o["select_p50"], count=counts[3:4], ws=ws, stream=stream),
            "select_p99": lambda: gc.select_if(dd["s99"], "nonzero", out=o["select_p99"], count=counts[4:5], ws=ws, stream=stream),
            "partition": lambda: gc.partition(dd["x"], "even", out=o["partition"], count_true=counts[5:6], ws=ws, stream=stream),
            "radix32": lambda: gc.split_radix(xk, dd["payload"], 0, 32, keys_out=o["radix32"].view(torch.uint32),
                                              vals_out=ov.view(torch.uint32), ws=ws, stream=stream),
            "atomic_tile_p50": lambda: gc.select_if_atomic(dd["s50"], "nonzero", out=o["atomic_tile_p50"], count=counts[7:8], ws=ws, stream=stream, per_tile=True),
        }

    def copy_back_selects(par, ready):
        """Step with parity `par` finished: copy back each select's survivors."""
        ready.synchronize()
        c = host_counts[par].numpy().view(np.uint32)
        s_sel.wait_event(ready)
        for name in SELECTS:
            m = int(c[COUNT_SLOT[name]])
            with torch.cuda.stream(s_sel):
                host_outs[name][:m].copy_(outs[par][name][:m], non_blocking=True)
            d2h_total[0] += 4 * m
            freed = torch.cuda.Event()
            freed.record(s_sel)
            out_free[par][name] = freed

    def e2e_step(k):
        par = k % 2
        dd = d_in[par]
        arrived = {}
        if set_free[par] is not None:
            s_h2d.wait_event(set_free[par])
        for key, v in pinned.items():
            dst = dd[key].view(torch.int32) if dd[key].dtype == torch.uint32 else dd[key]
            with torch.cuda.stream(s_h2d):
                dst.copy_(v, non_blocking=True)
            ev = torch.cuda.Event()
            ev.record(s_h2d)
            arrived[key] = ev
        calls = e2e_ops(dd, outs[par], out_vals[par])
        for name in OPS:
            for key in inputs_of[name]:
                stream.wait_event(arrived[key])
            if out_free[par][name] is not None:
                stream.wait_event(out_free[par][name])
            calls[name]()
            if name in SELECTS:
                continue
            done = torch.cuda.Event()
            done.record(stream)
            s_d2h.wait_event(done)
            with torch.cuda.stream(s_d2h):
                host_outs[name].copy_(outs[par][name], non_blocking=True)
                d2h_total[0] += 4 * n
                if name == "radix32":
                    host_vals.copy_(out_vals[par], non_blocking=True)
                    d2h_total[0] += 4 * n
            freed = torch.cuda.Event()
            freed.record(s_d2h)
            for q in ((par,) if name in DOUBLE else (0, 1)):
                out_free[q][name] = freed  # one buffer serves both parities unless doubled
        consumed = torch.cuda.Event()
        consumed.record(stream)
        set_free[par] = consumed
        with torch.cuda.stream(stream):
            host_counts[par].copy_(counts.view(torch.int32), non_blocking=True)
        d2h_total[0] += 4 * host_counts[par].numel()
        ready = torch.cuda.Event()
        ready.record(stream)
        pending.append((par, ready))
        if len(pending) > 1:  # the previous step's selects, while this step is queued
            copy_back_selects(*pending.pop(0))

    def drain():
        while pending:
            copy_back_selects(*pending.pop(0))

    e2e_step(0)
    e2e_step(1)
    drain()
    torch.cuda.synchronize(dev)
    e0 = torch.cuda.Event(enable_timing=True)
    e1 = torch.cuda.Event(enable_timing=True)
    barrier(world)
    torch.cuda.synchronize(dev)
    d2h_total[0] = 0
    e0.record(s_h2d)
    stream.wait_event(e0)
    s_d2h.wait_event(e0)
    s_sel.wait_event(e0)
    for k in range(args.steps):
        e2e_step(k)
    drain()
    sel_done = torch.cuda.Event()
    sel_done.record(s_sel)
    s_d2h.wait_event(sel_done)
    e1.record(s_d2h)  # the last copy back depends on every copy in and every kernel
    torch.cuda.synchronize(dev)
    barrier(world)
    e2e_ms = max_over_ranks(e0.elapsed_time(e1), world, dev) / args.steps
    d2h = d2h_total[0] / args.steps
    # the copied-back counts and survivors are the true ones (the step really ran)
    hc = host_counts[(args.steps - 1) % 2].numpy().view(np.uint32)
    assert int(hc[3]) == kept["select_p50"] and int(hc[7]) == kept["atomic_tile_p50"]
    m01 = int(hc[2])
    assert np.array_equal(host_outs["select_p01"][:m01].numpy(), h["s01"][h["s01"] != 0].view(np.int32))

    peak, peak_kind = read_peaks()
    elems_step = len(OPS) * n
    bytes_step = sum(alg_bytes(k, n, kept) for k in OPS)
    ops_report = {}
    for k in OPS:
        b = alg_bytes(k, n, kept)
        ops_report[k] = {"ms": round(op_ms[k], 4), "gelem_s": round(n / op_ms[k] / 1e6, 2),
                         "alg_gbs": round(b / op_ms[k] / 1e6, 1),
                         "frac_of_peak": round(b / op_ms[k] / 1e6 / peak, 4),
                         "launches": LAUNCHES_PER_OP[k]}
    # partition also reads its input in the count pre-pass: 12 B/element moved
    moved = 12.0 * n + 4
    ops_report["partition"]["moved_gbs"] = round(moved / op_ms["partition"] / 1e6, 1)
    ops_report["partition"]["frac_of_peak_moved"] = round(moved / op_ms["partition"] / 1e6 / peak, 4)
    # dominant kernel: the one-bit split of the radix sort (32 launches per sort)
    split_bytes = 16.0 * n
    split_ms = op_ms["radix32"] / 32.0
    achieved = split_bytes / split_ms / 1e6
    result = {
        "metric": METRIC,
        "value": round(sum_over_ranks(elems_step, world, dev) / (ms_step / 1e3) / 1e9, 3),
        "unit": "Gelem/s",
        "n_gpus": world,
        "steps": args.steps,
        "warmup": args.warmup,
        "ms_per_step": round(ms_step, 4),
        "higher_is_better": True,
        "scaling": "weak",
        "vs_baseline": None,
        "dtype": "int32/uint32/f32",
        "data": "synthetic (seeded SplitMix64)",
        "config": {"workload": workload_name(n), "n": n, "bytes_per_array": 4 * n,
                   "ops_per_step": OPS, "elements_per_step": elems_step,
                   "alg_bytes_per_step": bytes_step,
                   "alg_gbs": round(bytes_step / ms_step / 1e6, 1),
                   "frac_of_hbm_peak": round(bytes_step / ms_step / 1e6 / peak, 4),
                   "l2": f"inputs {4 * n / 2**20:.0f} MiB each, larger than the 126 MB L2: "
                         "no flush between steps",
                   "parallelism": f"replicas x{world}" if world > 1 else "single GPU"},
        "ops": ops_report,
        "next_ops": {k: dict(v, frac_of_peak=round(v["alg_gbs"] / peak, 4)) for k, v in next_ops.items()},
        "comparator": comparator,
        "roofline": {"kernel": "pipeline_kernel<256, 3, PartitionOp<256, 4, PredBitClear, VEC, payload>> (one-bit radix split)",
                     "bound": "hbm", "achieved": round(achieved, 1), "peak": peak,
                     "peak_kind": f"{peak_kind} hbm_gbs",
                     "unit": "GB/s", "frac": round(achieved / peak, 4),
                     "traffic": recorded_traffic("split_kernel", n),
                     "traffic_note": "ncu DRAM read+write bytes of one split launch at n=2^26, "
                                     "scaled by n/2^26 (profiles/dram_traffic.json); null if "
                                     "the kernels changed since",
                     "alg_bytes_per_launch": split_bytes,
                     "peak_nominal": NOMINAL_HBM_GBS,
                     "frac_of_nominal": round(achieved / NOMINAL_HBM_GBS, 4),
                     "duration_note": "radix32 call time / 32: includes the histogram pass "
                                      "(the splits clear their own status words)"},
        "clocks": clocks.summary(),
        "e2e": {"value": round(sum_over_ranks(elems_step, world, dev) / (e2e_ms / 1e3) / 1e9, 3),
                "unit": "Gelem/s", "ms_per_step": round(e2e_ms, 3),
                "h2d_bytes_per_step": int(h2d), "d2h_bytes_per_step": int(d2h),
                "path": "pinned host inputs -> H2D (own stream, inputs double-buffered by step) -> "
                        "gc_* through the C ABI -> D2H (own stream) of every result: the scans, the "
                        "partition, the sort's keys and payloads whole, each select's count survivors "
                        "(counts read one step late), every step"},
        "gpu_launches": sum(LAUNCHES_PER_OP.values()) * args.steps,
    }
    if rank == 0:
        if world == 1:
            result["cpu_baseline"] = cpu_baseline(h, args.cpu_sample)
        print(json.dumps(result), flush=True)
    if world > 1:
        import torch.distributed as dist
        dist.destroy_process_group()


# ---------------------------------------------------------------- reference arm

def run_reference(args):
    rank, _, world = dist_env()
    if rank != 0:
        return
    import oracle
    oracle.build()
    orc = oracle.default()
    sample = min(args.cpu_sample >> 2, args.n)
    h = host_inputs(sample, 0)
    with OneCore():
        for _ in range(max(args.warmup, 0)):
            oracle_step(orc, h, sample)
        t0 = time.perf_counter()
        for _ in range(args.steps):
            oracle_step(orc, h, sample)
        sec = (time.perf_counter() - t0) / max(args.steps, 1)
    value = len(OPS) * sample / sec / 1e9
    result = {
        "impl": "reference", "metric": METRIC, "value": round(value, 4), "unit": "Gelem/s",
        "n_gpus": world, "steps": args.steps, "warmup": args.warmup,
        "ms_per_step": round(sec * 1e3, 3), "higher_is_better": True, "scaling": "weak",
        "vs_baseline": None, "dtype": "int32/uint32/f64", "data": "synthetic (seeded SplitMix64)",
        "config": {"workload": workload_name(args.n), "n": args.n, "sample_n": sample,
                   "ops_per_step": OPS, "parallelism": "host CPU, one core"},
        "cpu_baseline": {"value": round(value, 4), "unit": "Gelem/s", "kind": "oracle",
                         "cores": 1, **host_cpu(),
                         "sample": f"each step: the first {sample} elements of every input "
                                   f"array of the n={args.n} workload, all {len(OPS)} "
                                   "operations, single-threaded C oracle pinned to one core"},
        "e2e": {"value": round(value, 4), "unit": "Gelem/s", "h2d_bytes_per_step": 0,
                "d2h_bytes_per_step": 0},
    }
    print(json.dumps(result), flush=True)


# ---------------------------------------------------------------- per-configuration rows

def run_configs(args):
    """One JSON line per benchmark configuration at its own size: the GPU time
    of the call through the C ABI (CUDA events on the launching stream, median
    of 20 runs, L2 flushed by a 256 MiB read before every run, so the small
    configurations are timed from HBM too), the same calls replayed from a
    CUDA graph, and the oracle's single-thread time on the same input (median
    of 3 runs below 2^24 elements, else one run).
    The flush reads, so that no dirty line of it is written back while the
    timed call runs; inputs of 2^26 elements and more exceed L2 by
    themselves and run without one."""
    import torch

    import oracle
    from partition_pass_tile_gb300 import gc, synth

    orc = oracle.default()
    torch.cuda.set_device(0)
    dev = torch.device("cuda", 0)
    stream = torch.cuda.Stream(device=dev)
    flush = torch.ones(64 << 20, dtype=torch.float32, device=dev)  # 256 MiB, twice L2
    peak, peak_kind = read_peaks()
    gc.load()

    def to_dev(a):
        t = torch.from_numpy(a.view(np.int32) if a.dtype == np.uint32 else a).to(dev)
        return t.view(torch.uint32) if a.dtype == np.uint32 else t

    def gpu_ms(fn, reps=20, n=0):
        """Median and best time of fn(), and the median of the same calls
        captured once in a CUDA graph and replayed (launch gaps shrink)."""
        for _ in range(3):
            fn()
        graph = torch.cuda.CUDAGraph()
        with torch.cuda.graph(graph, stream=stream):
            fn()
        torch.cuda.synchronize(dev)
        out = []
        for run in (fn, graph.replay):
            times = []
            for _ in range(reps):
                if n < (1 << 26):
                    with torch.cuda.stream(stream):
                        torch.max(flush)
                a, b = torch.cuda.Event(enable_timing=True), torch.cuda.Event(enable_timing=True)
                a.record(stream)
                if run is fn:
                    fn()
                else:
                    with torch.cuda.stream(stream):
                        graph.replay()
                b.record(stream)
                times.append((a, b))
            torch.cuda.synchronize(dev)
            out.append([a.elapsed_time(b) for a, b in times])
        return float(np.median(out[0])), float(np.min(out[0])), float(np.median(out[1]))

    def cpu_ms(fn, n):
        reps = 3 if n < (1 << 24) else 1
        ts = []
        with OneCore():
            for _ in range(reps):
                t0 = time.perf_counter()
                fn()
                ts.append((time.perf_counter() - t0) * 1e3)
        return float(np.median(ts))

    ws = gc.workspace(gc.OP_SPLIT_RADIX, 1 << 28, gc.F32, dev)
    cnt = torch.zeros(4, dtype=torch.uint32, device=dev)

    def row(config, n, op, t, nbytes, oms, note=""):
        ms, best, graphed = t
        r = {"config": config, "n": n, "op": op, "ms": round(ms, 4), "ms_best": round(best, 4),
             "ms_graph": round(graphed, 4),
             "gelem_s": round(n / ms / 1e6, 2), "alg_gbs": round(nbytes / ms / 1e6, 1),
             "frac_of_peak": round(nbytes / ms / 1e6 / peak, 4), "peak": peak,
             "peak_kind": peak_kind, "frac_of_nominal": round(nbytes / ms / 1e6 / NOMINAL_HBM_GBS, 4),
             "oracle_ms_1core": round(oms, 1), **host_cpu()}
        if note:
            r["note"] = note
        print(json.dumps(r), flush=True)

    def select_row(config, x, pred, name):
        n = x.shape[0]
        xd = to_dev(x)
        out = torch.empty_like(xd)
        kept = int(np.count_nonzero(x != 0) if pred == "nonzero" else np.count_nonzero(x & 1))
        ms = gpu_ms(lambda: gc.select_if(xd, pred, out=out, count=cnt[0:1], ws=ws, stream=stream), n=n)
        code = oracle.NONZERO if pred == "nonzero" else oracle.ODD
        row(config, n, name, ms, 4.0 * n + 4.0 * kept + 4, cpu_ms(lambda: orc.select_if(x, code), n))

    def scan_row(config, x, name):
        n = x.shape[0]
        xd = to_dev(x)
        out = torch.empty_like(xd)
        tot = torch.empty(1, dtype=xd.dtype, device=dev)
        ms = gpu_ms(lambda: gc.exclusive_scan(xd, out=out, total=tot, ws=ws, stream=stream), n=n)
        row(config, n, name, ms, 8.0 * n, cpu_ms(lambda: orc.exclusive_scan(x), n))

    select_row("1 remove zeros", synth.remove_zeros(), "nonzero", "select NONZERO")
    scan_row("2 scan", synth.scan_mod8(), "exclusive scan int32 (i%8)+1")
    scan_row("2 scan", synth.scan_unit_f32(), "exclusive scan float32 U[0,1)")
    for n in (synth.SIZES["keep_odd"], synth.SIZES["keep_odd_literal"]):
        x = synth.uniform_i32(n, synth.SEEDS["keep_odd"])
        select_row("3 keep odd", x, "odd", "select ODD")
        xd = to_dev(x)
        out = torch.empty_like(xd)
        kept = int(np.count_nonzero(x & 1))
        for per_tile, label in ((False, "one atomic per survivor"), (True, "one atomic per tile")):
            ms = gpu_ms(lambda: gc.select_if_atomic(xd, "odd", out=out, count=cnt[1:2], ws=ws, stream=stream,
                                                    per_tile=per_tile), n=n)
            row("3 keep odd", n, f"atomic comparator ODD, {label} (multiset)", ms, 4.0 * n + 4.0 * kept + 4,
                cpu_ms(lambda: orc.select_if(x, oracle.ODD), n), "oracle: the ordered select")
        del xd, out
    n = synth.SIZES["partition"]
    x = synth.uniform_i32(n, synth.SEEDS["partition"])
    xd = to_dev(x)
    out = torch.empty_like(xd)
    ms = gpu_ms(lambda: gc.partition(xd, "even", out=out, count_true=cnt[2:3], ws=ws, stream=stream), n=n)
    row("4 partition", n, "partition EVEN", ms, 8.0 * n, cpu_ms(lambda: orc.partition(x, oracle.EVEN), n),
        "algorithmic 8 B/elem; the count pre-pass makes 12 B moved")
    del xd, out
    for p, seed in ((0.01, 41), (0.50, 42), (0.99, 43)):
        select_row("4 sweep", synth.keep_fraction(n, p, seed), "nonzero", f"select NONZERO p={p}")
    n = synth.SIZES["radix"]
    keys, vals = synth.radix_keys(n, synth.SEEDS["radix"])
    kd, vd = to_dev(keys), to_dev(vals)
    ko, vo = torch.empty_like(kd), torch.empty_like(vd)
    ms = gpu_ms(lambda: gc.split_radix(kd, vd, 0, 32, keys_out=ko, vals_out=vo, ws=ws, stream=stream), reps=5, n=n)
    row("5 radix", n, "32 one-bit splits, uint32 keys + payload", ms, (16.0 * 32 + 4.0) * n,
        cpu_ms(lambda: orc.split_radix(keys, vals), n))
    ws_sort = gc.workspace(gc.OP_RADIX_SORT, n, gc.U32, dev)
    ms = gpu_ms(lambda: gc.radix_sort(kd, vd, keys_out=ko, vals_out=vo, ws=ws_sort, stream=stream), reps=5, n=n)
    row("5 radix", n, "gc_radix_sort (four 8-bit digit passes), same keys + payload", ms, 64.0 * n,
        cpu_ms(lambda: orc.radix_sort(keys, vals), n), "algorithmic 64 B/key: keys and payloads once per pass")
    del kd, vd, ko, vo, ws_sort
    for n in (1 << 26, 1 << 28):
        scan_row("roofline", synth.uniform_i32(n, synth.SEEDS["partition"]), "exclusive scan int32")
        scan_row("roofline", synth.scan_unit_f32(n, synth.SEEDS["scan_f32"]), "exclusive scan float32")
        select_row("roofline", synth.keep_fraction(n, 0.5, 42), "nonzero", "select NONZERO p=0.5")
        select_row("roofline", synth.keep_fraction(n, 0.01, 41), "nonzero", "select NONZERO p=0.01")

    # Pointers 4-byte but not 16-byte aligned: the one-tile-per-CTA kernels
    # (dynamic tile ids, warp look-back, register tiles), at 2^26.
    n = 1 << 26
    for name, a, op in (("exclusive scan int32", synth.uniform_i32(n, 4), "scan"),
                        ("select NONZERO p=0.5", synth.keep_fraction(n, 0.5, 42), "select"),
                        ("partition EVEN", synth.uniform_i32(n, 4), "partition")):
        big = torch.zeros(n + 1, dtype=torch.int32)
        big[1:] = torch.from_numpy(a)
        xd = big.to(dev)[1:]
        ob = torch.empty(n + 1, dtype=torch.int32, device=dev)
        out = ob[1:]
        if op == "scan":
            ms = gpu_ms(lambda: gc.exclusive_scan(xd, out=out, total=cnt[0:1].view(torch.int32), ws=ws, stream=stream), n=n)
            nbytes, oms = 8.0 * n, cpu_ms(lambda: orc.exclusive_scan(a), n)
        elif op == "select":
            kept = int(np.count_nonzero(a))
            ms = gpu_ms(lambda: gc.select_if(xd, "nonzero", out=out, count=cnt[0:1], ws=ws, stream=stream), n=n)
            nbytes, oms = 4.0 * n + 4.0 * kept + 4, cpu_ms(lambda: orc.select_if(a, oracle.NONZERO), n)
        else:
            ms = gpu_ms(lambda: gc.partition(xd, "even", out=out, count_true=cnt[0:1], ws=ws, stream=stream), n=n)
            nbytes, oms = 8.0 * n, cpu_ms(lambda: orc.partition(a, oracle.EVEN), n)
        row("misaligned (4-byte) pointers", n, name, ms, nbytes, oms,
            "input and output one element into their allocations: the one-tile-per-CTA kernels")
        del xd, ob, out

    # The sharded path on one GPU: P = 4 shards of the 2^28 array, each a
    # pre-pass, the offsets of its shard and the placed pass; the whole
    # sequence timed.  Algorithmic bytes are the whole array's; the pre-pass
    # reads every element once more.
    from partition_pass_tile_gb300 import shard
    n, P = 1 << 28, 4
    bounds = [shard.shard_bounds(n, P, r) for r in range(P)]
    sizes = [b - a for a, b in bounds]
    totals = torch.empty(P, dtype=torch.uint32, device=dev)
    itot = totals.view(torch.int32)
    offs = torch.empty((P, 2), dtype=torch.int64, device=dev)
    carries = torch.empty(P, dtype=torch.int32, device=dev)
    x = synth.uniform_i32(n, synth.SEEDS["partition"])
    xd = to_dev(x)
    out = torch.empty_like(xd)

    def sharded_scan():
        for r, (a, b) in enumerate(bounds):
            gc.reduce(xd[a:b], total=itot[r:r + 1], ws=ws, stream=stream)
        for r, (a, b) in enumerate(bounds):
            gc.shard_offsets(gc.OP_EXCLUSIVE_SCAN, itot, r, out=carries[r:r + 1], stream=stream)
            gc.exclusive_scan_carry(xd[a:b], carries[r:r + 1], out=out[a:b], with_total=False, ws=ws,
                                    stream=stream)

    def sharded_partition():
        for r, (a, b) in enumerate(bounds):
            gc.count_if(xd[a:b], "even", count=totals[r:r + 1], ws=ws, stream=stream)
        for r, (a, b) in enumerate(bounds):
            gc.shard_offsets(gc.OP_PARTITION, totals, r, sizes=sizes, dtype=gc.U32, out=offs[r], stream=stream)
            gc.partition_at(xd[a:b], "even", out, offs[r], count_true=cnt[r:r + 1] if r < 4 else None,
                            ws=ws, stream=stream)
    ms = gpu_ms(sharded_scan, reps=5, n=n)
    row("sharded, 4 shards on one GPU", n, "exclusive scan int32 (reduce + carry-in scan)", ms, 8.0 * n,
        cpu_ms(lambda: orc.exclusive_scan(x), n), "moves 12 B/element: the pre-pass reads the input once more")
    ms = gpu_ms(sharded_partition, reps=5, n=n)
    row("sharded, 4 shards on one GPU", n, "partition EVEN (count + placed pass)", ms, 8.0 * n,
        cpu_ms(lambda: orc.partition(x, oracle.EVEN), n), "moves 12 B/element, as the one-array partition")
    del xd, out
    y = synth.keep_fraction(n, 0.5, 42)
    yd = to_dev(y)
    out = torch.empty_like(yd)
    kept = int(np.count_nonzero(y))

    def sharded_select():
        for r, (a, b) in enumerate(bounds):
            gc.count_if(yd[a:b], "nonzero", count=totals[r:r + 1], ws=ws, stream=stream)
        for r, (a, b) in enumerate(bounds):
            gc.shard_offsets(gc.OP_SELECT_IF, totals, r, dtype=gc.U32, out=offs[r, :1], stream=stream)
            gc.select_if_at(yd[a:b], "nonzero", out, offs[r, :1], count=cnt[r:r + 1], ws=ws, stream=stream)
    ms = gpu_ms(sharded_select, reps=5, n=n)
    row("sharded, 4 shards on one GPU", n, "select NONZERO p=0.5 (count + placed pass)", ms,
        4.0 * n + 4.0 * kept + 4, cpu_ms(lambda: orc.select_if(y, oracle.NONZERO), n),
        "moves 8 + 4 * kept B/element: the pre-pass reads the input once more")


# ---------------------------------------------------------------- every kernel once

def run_kernels(args):
    """Every entry point of the library once at n elements, on one stream, in
    a fixed order, so that an ncu capture of this process lists every kernel
    (the persistent pipelines for each op and predicate kind, the
    one-tile-per-CTA kernels through pointers one element into their
    allocations, the pre-passes, the comparators, the sorts and the sharded
    calls).  Prints one JSON line per call: its name, kernels launched and
    algorithmic bytes, for the summary of the capture."""
    import torch

    from partition_pass_tile_gb300 import gc, synth

    n = args.n
    dev = torch.device("cuda", 0)
    torch.cuda.set_device(dev)
    s = torch.cuda.Stream(device=dev)
    gc.load()

    def to_dev(a, off=0):
        base = a.view(np.int32) if a.dtype == np.uint32 else a
        t = torch.from_numpy(base)
        if off:
            big = torch.zeros(t.numel() + off, dtype=t.dtype)
            big[off:] = t
            g = big.to(dev)[off:]
        else:
            g = t.to(dev)
        return g.view(torch.uint32) if a.dtype == np.uint32 else g

    x = synth.uniform_i32(n, 4)
    f = synth.scan_unit_f32(n, 2)
    y = synth.keep_fraction(n, 0.5, 42)
    keys, vals = synth.radix_keys(n, 5)
    xd, fd, yd = to_dev(x), to_dev(f), to_dev(y)
    kd, vd = to_dev(keys), to_dev(vals)
    xo, yo = to_dev(x, 1), to_dev(y, 1)  # 4-byte, not 16-byte aligned
    out = torch.empty(n + 4, dtype=torch.int32, device=dev)
    out2 = torch.empty(n + 4, dtype=torch.int32, device=dev)
    o_al, o_mis = out[:n], out[1:n + 1]
    cnt = torch.zeros(8, dtype=torch.uint32, device=dev)
    ws = gc.workspace(gc.OP_RADIX_SORT, n, gc.F32, dev)
    kept = int(np.count_nonzero(y))
    sel_b = 4.0 * n + 4.0 * kept + 4
    from partition_pass_tile_gb300 import shard
    P = 4
    bounds = [shard.shard_bounds(n, P, r) for r in range(P)]
    totals = torch.empty(P, dtype=torch.int32, device=dev)
    carry = torch.empty(1, dtype=torch.int32, device=dev)
    pf = gc.predicate(fd, ">", 0.75)
    calls = [
        ("scan_i32", 1, 8.0 * n, lambda: gc.exclusive_scan(xd, out=o_al, total=cnt[0:1].view(torch.int32), ws=ws, stream=s)),
        ("scan_f32", 1, 8.0 * n, lambda: gc.exclusive_scan(fd, out=o_al.view(torch.float32), total=cnt[0:1].view(torch.float32), ws=ws, stream=s)),
        ("inclusive_scan_i32", 1, 8.0 * n, lambda: gc.inclusive_scan(xd, out=o_al, total=cnt[0:1].view(torch.int32), ws=ws, stream=s)),
        ("select_p50", 1, sel_b, lambda: gc.select_if(yd, "nonzero", out=o_al, count=cnt[1:2], ws=ws, stream=s)),
        ("select_pred_f32_gt_0.75", 1, None, lambda: gc.select_if_pred(fd, pf, out=o_al, count=cnt[1:2], ws=ws, stream=s)),
        ("partition_even", 2, 8.0 * n, lambda: gc.partition(xd, "even", out=o_al, count_true=cnt[2:3], ws=ws, stream=s)),
        ("partition_pred_i32_lt_0", 2, 8.0 * n, lambda: gc.partition_pred(xd, gc.predicate(xd, "<", 0), out=o_al, count_true=cnt[2:3], ws=ws, stream=s)),
        ("atomic_per_survivor_p50", 1, sel_b, lambda: gc.select_if_atomic(yd, "nonzero", out=o_al, count=cnt[3:4], ws=ws, stream=s)),
        ("atomic_per_tile_p50", 1, sel_b, lambda: gc.select_if_atomic(yd, "nonzero", out=o_al, count=cnt[3:4], ws=ws, stream=s, per_tile=True)),
        ("misaligned_scan_i32", 1, 8.0 * n, lambda: gc.exclusive_scan(xo, out=o_mis, total=cnt[0:1].view(torch.int32), ws=ws, stream=s)),
        ("misaligned_select_p50", 1, sel_b, lambda: gc.select_if(yo, "nonzero", out=o_mis, count=cnt[1:2], ws=ws, stream=s)),
        ("misaligned_partition_even", 2, 8.0 * n, lambda: gc.partition(xo, "even", out=o_mis, count_true=cnt[2:3], ws=ws, stream=s)),
        ("reduce_i32", 1, 4.0 * n, lambda: gc.reduce(xd, total=totals[0:1], ws=ws, stream=s)),
        ("count_if_even", 1, 4.0 * n, lambda: gc.count_if(xd, "even", count=cnt[4:5], ws=ws, stream=s)),
        ("shard_offsets", 1, 0.0, lambda: gc.shard_offsets(gc.OP_EXCLUSIVE_SCAN, totals, 2, out=carry, stream=s)),
        ("scan_carry_i32", 1, 8.0 * n, lambda: gc.exclusive_scan_carry(xd, carry, out=o_al, with_total=False, ws=ws, stream=s)),
        ("split_radix_1bit", 2, 16.0 * n + 4.0 * n, lambda: gc.split_radix(kd, vd, 0, 1, keys_out=o_al.view(torch.uint32), vals_out=out2[:n].view(torch.uint32), ws=ws, stream=s)),
        ("radix_sort_u32_digits", 12, 64.0 * n, lambda: gc.radix_sort(kd, vd, keys_out=o_al.view(torch.uint32), vals_out=out2[:n].view(torch.uint32), ws=ws, stream=s)),
    ]
    for name, launches, nbytes, fn in calls:
        fn()
        torch.cuda.synchronize(dev)
        if nbytes is None:
            m = int(cnt[1:2].view(torch.int32).item())
            nbytes = 4.0 * n + 4.0 * m + 4
        print(json.dumps({"call": name, "n": n, "launches": launches, "alg_bytes": nbytes}), flush=True)
    # the placed passes of one shard (shard 2 of 4), as the first shard of
    # its own output: base 0, and the partition's rejected run from T
    a, b = bounds[2]
    base = torch.zeros(1, dtype=torch.int64, device=dev)
    gc.select_if_at(yd[a:b], "nonzero", o_al, base, count=cnt[6:7], ws=ws, stream=s)
    torch.cuda.synchronize(dev)
    print(json.dumps({"call": "select_at_shard", "n": b - a, "launches": 1,
                      "alg_bytes": 4.0 * (b - a) + 4.0 * int(cnt[6:7].view(torch.int32).item())}), flush=True)
    gc.count_if(xd[a:b], "even", count=cnt[5:6], ws=ws, stream=s)
    offs = gc.shard_offsets(gc.OP_PARTITION, cnt[5:6], 0, sizes=[b - a], dtype=gc.U32, stream=s)
    gc.partition_at(xd[a:b], "even", o_al, offs, count_true=cnt[7:8], ws=ws, stream=s)
    torch.cuda.synchronize(dev)
    print(json.dumps({"call": "partition_at_shard", "n": b - a, "launches": 3, "alg_bytes": 8.0 * (b - a)}),
          flush=True)


def main(argv=None):
    args = parse_args(argv)
    if args.kernels:
        run_kernels(args)
        return
    if args.configs:
        run_configs(args)
        return
    if args.impl == "reference":
        run_reference(args)
    else:
        run_gc(args)


if __name__ == "__main__":
    main()
