#!/usr/bin/env python
"""Benchmark: GDN speculative verify + all-layer replay commit on one GB300.

A step is one pass of the whole hot path over one batch: the verify of
every GDN layer (one launch per layer, replayed from a CUDA graph captured
from the public API calls, as a serving engine runs its forward) followed by
the single all-layer commit launch (called eagerly, outside the graph, as an
engine commits after sampling).  Inputs are resident in HBM.  A timed unit
whose bytes are under three times the L2 size (the one-layer workload, the
conv-state commit) gets a write of twice the L2 size before every timed
iteration, outside its events, so that each iteration starts cold; the
36-layer steps touch ~100x the L2 and need none.

The same run then measures every benchmark configuration (tiny, the
one-layer serving shape, the three long/ragged seeds, align mode with fp32
and bf16 states) and reports µs per verify, per native snapshot and per
all-layer commit with their HBM fractions in the line's `configs` block.

Prints one JSON line (rank 0).  --impl reference times the fp64 CPU oracle
instead: whole steps of the same workload when they fit the time budget,
else a bounded sample of each step.  --gpus N without a torchrun
environment re-launches this script under torchrun with N ranks.
"""
from __future__ import annotations

import argparse
import hashlib
import json
import os
import re
import statistics
import subprocess
import sys
import tempfile
import time

ROOT = os.path.dirname(os.path.abspath(__file__))
sys.path.insert(0, ROOT)

import torch  # noqa: E402

from spec_decode_recurrent_gb300 import api, build, dist, roofline, step, workloads  # noqa: E402

METRIC = "GDN verify+all-layer commit µs/step and achieved HBM GB/s vs ~8 TB/s roofline"
UNIT = "us/step"
NOMINAL_HBM_GBS = 7900.0  # GB300 HBM3e nominal bandwidth, reported beside the measured peak

DESCR = {
    "tiny": "1 GDN layer, batch 2, HK=HV=2, K=V=16, window 4, accepted [1,3], fp32 q/k/v and "
            "state, slots [0,1], seed 0",
    "all_layer": "36 GDN layers, batch 64 (56 live rows + 8 graph-padding rows with null slot "
                 "and window 0), HK=16 HV=32 K=V=128, window 4 (MTP 3), accepted uniform 1..4, "
                 "bf16 q/k/v, fp32 [V,K] state, slots a random permutation of a 256-slot pool, seed 2",
    "layer": "1 GDN layer at serving shape, batch 16, HK=16 HV=32 K=V=128, window 4, "
             "accepted uniform 1..4, bf16 q/k/v, fp32 state, seed 1",
    "mtp5": "all_layer shapes with window 6 (MTP 5) and accepted lengths drawn from measured "
            "per-position acceptance .856/.694/.558/.457/.376 (mean 3.941), seed 5",
    "long_ragged": "36 GDN layers, batch 256, window 6 mixed with ragged 4/1/3, permuted "
                   "non-contiguous rows, strided fused q/k/v, gates U(-20,20), 512-slot pools, seed 30",
    "align": "36 GDN layers, batch 128, window 4, align mode with block size 4, boundary "
             "slot often equal to the source slot, 384-slot pools, seed 4",
    "kda_all_layer": "all_layer shapes (36 layers, batch 64 with 8 padding rows, HK=16 HV=32 "
                     "K=V=128, window 4) with the per-channel (KDA) decay: gate inputs "
                     "a [T,HV,K] ~ N(0,1), dt_bias [HV,K] ~ U(-1,1), gate records [B,HV,W,K], "
                     "seed 6",
}


def parse(argv=None):
    p = argparse.ArgumentParser(description=__doc__)
    p.add_argument("--gpus", type=int, default=1)
    p.add_argument("--steps", type=int, default=500)
    p.add_argument("--warmup", type=int, default=10)
    p.add_argument("--impl", choices=["gb300", "reference"], default="gb300")
    p.add_argument("--workload", choices=sorted(DESCR), default="all_layer")
    p.add_argument("--state-dtype", choices=["f32", "bf16"], default="f32")
    p.add_argument("--e2e-steps", type=int, default=50)
    p.add_argument("--cpu-seconds", type=float, default=15.0,
                   help="CPU time budget of the oracle baseline sample")
    p.add_argument("--no-cpu-baseline", action="store_true")
    p.add_argument("--no-e2e", action="store_true")
    p.add_argument("--layers", type=int, default=None,
                   help="fewer layers (for small profiler captures; not a bench line)")
    p.add_argument("--grouped-commit", action="store_true",
                   help="measure the grouped commit (3 KV-cache groups x 6 layers, one launch) "
                        "against one commit call per group; prints its own JSON line")
    p.add_argument("--no-configs", action="store_true",
                   help="skip the per-configuration block (profiler runs)")
    p.add_argument("--seed", type=int, default=None, help="workload seed (default: its own)")
    return p.parse_args(argv)


DEFAULT_SEED = {"tiny": 0, "all_layer": 2, "layer": 1, "long_ragged": 30, "align": 4, "mtp5": 5,
                "kda_all_layer": 6}


def make_workload(name, device, rank, state_dtype, layers=None, seed=None):
    fn = workloads.WORKLOADS[name]
    kw = dict(device=device, sentinel=False)
    if layers is not None:
        kw["L"] = layers
    base = DEFAULT_SEED[name] if seed is None else seed
    kw["seed"] = dist.replica_seed(base, rank)
    if state_dtype == torch.bfloat16:
        import inspect
        if "state_dtype" not in inspect.signature(fn).parameters:
            raise SystemExit(f"workload {name} has no bf16-state form")
        kw["state_dtype"] = state_dtype
    return fn(**kw)


# --------------------------------------------------------------- clocks
CLOCK_FIELDS = ("index,clocks.sm,clocks.max.sm,power.draw,clocks_event_reasons.active,"
                "clocks_event_reasons.hw_slowdown,clocks_event_reasons.hw_thermal_slowdown,"
                "clocks_event_reasons.sw_thermal_slowdown,clocks_event_reasons.sw_power_cap")


class ClockSampler:
    def __init__(self, device):
        self.proc = None
        self.file = None
        try:
            uuid = str(torch.cuda.get_device_properties(device).uuid)
            self.gpu_id = uuid if uuid.startswith("GPU-") else "GPU-" + uuid
        except Exception:
            self.gpu_id = None

    def start(self):
        self.file = tempfile.NamedTemporaryFile("w+", suffix=".csv", delete=False)
        cmd = ["nvidia-smi", f"--query-gpu={CLOCK_FIELDS}", "--format=csv,noheader,nounits",
               "-lms", "100"]
        if self.gpu_id:
            cmd.insert(1, f"--id={self.gpu_id}")
        try:
            self.proc = subprocess.Popen(cmd, stdout=self.file, stderr=subprocess.DEVNULL)
        except OSError:
            self.proc = None

    def stop(self):
        if self.proc is None:
            return {"sm_mhz": None, "sm_max_mhz": None, "reasons": ["nvidia-smi unavailable"]}
        self.proc.terminate()
        try:
            self.proc.wait(timeout=5)
        except subprocess.TimeoutExpired:
            self.proc.kill()
        self.file.flush()
        self.file.seek(0)
        sm, smax, power, reasons = [], [], [], set()
        names = ["hw_slowdown", "hw_thermal_slowdown", "sw_thermal_slowdown", "sw_power_cap"]
        for line in self.file.read().splitlines():
            cols = [c.strip() for c in line.split(",")]
            if len(cols) < 9:
                continue
            try:
                sm.append(float(cols[1]))
                smax.append(float(cols[2]))
                power.append(float(cols[3]))
            except ValueError:
                continue
            for n, c in zip(names, cols[5:9]):
                if c.lower() == "active":
                    reasons.add(n)
        os.unlink(self.file.name)
        return {"sm_mhz": statistics.median(sm) if sm else None,
                "sm_max_mhz": max(smax) if smax else None,
                "power_w_max": max(power) if power else None,
                "samples": len(sm), "reasons": sorted(reasons)}


# ---------------------------------------------------------------- peaks
def l2_bytes(dev=None):
    """L2 size of the device (GB300: ~126 MB); the nominal size without one."""
    if torch.cuda.is_available():
        return int(torch.cuda.get_device_properties(dev or 0).L2_cache_size)
    return 126 * 1024 * 1024


def l2_rule(footprint, l2):
    """(flush?, description) for a timed unit touching `footprint` bytes."""
    mb = footprint / 1e6
    if footprint < 3 * l2:
        return True, (f"flush: {mb:.0f} MB per timed unit < 3x the {l2 / 1e6:.0f} MB L2; before "
                      f"every timed iteration, outside its events, a {2 * l2 / 1e6:.0f} MB buffer "
                      f"is written and another {2 * l2 / 1e6:.0f} MB buffer read, so the unit "
                      "starts with none of its data in L2 and no dirty lines left to write back")
    return False, (f"no flush: inputs larger than L2 ({mb / 1e3:.1f} GB per step vs "
                   f"{l2 / 1e9:.2f} GB L2)")


class L2Scrub:
    """Before a timed iteration whose bytes are under three times the L2:
    write a buffer of twice the L2 size (evicting the unit's data), then read
    another of twice the L2 size, so that the write's dirty lines drain to
    DRAM here, outside the timed region, instead of during the timed kernel
    (which would then pay for writing back a buffer it never touched)."""

    def __init__(self, dev, footprint):
        self.l2 = l2_bytes(dev)
        self.footprint = int(footprint)
        self.on, self.text = l2_rule(self.footprint, self.l2)
        n = 2 * self.l2 // 4
        self.wbuf = torch.empty(n, dtype=torch.float32, device=dev) if self.on else None
        self.rbuf = torch.ones(n, dtype=torch.float32, device=dev) if self.on else None
        self.sink = torch.empty((), dtype=torch.float32, device=dev) if self.on else None
        self.n = 0

    def __call__(self):
        if self.on:
            self.n += 1
            self.wbuf.fill_(float(self.n & 1))
            torch.sum(self.rbuf, dim=0, out=self.sink)

    def describe(self):
        return self.text


def measured_peaks():
    path = os.path.join(ROOT, "MEASURED_PEAKS.json")
    try:
        with open(path) as f:
            d = json.load(f)
        return float(d["hbm_gbs"]), "measured"
    except Exception:
        return 6800.0, "fallback"


def source_hash(files):
    """Hash of the kernel sources with comments and whitespace runs removed:
    an edit to a comment leaves a profile's counters valid, a code edit
    does not."""
    h = hashlib.sha256()
    for f in files:
        with open(os.path.join(ROOT, f), encoding="utf-8") as fh:
            text = fh.read()
        text = re.sub(r"/\*.*?\*/", " ", text, flags=re.S)
        text = re.sub(r"//[^\n]*", " ", text)
        h.update(" ".join(text.split()).encode())
    return h.hexdigest()[:16]


COMMIT_SOURCES = ["spec_decode_recurrent_gb300/csrc/gdn_commit.cu",
                  "spec_decode_recurrent_gb300/csrc/gdn_device.cuh",
                  "spec_decode_recurrent_gb300/csrc/gdn_async.cuh"]
VERIFY_SOURCES = ["spec_decode_recurrent_gb300/csrc/gdn_verify.cu",
                  "spec_decode_recurrent_gb300/csrc/gdn_verify_impl.cuh",
                  "spec_decode_recurrent_gb300/csrc/gdn_verify_k128.cu",
                  "spec_decode_recurrent_gb300/csrc/gdn_verify_k128_kda.cu",
                  "spec_decode_recurrent_gb300/csrc/gdn_verify_k64.cu",
                  "spec_decode_recurrent_gb300/csrc/gdn_verify_k16_k32.cu",
                  "spec_decode_recurrent_gb300/csrc/gdn_device.cuh",
                  "spec_decode_recurrent_gb300/csrc/gdn_async.cuh"]


def profiled_traffic(kernel, workload, sources, state_dtype="f32"):
    """DRAM bytes per launch from the committed ncu summary
    profiles/<kernel>_<workload>[_bf16].md (the suffix for a bf16 state), if
    it was taken from the current kernel source (else None)."""
    suffix = "_bf16" if state_dtype == "bf16" else ""
    path = os.path.join(ROOT, "profiles", f"{kernel}_{workload}{suffix}.md")
    if not os.path.exists(path):
        return None
    text = open(path).read()
    m = re.search(r"source_sha:\s*([0-9a-f]+)", text)
    t = re.search(r"traffic_bytes_per_launch:\s*([0-9.eE+]+)", text)
    if not m or not t or m.group(1) != source_hash(sources):
        return None
    return float(t.group(1))


def workload_text(args):
    text = f"{args.workload}: {DESCR[args.workload]}"
    if args.seed is not None:
        text += f" (seed overridden: {args.seed})"
    return text


def config_dict(args, sb, world_size):
    """The `config` object of the JSON line; both arms print the same one."""
    footprint = roofline.commit_bytes(sb) + roofline.verify_bytes_per_layer(sb) * sb.L
    return {
        "workload": workload_text(args),
        "layers": sb.L, "batch": sb.B, "heads_k": sb.HK, "heads_v": sb.HV,
        "head_k": sb.K, "head_v": sb.V, "window": sb.W,
        "state_dtype": args.state_dtype,
        "qkv_dtype": "bf16" if sb.qkv_dtype == torch.bfloat16 else "f32",
        "parallelism": f"replicas x{world_size} (no collective on the path)",
        "l2": l2_rule(footprint, l2_bytes())[1],
        "step": "verify of every layer (CUDA graph of the per-layer API calls) + one "
                "all-layer commit call",
    }


# ---------------------------------------------------------- the GPU arm
def run_gpu(args, rank, local_rank, world_size):
    torch.cuda.set_device(local_rank)
    dev = torch.device("cuda", local_rank)
    build.build()
    api.load()
    sd = torch.bfloat16 if args.state_dtype == "bf16" else torch.float32
    sb = make_workload(args.workload, dev, rank, sd, args.layers, args.seed)
    arena = step.pack_inputs(sb)   # one contiguous buffer of the step's inputs
    bufs = step.StepBuffers(sb)
    stream = torch.cuda.current_stream()

    # eager warm-up (loads the kernels), then capture the verify of all layers
    for _ in range(2):
        step.verify_all(sb, bufs)
        step.commit(sb, bufs)
    torch.cuda.synchronize()
    graph = torch.cuda.CUDAGraph()
    with torch.cuda.graph(graph):
        step.verify_all(sb, bufs)
    torch.cuda.synchronize()

    def one_step():
        graph.replay()
        step.commit(sb, bufs)

    for _ in range(args.warmup):
        one_step()
    torch.cuda.synchronize()
    dist.barrier()

    K = args.steps
    cbytes = roofline.commit_bytes(sb)
    vbytes = roofline.verify_bytes_per_layer(sb)
    scrub = L2Scrub(dev, cbytes + vbytes * sb.L)
    ev = [[torch.cuda.Event(enable_timing=True) for _ in range(4)] for _ in range(K)]
    clocks = ClockSampler(dev)
    clocks.start()
    time.sleep(0.3)
    dist.barrier()
    torch.cuda.synchronize()
    t0 = time.perf_counter()
    for i in range(K):
        scrub()
        ev[i][0].record(stream)
        graph.replay()
        ev[i][1].record(stream)
        scrub()     # a small step: the commit starts cold too, as after a model's forward
        ev[i][2].record(stream)
        step.commit(sb, bufs)
        ev[i][3].record(stream)
    torch.cuda.synchronize()
    wall = time.perf_counter() - t0
    dist.barrier()
    clk = clocks.stop()
    # device time of the K steps: back to back without a scrub, the sum of
    # the verify and commit events with one (the scrubs fall between them)
    verify_ms = [e[0].elapsed_time(e[1]) for e in ev]
    commit_ms = [e[2].elapsed_time(e[3]) for e in ev]
    total_ms = (sum(verify_ms) + sum(commit_ms) if scrub.on
                else ev[0][0].elapsed_time(ev[-1][3]))
    assert int(bufs.err.item()) == 0, "row errors in the benchmark workload"
    total_ms = dist.max_over_ranks(total_ms, dev)
    ms_per_step = total_ms / K

    commit_us = statistics.mean(commit_ms) * 1e3
    verify_us_layer = statistics.mean(verify_ms) * 1e3 / sb.L

    def spread(ms, per=1):
        """p10 / median / p90 of per-step event durations, in µs per launch."""
        q = statistics.quantiles([x * 1e3 / per for x in ms], n=10, method="inclusive") if len(ms) > 1 else [ms[0] * 1e3 / per] * 9
        return {"p10": round(q[0], 2), "p50": round(statistics.median(ms) * 1e3 / per, 2), "p90": round(q[8], 2)}
    peak, peak_kind = measured_peaks()
    achieved = cbytes / (commit_us * 1e-6) / 1e9
    v_achieved = vbytes / (verify_us_layer * 1e-6) / 1e9

    # roofline of both kernels of the step; "roofline" is the one that takes
    # the larger share of the measured step time
    step_us = commit_us + verify_us_layer * sb.L
    commit_rf = {
        "kernel": "gdn_commit_kernel (all-layer replay commit, 1 launch per step)",
        "bound": "hbm", "achieved": round(achieved, 1), "peak": peak, "unit": "GB/s",
        "frac": round(achieved / peak, 4), "peak_kind": f"{peak_kind} copy bandwidth",
        "frac_of_nominal": round(achieved / NOMINAL_HBM_GBS, 4),
        # the summary covers the default layer count; a commit launch's bytes scale with it
        "traffic": (profiled_traffic("commit", args.workload, COMMIT_SOURCES, args.state_dtype)
                    if args.layers is None else None),
        "algorithmic_bytes_per_launch": cbytes, "launch_us": round(commit_us, 2),
        "launch_us_spread": spread(commit_ms),
        "share_of_step": round(commit_us / step_us, 4),
    }
    verify_rf = {
        "kernel": f"gdn_verify_kernel (verify of one layer, {sb.L} launches per step)",
        "bound": "hbm", "achieved": round(v_achieved, 1), "peak": peak, "unit": "GB/s",
        "frac": round(v_achieved / peak, 4), "peak_kind": f"{peak_kind} copy bandwidth",
        "frac_of_nominal": round(v_achieved / NOMINAL_HBM_GBS, 4),
        "traffic": profiled_traffic("verify", args.workload, VERIFY_SOURCES, args.state_dtype),
        "algorithmic_bytes_per_launch": vbytes, "launch_us": round(verify_us_layer, 2),
        "launch_us_spread": spread(verify_ms, sb.L),
        "share_of_step": round(verify_us_layer * sb.L / step_us, 4),
    }
    for rf in (commit_rf, verify_rf):
        # the DRAM bytes ncu counted for the same launch, over the same time
        rf["achieved_dram_gbs"] = (round(rf["traffic"] / (rf["launch_us"] * 1e-6) / 1e9, 1)
                                   if rf["traffic"] else None)
        rf["note"] = ("achieved = algorithmic bytes / event time; frac can exceed 1 because the "
                      "peak is a plain copy (torch copy_, 1:1 read:write) and because writes "
                      "still dirty in L2 when the kernel ends drain after its end event "
                      "(achieved_dram_gbs: the DRAM bytes ncu counted for one launch over the "
                      "same time)")
    dominant, other = ((verify_rf, commit_rf) if verify_rf["share_of_step"] >= 0.5
                       else (commit_rf, verify_rf))

    # native per-draft-snapshot baseline of one layer (the comparison, not the step)
    out_n, snaps = step.native_buffers(sb)
    for _ in range(3):
        step.native_layer(sb, 0, out_n, snaps)
    torch.cuda.synchronize()
    reps = max(sb.L, 8)
    nbytes = roofline.native_bytes_per_layer(sb)
    # the reps cycle over the layers: the bytes they revisit are every layer's
    nscrub = L2Scrub(dev, nbytes * min(sb.L, reps))
    nev = [(torch.cuda.Event(enable_timing=True), torch.cuda.Event(enable_timing=True))
           for _ in range(reps)]
    for i in range(reps):
        nscrub()
        nev[i][0].record(stream)
        step.native_layer(sb, i % sb.L, out_n, snaps)
        nev[i][1].record(stream)
    torch.cuda.synchronize()
    native_us = sum(a.elapsed_time(b) for a, b in nev) * 1e3 / reps
    del out_n, snaps

    conv = run_conv_commit(sb, stream, peak, dev)

    e2e = None if args.no_e2e else run_e2e(args, sb, bufs, graph, stream, arena)

    result = {
        "metric": METRIC, "value": round(ms_per_step * 1e3, 3), "unit": UNIT,
        "n_gpus": world_size, "steps": K, "warmup": args.warmup,
        "ms_per_step": round(ms_per_step, 5), "higher_is_better": False,
        "scaling": "weak", "vs_baseline": None, "dtype": "f32",
        "data": "synthetic (seeded; see workloads.py)",
        "config": config_dict(args, sb, world_size),
        "roofline": dominant,
        "other_roofline": other,
        "native_snapshot": {
            "kernel": "gdn_verify_kernel<native>", "us_per_layer": round(native_us, 2),
            "algorithmic_bytes_per_layer": nbytes,
            "achieved_gbs": round(nbytes / (native_us * 1e-6) / 1e9, 1),
            "note": "comparison baseline, not part of the step", "l2": nscrub.describe(),
        },
        "conv_commit": conv,
        "gpu_launches": K * (sb.L + 1),
        "clocks": clk,
        "wall_s_timed": round(wall, 3),
    }
    if e2e:
        result["e2e"] = e2e
    if rank == 0 and world_size == 1 and not args.no_cpu_baseline:
        result["cpu_baseline"] = cpu_baseline(sb, args.cpu_seconds)
    if not args.no_configs and args.layers is None and args.seed is None:
        main_entry = {
            "workload": DESCR[args.workload], "layers": sb.L, "batch": sb.B, "window": sb.W,
            "state_dtype": args.state_dtype, "step_us": round(step_us, 2),
            "verify_us_per_layer": round(verify_us_layer, 2),
            "verify_bytes_per_layer": vbytes, "verify_gbs": round(v_achieved, 1),
            "verify_frac": round(v_achieved / peak, 4),
            "native_us_per_layer": round(native_us, 2), "native_bytes_per_layer": nbytes,
            "native_gbs": round(nbytes / (native_us * 1e-6) / 1e9, 1),
            "commit_us": round(commit_us, 2), "commit_bytes": cbytes,
            "commit_gbs": round(achieved, 1), "commit_frac": round(achieved / peak, 4),
            "l2": scrub.describe(), "steps": K, "source": "the line's own timed steps"}
        del sb, bufs, graph, arena
        torch.cuda.synchronize()
        torch.cuda.empty_cache()
        result["configs"] = run_configs(args, dev, rank, stream, peak,
                                        {(args.workload, args.state_dtype): main_entry})
    return result


# Every benchmark configuration, measured in the same run: (key, workload,
# state dtype, seed).  The long/ragged configuration runs its three seeds.
CONFIGS = [
    ("tiny", "tiny", "f32", None),
    ("layer", "layer", "f32", None),
    ("all_layer", "all_layer", "f32", None),
    ("long_ragged_seed30", "long_ragged", "f32", 30),
    ("long_ragged_seed31", "long_ragged", "f32", 31),
    ("long_ragged_seed32", "long_ragged", "f32", 32),
    ("align_fp32", "align", "f32", None),
    ("align_bf16", "align", "bf16", None),
    ("kda_all_layer", "kda_all_layer", "f32", None),
]


def measure_config(sb, dev, stream, peak, steps, warmup=3):
    """µs per verify (one layer), per native snapshot (one layer) and per
    all-layer commit on one workload, with their algorithmic bytes and HBM
    fractions.  The verify of all layers runs from a CUDA graph, the commit
    eagerly, as in the main step; a workload under three times the L2 gets
    the clean scrub before its verify and before its commit."""
    bufs = step.StepBuffers(sb)
    step.verify_all(sb, bufs)
    step.commit(sb, bufs)
    torch.cuda.synchronize()
    graph = torch.cuda.CUDAGraph()
    with torch.cuda.graph(graph):
        step.verify_all(sb, bufs)
    torch.cuda.synchronize()
    cbytes = roofline.commit_bytes(sb)
    vbytes = roofline.verify_bytes_per_layer(sb)
    scrub = L2Scrub(dev, cbytes + vbytes * sb.L)
    for _ in range(warmup):
        graph.replay()
        step.commit(sb, bufs)
    ev = [[torch.cuda.Event(enable_timing=True) for _ in range(4)] for _ in range(steps)]
    for i in range(steps):
        scrub()
        ev[i][0].record(stream)
        graph.replay()
        ev[i][1].record(stream)
        scrub()
        ev[i][2].record(stream)
        step.commit(sb, bufs)
        ev[i][3].record(stream)
    torch.cuda.synchronize()
    assert int(bufs.err.item()) == 0, "row errors in a benchmark workload"
    verify_us = statistics.mean(e[0].elapsed_time(e[1]) for e in ev) * 1e3 / sb.L
    commit_us = statistics.mean(e[2].elapsed_time(e[3]) for e in ev) * 1e3
    del graph, bufs
    out_n, snaps = step.native_buffers(sb)
    step.native_layer(sb, 0, out_n, snaps)
    torch.cuda.synchronize()
    reps = max(sb.L, 8)
    nbytes = roofline.native_bytes_per_layer(sb)
    nscrub = L2Scrub(dev, nbytes * min(sb.L, reps))
    nev = [(torch.cuda.Event(enable_timing=True), torch.cuda.Event(enable_timing=True))
           for _ in range(reps)]
    for i in range(reps):
        nscrub()
        nev[i][0].record(stream)
        step.native_layer(sb, i % sb.L, out_n, snaps)
        nev[i][1].record(stream)
    torch.cuda.synchronize()
    native_us = sum(a.elapsed_time(b) for a, b in nev) * 1e3 / reps
    del out_n, snaps
    gbs = lambda b, us: b / (us * 1e-6) / 1e9
    return {
        "layers": sb.L, "batch": sb.B, "window": sb.W,
        "step_us": round(verify_us * sb.L + commit_us, 2),
        "verify_us_per_layer": round(verify_us, 2), "verify_bytes_per_layer": vbytes,
        "verify_gbs": round(gbs(vbytes, verify_us), 1),
        "verify_frac": round(gbs(vbytes, verify_us) / peak, 4),
        "native_us_per_layer": round(native_us, 2), "native_bytes_per_layer": nbytes,
        "native_gbs": round(gbs(nbytes, native_us), 1),
        "commit_us": round(commit_us, 2), "commit_bytes": cbytes,
        "commit_gbs": round(gbs(cbytes, commit_us), 1),
        "commit_frac": round(gbs(cbytes, commit_us) / peak, 4),
        "l2": scrub.describe(), "steps": steps,
    }


def run_configs(args, dev, rank, stream, peak, done):
    """The `configs` block: every configuration in CONFIGS, one workload in
    memory at a time (the main workload's numbers are reused)."""
    out = {}
    steps = max(5, min(args.steps, 20))
    for key, name, sdt, seed in CONFIGS:
        if seed is None and (name, sdt) in done:
            out[key] = done[(name, sdt)]
            continue
        sd = torch.bfloat16 if sdt == "bf16" else torch.float32
        sb = make_workload(name, dev, rank, sd, seed=seed)
        entry = {"workload": DESCR[name] if seed is None else
                 re.sub(r"seed \d+", f"seed {seed}", DESCR[name]), "state_dtype": sdt}
        entry.update(measure_config(sb, dev, stream, peak, steps))
        del sb
        torch.cuda.synchronize()
        torch.cuda.empty_cache()
        if name == "layer":
            # the same per-layer shape as eight independent layers back to back
            # (one verify graph, one all-layer commit), as a model forward runs
            # them: each launch's inputs come from HBM, and the launch start-up
            # overlaps the previous launch instead of following an L2 flush
            sb = make_workload(name, dev, rank, sd, layers=8, seed=seed)
            m = measure_config(sb, dev, stream, peak, steps)
            entry["back_to_back"] = {
                "layers": 8, "verify_us_per_layer": m["verify_us_per_layer"],
                "verify_frac": m["verify_frac"], "commit_us": m["commit_us"],
                "commit_bytes": m["commit_bytes"], "commit_frac": m["commit_frac"], "l2": m["l2"]}
            del sb
            torch.cuda.synchronize()
            torch.cuda.empty_cache()
        out[key] = entry
    out["peak"] = {"hbm_gbs": peak, "kind": "measured copy bandwidth"}
    return out


def run_conv_commit(sb, stream, peak, dev, state_len=3):
    """Short-conv state commit of every layer (bf16 states, width-4
    convolution) with the step's plan: one launch, timed from a CUDA graph
    replay per iteration (each after an L2 scrub when its bytes are small).
    Reported beside the step, not inside it."""
    pools, inputs = workloads.conv_state(sb, state_len=state_len, dtype=torch.bfloat16)
    tab = api.ConvTable(pools, inputs)

    def call():
        api.gdn_conv_state_commit(table=tab, token_start=sb.token_start, window_len=sb.window_len,
                                  accepted_len=sb.accepted_len, slot_tables=sb.slot_table,
                                  max_window=sb.W, seq_pos=sb.seq_pos, block_size=sb.block_size)

    call()
    torch.cuda.synchronize()
    g = torch.cuda.CUDAGraph()
    with torch.cuda.graph(g):
        call()
    for _ in range(3):
        g.replay()
    reps = 50
    C = tab.C
    nbytes = roofline.conv_commit_bytes(sb, C, state_len, 2)
    cscrub = L2Scrub(dev, nbytes)
    cev = [(torch.cuda.Event(enable_timing=True), torch.cuda.Event(enable_timing=True))
           for _ in range(reps)]
    for i in range(reps):
        cscrub()
        cev[i][0].record(stream)
        g.replay()
        cev[i][1].record(stream)
    torch.cuda.synchronize()
    us = sum(a.elapsed_time(b) for a, b in cev) * 1e3 / reps
    del pools, inputs, tab, g
    return {"kernel": "gdn_conv_commit_kernel", "us": round(us, 2), "channels": C, "l2": cscrub.describe(),
            "state_len": state_len, "dtype": "bf16", "algorithmic_bytes": nbytes,
            "achieved_gbs": round(nbytes / (us * 1e-6) / 1e9, 1),
            "frac": round(nbytes / (us * 1e-6) / 1e9 / peak, 4)}


def run_e2e(args, sb, bufs, graph, stream, arena):
    """The same step through the public API with host buffers: every step
    copies all of its inputs (q/k/v, gates, row metadata of every layer)
    from pinned host memory in one copy, runs, and reads back every layer's
    output and the error word.  Measured twice: serially (copy in, compute,
    copy out, one after the other) and pipelined, as a serving loop runs it,
    with two input arenas and two output sets so that step i+1's inputs and
    step i-1's outputs cross the bus on their own streams while step i
    computes.  `value` is the pipelined figure; every step still moves its
    own bytes inside the timed region."""
    import dataclasses
    # second arena, outputs and verify graph (they bake in their addresses);
    # the state pools are shared, as they are in a serving engine
    sb2 = dataclasses.replace(sb, q=list(sb.q), k=list(sb.k), v=list(sb.v), a=list(sb.a),
                              b=list(sb.b),
                              fused_qkv=None if sb.fused_qkv is None else list(sb.fused_qkv))
    arena2 = step.pack_inputs(sb2)
    bufs2 = step.StepBuffers(sb2)
    step.verify_all(sb2, bufs2)
    torch.cuda.synchronize()
    graph2 = torch.cuda.CUDAGraph()
    with torch.cuda.graph(graph2):
        step.verify_all(sb2, bufs2)
    torch.cuda.synchronize()
    sets = [(sb, bufs, graph, arena), (sb2, bufs2, graph2, arena2)]
    host_in = arena.cpu().pin_memory()
    host_out = [torch.empty(bufs.out_all.shape, dtype=torch.float32, pin_memory=True) for _ in range(2)]
    host_err = [torch.empty(1, dtype=torch.int32, pin_memory=True) for _ in range(2)]
    bi = host_in.numel()
    bo = host_out[0].numel() * 4 + 4
    E = max(2, args.e2e_steps)

    def serial(n):
        for _ in range(n):
            arena.copy_(host_in, non_blocking=True)
            graph.replay()
            step.commit(sb, bufs)
            host_out[0].copy_(bufs.out_all, non_blocking=True)
            host_err[0].copy_(bufs.err, non_blocking=True)

    h2d, d2h = torch.cuda.Stream(), torch.cuda.Stream()
    ev = lambda: torch.cuda.Event(enable_timing=False)

    def pipelined(n, t0=None, t1=None):
        ready, done, drained = [ev(), ev()], [ev(), ev()], [ev(), ev()]
        used = [False, False]
        if t0 is not None:
            t0.record(h2d)

        def copy_in(i):
            s_ = i % 2
            with torch.cuda.stream(h2d):
                if used[s_]:
                    h2d.wait_event(done[s_])        # the step that last read this arena is over
                sets[s_][3].copy_(host_in, non_blocking=True)
                ready[s_].record(h2d)

        copy_in(0)
        for i in range(n):
            s_ = i % 2
            sbi, bfi, gi, _ = sets[s_]
            if i + 1 < n:
                copy_in(i + 1)
            stream.wait_event(ready[s_])
            if used[s_]:
                stream.wait_event(drained[s_])      # its outputs of two steps ago are read back
            gi.replay()
            step.commit(sbi, bfi)
            done[s_].record(stream)
            used[s_] = True
            with torch.cuda.stream(d2h):
                d2h.wait_event(done[s_])
                host_out[s_].copy_(bfi.out_all, non_blocking=True)
                host_err[s_].copy_(bfi.err, non_blocking=True)
                drained[s_].record(d2h)
        if t1 is not None:
            for e_ in (done[(n - 1) % 2], drained[0], drained[1]):
                d2h.wait_event(e_)
            t1.record(d2h)

    serial(3)
    pipelined(4)
    torch.cuda.synchronize()
    dist.barrier()
    a, b = torch.cuda.Event(enable_timing=True), torch.cuda.Event(enable_timing=True)
    a.record(stream)
    serial(E)
    b.record(stream)
    torch.cuda.synchronize()
    serial_ms = dist.max_over_ranks(a.elapsed_time(b), torch.cuda.current_device()) / E
    c, d = torch.cuda.Event(enable_timing=True), torch.cuda.Event(enable_timing=True)
    pipelined(E, c, d)
    torch.cuda.synchronize()
    pipe_ms = dist.max_over_ranks(c.elapsed_time(d), torch.cuda.current_device()) / E
    assert int(host_err[0].item()) == 0 and int(host_err[1].item()) == 0
    del sb2, bufs2, graph2, arena2
    return {"value": round(pipe_ms * 1e3, 3), "unit": UNIT, "h2d_bytes_per_step": bi,
            "d2h_bytes_per_step": bo, "steps": E, "serial_value": round(serial_ms * 1e3, 3),
            "path": "one pinned host -> device copy of every input of the step, verify graph + "
                    "commit call, one device -> host copy of every layer's output and the error "
                    "word; value: copies of neighbouring steps overlap the compute (two arenas, "
                    "copy streams); serial_value: copy, compute, copy in sequence"}


def run_grouped(args):
    """Grouped all-layer commit: 18 GDN layers in 3 KV-cache groups of 6, each
    group with its own state-index table, committed by one grouped launch or
    by one commit call per group.  Device time by CUDA events, host time of
    the calls by the wall clock (the calls enqueue and return)."""
    torch.cuda.set_device(0)
    dev = torch.device("cuda", 0)
    build.build()
    api.load()
    G, per = 3, 6
    sb = workloads.all_layer(device=dev, sentinel=False, L=G * per)
    gen = torch.Generator().manual_seed(11)
    tables = [sb.slot_table.cpu()]
    for _ in range(1, G):
        perm = torch.randperm(sb.num_slots, generator=gen)[:sb.B].view(-1, 1).to(torch.int32)
        perm[sb.window_len.cpu() == 0] = -1
        tables.append(perm)
    slot_tables = torch.stack(tables).to(dev).contiguous()
    layer_group = torch.tensor([l // per for l in range(sb.L)], dtype=torch.int32, device=dev)
    bufs = step.StepBuffers(sb)
    for l in range(sb.L):
        g = l // per
        api.gdn_spec_verify(q=sb.q[l], k=sb.k[l], v=sb.v[l], a=sb.a[l], b=sb.b[l],
                            A_log=sb.A_log[l], dt_bias=sb.dt_bias[l], token_start=sb.token_start,
                            window_len=sb.window_len, state_pool=sb.pools[l],
                            slot_table=slot_tables[g], out=bufs.out[l], rec_u=bufs.rec_u[l],
                            rec_k=bufs.rec_k[l], rec_g=bufs.rec_g[l], max_window=sb.W,
                            err=bufs.err)
    group_tabs = [api.LayerTable(sb.pools[g * per:(g + 1) * per], bufs.rec_u[g * per:(g + 1) * per],
                                 bufs.rec_k[g * per:(g + 1) * per], bufs.rec_g[g * per:(g + 1) * per])
                  for g in range(G)]

    def grouped():
        api.gdn_replay_commit_grouped(table=bufs.table, num_k_heads=sb.HK, layer_group=layer_group,
                                      window_len=sb.window_len, accepted_len=sb.accepted_len,
                                      slot_tables=slot_tables, err=bufs.err)

    def per_group():
        for g in range(G):
            api.gdn_replay_commit(table=group_tabs[g], num_k_heads=sb.HK, window_len=sb.window_len,
                                  accepted_len=sb.accepted_len, slot_table=slot_tables[g],
                                  err=bufs.err)

    stream = torch.cuda.current_stream()
    out = {"impl": "gb300", "measurement": "grouped all-layer commit",
           "config": {"workload": f"{G} KV-cache groups x {per} GDN layers, all_layer shapes "
                                  "(batch 64 with 8 padding rows, HK=16 HV=32 K=V=128, window 4)"}}
    cbytes = roofline.commit_bytes(sb)
    for name, fn in (("grouped_one_launch", grouped), ("one_call_per_group", per_group)):
        for _ in range(3):
            fn()
        torch.cuda.synchronize()
        K = max(20, args.steps // 10)
        a, b = torch.cuda.Event(enable_timing=True), torch.cuda.Event(enable_timing=True)
        host = 0.0
        a.record(stream)
        for _ in range(K):
            t0 = time.perf_counter()
            fn()
            host += time.perf_counter() - t0
        b.record(stream)
        torch.cuda.synchronize()
        dev_us = a.elapsed_time(b) * 1e3 / K
        out[name] = {"device_us": round(dev_us, 2), "host_us_per_step": round(host / K * 1e6, 2),
                     "launches_per_step": 1 if name.startswith("grouped") else G,
                     "achieved_gbs": round(cbytes / (dev_us * 1e-6) / 1e9, 1)}
    assert int(bufs.err.item()) == 0
    return out


# ---------------------------------------------------- CPU oracle timing
def _compact_layer(sb, l, rows):
    """Host copies of one layer restricted to `rows`, with the pool reduced
    to the slots those rows read and write (the oracle's input; not timed)."""
    import numpy as np
    table = sb.slot_table[rows].cpu()
    used = sorted({int(s) for s in table.flatten().tolist() if s >= 0})
    remap = {s: i for i, s in enumerate(used)}
    new_table = table.clone()
    for i in range(new_table.shape[0]):
        for j in range(new_table.shape[1]):
            s = int(new_table[i, j])
            new_table[i, j] = remap[s] if s >= 0 else -1
    win = sb.window_len[rows].cpu()
    start = sb.token_start[rows].cpu()
    # gather each row's token rows contiguously
    tok = [int(start[i]) + t for i in range(len(rows)) for t in range(int(win[i]))]
    new_start = torch.tensor(np.concatenate([[0], np.cumsum(win.numpy())[:-1]]), dtype=torch.int32)
    idx = torch.tensor(tok, dtype=torch.long, device=sb.device)
    f64 = lambda t: np.ascontiguousarray(t.to("cpu", torch.float64).numpy())
    pool = f64(sb.pools[l][torch.tensor(used, dtype=torch.long, device=sb.device)]) if used else \
        np.zeros((1, sb.HV, sb.V, sb.K))
    return dict(q=f64(sb.q[l][idx]), k=f64(sb.k[l][idx]), v=f64(sb.v[l][idx]),
                a=f64(sb.a[l][idx]), b=f64(sb.b[l][idx]), A_log=f64(sb.A_log[l]),
                dt_bias=f64(sb.dt_bias[l]), token_start=new_start.numpy(), window_len=win.numpy(),
                pool=pool, slot_table=new_table.numpy(),
                seq_pos=None if sb.seq_pos is None else sb.seq_pos[rows].cpu().numpy(),
                accepted_len=sb.accepted_len[rows].cpu().numpy(), block_size=sb.block_size,
                W=sb.W)


def _oracle_unit_of_work(oracle, d):
    """Oracle verify, then commit, of one compacted layer."""
    v = oracle.spec_verify(q=d["q"], k=d["k"], v=d["v"], a=d["a"], b=d["b"], A_log=d["A_log"],
                           dt_bias=d["dt_bias"], token_start=d["token_start"],
                           window_len=d["window_len"], pool=d["pool"],
                           slot_table=d["slot_table"], seq_pos=d["seq_pos"],
                           block_size=d["block_size"], max_window=d["W"])
    oracle.replay_commit(pools=d["pool"][None], rec_u=v["rec_u"][None], rec_k=v["rec_k"][None],
                         rec_g=v["rec_g"][None], window_len=d["window_len"],
                         accepted_len=d["accepted_len"], slot_table=d["slot_table"],
                         seq_pos=d["seq_pos"], block_size=d["block_size"], max_window=d["W"])


def _time_layers(oracle, sb, seconds):
    """Oracle verify + commit over whole layers (all rows) until `seconds` of
    oracle time are spent; returns (layers done, seconds).  The host copies
    each layer needs are made outside the timed calls."""
    rows = list(range(sb.B))
    layers_done, spent = 0, 0.0
    for l in range(sb.L):
        d = _compact_layer(sb, l, rows)
        t0 = time.perf_counter()
        _oracle_unit_of_work(oracle, d)
        spent += time.perf_counter() - t0
        layers_done += 1
        if spent >= seconds:
            break
    return layers_done, spent


def cpu_baseline(sb, seconds, seconds_one_core=6.0):
    """The fp64 oracle as it stands, on all host cores and on one, over whole
    layers of the same workload until each time budget is spent; scaled to a
    full step."""
    import oracle
    oracle.build()
    cores = oracle.num_threads()
    n_all, t_all = _time_layers(oracle, sb, seconds)
    oracle.set_num_threads(1)
    try:
        n_one, t_one = _time_layers(oracle, sb, seconds_one_core)
    finally:
        oracle.set_num_threads(cores)
    scaled = lambda n, t: round(t / n * sb.L * 1e6, 1)
    return {"value": scaled(n_all, t_all), "unit": UNIT, "cores": cores, "kind": "oracle",
            "sample": f"{n_all} of {sb.L} layers (all {sb.B} rows), verify + commit, "
                      f"{t_all:.1f} s of oracle time on {cores} threads, scaled to {sb.L} layers",
            "single_core": {"value": scaled(n_one, t_one), "unit": UNIT, "cores": 1,
                            "sample": f"{n_one} of {sb.L} layers (all {sb.B} rows), "
                                      f"{t_one:.1f} s of oracle time on 1 thread, scaled to "
                                      f"{sb.L} layers"}}


# ------------------------------------------------------ reference arm
REFERENCE_BUDGET_S = 150.0


def run_reference(args, rank, world_size):
    """The oracle on this workload, timed on the host cores.  Each step runs
    verify + commit of every layer over all rows when K + W such steps fit
    the time budget; otherwise each step runs a cycling subset of the layers
    (all rows), scaled to the full step.  Under torchrun only rank 0 works;
    the other ranks join the process group and leave."""
    if world_size > 1:
        dist.init("gloo")
    try:
        if rank != 0:
            dist.barrier()
            return None
        result = _reference_rank0(args, world_size)
        dist.barrier()
        return result
    finally:
        dist.finalize()


def host_cores():
    try:
        return len(os.sched_getaffinity(0))
    except AttributeError:
        return os.cpu_count() or 1


def _reference_rank0(args, world_size):
    import oracle
    oracle.build()
    # all of the host's cores (torchrun would otherwise leave one thread per rank)
    oracle.set_num_threads(host_cores())
    dev = torch.device("cuda", 0) if torch.cuda.is_available() else torch.device("cpu")
    sd = torch.bfloat16 if args.state_dtype == "bf16" else torch.float32
    sb = make_workload(args.workload, dev, 0, sd, args.layers, args.seed)
    rows = list(range(sb.B))
    layers = [_compact_layer(sb, l, rows) for l in range(sb.L)]   # host copies, once
    config = config_dict(args, sb, world_size)
    del sb

    def run_layers(ids):
        for l in ids:
            _oracle_unit_of_work(oracle, layers[l])

    n_steps = args.warmup + args.steps
    t0 = time.perf_counter()
    run_layers([0])
    per_layer = time.perf_counter() - t0
    L = len(layers)
    m = L if n_steps * per_layer * L <= REFERENCE_BUDGET_S else \
        max(1, min(L, int(REFERENCE_BUDGET_S / (n_steps * per_layer))))
    samples, nxt = [], 0
    for i in range(n_steps):
        ids = [(nxt + j) % L for j in range(m)]
        nxt = (nxt + m) % L
        t0 = time.perf_counter()
        run_layers(ids)
        dt = time.perf_counter() - t0
        if i >= args.warmup:
            samples.append(dt)
    us = statistics.mean(samples) * (L / m) * 1e6
    sample = (f"each step: verify + commit of all {L} layers x {len(rows)} rows (the whole step)"
              if m == L else
              f"each step: verify + commit of {m} of {L} layers (cycling) x all {len(rows)} rows, "
              f"scaled to {L} layers to keep {n_steps} steps within {REFERENCE_BUDGET_S:.0f} s")
    return {
        "impl": "reference", "metric": METRIC, "value": round(us, 1), "unit": UNIT,
        "n_gpus": world_size, "steps": args.steps, "warmup": args.warmup,
        "ms_per_step": round(us / 1e3, 3), "higher_is_better": False, "scaling": "weak",
        "vs_baseline": None, "dtype": "f64", "data": "synthetic (seeded; see workloads.py)",
        "config": config,
        "cpu_baseline": {"value": round(us, 1), "unit": UNIT, "cores": oracle.num_threads(),
                         "kind": "oracle", "sample": sample},
        "e2e": {"value": round(us, 1), "unit": UNIT, "h2d_bytes_per_step": 0,
                "d2h_bytes_per_step": 0},
    }


# ------------------------------------------------------------ launcher
def _free_port():
    import socket
    s_ = socket.socket()
    s_.bind(("127.0.0.1", 0))
    port = s_.getsockname()[1]
    s_.close()
    return port


def relaunch(argv, n):
    """Run this script under torchrun with n ranks on this node (one per
    GPU), passing the same arguments; returns torchrun's exit code."""
    cmd = [sys.executable, "-m", "torch.distributed.run", "--nnodes=1",
           f"--nproc-per-node={n}", "--master-addr", "127.0.0.1",
           "--master-port", str(_free_port()), os.path.abspath(__file__), *argv]
    return subprocess.call(cmd)


def main(argv=None):
    argv = sys.argv[1:] if argv is None else list(argv)
    args = parse(argv)
    if "WORLD_SIZE" not in os.environ and args.gpus > 1:
        return relaunch(argv, args.gpus)
    rank, local_rank, world_size = dist.world()
    if "WORLD_SIZE" in os.environ and world_size != args.gpus:
        print(f"bench.py: --gpus {args.gpus} but WORLD_SIZE={world_size}", file=sys.stderr)
        return 2
    if args.impl == "reference":
        res = run_reference(args, rank, world_size)
        if res is not None:
            print(json.dumps(res), flush=True)
        return 0
    if args.grouped_commit:
        print(json.dumps(run_grouped(args)), flush=True)
        return 0
    rank, local_rank, world_size = dist.init("nccl")
    try:
        result = run_gpu(args, rank, local_rank, world_size)
        if rank == 0:
            print(json.dumps(result), flush=True)
    finally:
        dist.finalize()
    return 0


if __name__ == "__main__":
    sys.exit(main())
