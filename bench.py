#!/usr/bin/env python3
"""Benchmark of the GB300 merge-path replacement merge (one JSON line).

Headline workload: the stable merge of two sorted uint64 key arrays of 2^26
elements each, every key carrying a uint32 payload (its source index). One
step is one lsm_merge_stable call (merge path partition + tile merge) over
inputs already resident in HBM. The metric is merged elements per second
(input elements / time); the line also reports the tile kernel's achieved HBM
bandwidth against the measured copy peak.

A line before the result carries, under "workloads", the other hot-path
pipelines, each timed as a whole path:
  int32 4096+4096 merge          (latency-bound)
  replacement 12,000,000 + 4,000,000 uint64 keys: replacement_merge (mark,
                                 rank512 build, compaction in one call)
  skewed replacement 2^24-1 + 65,536 keys (clustered)
  merge sort of 2^27 uint64 keys with payloads
  string replacement + FC encode, 4,000,000 + 4,000,000 keys:
                                 replacement_merge_str, fc_lengths_scan, fc_emit

Usage: python bench.py [--gpus N] [--steps K] [--warmup W] [--impl reference]
Under torchrun (N > 1) every rank merges its own independent problem of the
headline size (replicas; no data-path collective) and the value is the total
over ranks divided by the slowest rank's time.
"""
from __future__ import annotations

import argparse
import hashlib
import json
import os
import statistics
import subprocess
import sys
import threading
import time

import numpy as np

ROOT = os.path.dirname(os.path.abspath(__file__))
sys.path.insert(0, ROOT)

import synth  # noqa: E402

METRIC = "merged Gelem/s and achieved HBM GB/s (% of GB300 peak), 1 GPU, vs CPU oracle"
UNIT = "Gelem/s"
PROFILE_EVERY = 4  # headline steps whose tile kernel is timed by events
FALLBACK_HBM_GBS = 6800.0
L2_BYTES = 129 * 1024 * 1024


def parse_args():
    ap = argparse.ArgumentParser()
    ap.add_argument("--gpus", type=int, default=1)
    ap.add_argument("--steps", type=int, default=400)
    ap.add_argument("--warmup", type=int, default=5)
    ap.add_argument("--impl", default="ours", choices=["ours", "reference"])
    ap.add_argument("--no-extra", action="store_true", help="headline workload only")
    ap.add_argument("--no-strings", action="store_true", help="skip the string/FC workload")
    ap.add_argument("--merge-config", default="11,2,1",
                    help="merge tile configuration: items per thread, stages, output tiles")
    ap.add_argument("--sweep", action="store_true", help="also time every items-per-thread setting")
    ap.add_argument("--only", default="",
                    help="run only this extra workload (merge_i32_4096, replace_u64_12M_4M, "
                         "replace_skewed_2pow24_65536, merge_sort_u64_2pow27, strings_fc_4M_4M) "
                         "and print its result; "
                         "for profiler captures")
    ap.add_argument("--log2", type=int, default=26,
                    help="headline inputs hold 2^log2 keys each (26 = the full workload; smaller "
                         "values serve profiler captures)")
    return ap.parse_args()


# ---------------------------------------------------------------------------
# environment: ranks, peaks, clocks
# ---------------------------------------------------------------------------
def dist_env():
    world = int(os.environ.get("WORLD_SIZE", "1"))
    rank = int(os.environ.get("RANK", "0"))
    local = int(os.environ.get("LOCAL_RANK", "0"))
    return world, rank, local


def hbm_peak():
    path = os.path.join(ROOT, "MEASURED_PEAKS.json")
    try:
        with open(path) as f:
            return float(json.load(f)["hbm_gbs"]), "measured"
    except Exception:
        return FALLBACK_HBM_GBS, "fallback"


class ClockSampler:
    """nvidia-smi sampling of SM clocks and throttle reasons while running."""

    FIELDS = ("index,clocks.sm,clocks.max.sm,power.draw,clocks_event_reasons.active,"
              "clocks_event_reasons.hw_slowdown,clocks_event_reasons.hw_thermal_slowdown,"
              "clocks_event_reasons.sw_thermal_slowdown,clocks_event_reasons.sw_power_cap")

    def __init__(self, gpu_index):
        self.gpu = gpu_index
        self.proc = None
        self.lines = []

    def start(self):
        try:
            self.proc = subprocess.Popen(
                ["nvidia-smi", "-i", str(self.gpu), "--query-gpu=" + self.FIELDS,
                 "--format=csv,noheader,nounits", "-lms", "100"],
                stdout=subprocess.PIPE, stderr=subprocess.DEVNULL, text=True)
            self.t = threading.Thread(target=self._read, daemon=True)
            self.t.start()
        except Exception:
            self.proc = None
        return self

    def _read(self):
        for line in self.proc.stdout:
            self.lines.append((time.time(), line.strip()))

    def wait_first(self, timeout=3.0):
        t0 = time.time()
        while self.proc and not self.lines and time.time() - t0 < timeout:
            time.sleep(0.02)

    def stop(self):
        if self.proc:
            self.proc.terminate()
            try:
                self.proc.wait(timeout=5)
            except Exception:
                self.proc.kill()
            self.t.join(timeout=2)

    def summary(self, t_begin, t_end):
        rows = []
        for ts, line in self.lines:
            parts = [p.strip() for p in line.split(",")]
            if len(parts) < 9:
                continue
            rows.append((ts, parts))
        inside = [p for ts, p in rows if t_begin <= ts <= t_end] or \
                 [p for ts, p in rows if t_begin - 0.3 <= ts <= t_end + 0.3]
        if not inside:
            return {"sm_mhz": None, "sm_max_mhz": None, "reasons": ["no samples in timed region"],
                    "samples": 0}
        sm = [float(p[1]) for p in inside if p[1].replace(".", "").isdigit()]
        smax = [float(p[2]) for p in inside if p[2].replace(".", "").isdigit()]
        names = ["hw_slowdown", "hw_thermal_slowdown", "sw_thermal_slowdown", "sw_power_cap"]
        reasons = sorted({names[k] for p in inside for k in range(4) if p[5 + k].lower() == "active"})
        return {"sm_mhz": statistics.median(sm) if sm else None,
                "sm_max_mhz": max(smax) if smax else None, "reasons": reasons,
                "samples": len(inside)}


def kernel_source_digest():
    h = hashlib.sha256()
    for name in ("merge.cu", "common.cuh"):
        with open(os.path.join(ROOT, "lsm_replacement_merge_gb300", "csrc", name), "rb") as f:
            h.update(f.read())
    return h.hexdigest()[:16]


def host_info():
    """Core count and CPU model of the host running the bench."""
    model = None
    try:
        with open("/proc/cpuinfo") as f:
            txt = f.read()
        for key in ("model name", "Model Name", "CPU part"):
            for line in txt.splitlines():
                if line.split(":")[0].strip() == key:
                    model = line.split(":", 1)[1].strip()
                    break
            if model:
                break
    except OSError:
        pass
    # Arm hosts report an implementer and part number instead of a name
    arm_parts = {("0x41", "0xd4f"): "Arm Neoverse-V2", ("0x41", "0xd40"): "Arm Neoverse-V1",
                 ("0x41", "0xd0c"): "Arm Neoverse-N1", ("0x41", "0xd49"): "Arm Neoverse-N2"}
    try:
        impl = next((ln.split(":", 1)[1].strip() for ln in txt.splitlines()
                     if ln.split(":")[0].strip() == "CPU implementer"), None)
        if model and impl and (impl, model) in arm_parts:
            model = "%s (implementer %s, part %s)" % (arm_parts[(impl, model)], impl, model)
    except NameError:
        pass
    import platform
    return {"cpu_count": os.cpu_count(), "cpu_model": model or platform.processor() or None,
            "machine": platform.machine()}


def build_info():
    """How the library was built: nvcc flags, a digest of every kernel source
    and the git commit when the tree is a checkout."""
    from lsm_replacement_merge_gb300 import _build
    h = hashlib.sha256()
    for src in sorted(_build._deps()):
        with open(src, "rb") as f:
            h.update(f.read())
    sha = None
    try:
        sha = subprocess.run(["git", "-C", ROOT, "rev-parse", "HEAD"], capture_output=True,
                             text=True, timeout=10).stdout.strip() or None
    except (OSError, subprocess.SubprocessError):
        pass
    flags = " ".join(_build.ARCH + _build.NVCC_FLAGS).replace(ROOT + os.sep, "")
    return {"nvcc_flags": flags, "source_digest": h.hexdigest()[:16], "git_sha": sha}


def ncu_traffic(kernel_key):
    """DRAM bytes per launch from the committed ncu summary, or None when the
    kernel source changed since the counters were taken."""
    path = os.path.join(ROOT, "profiles", "ncu_traffic.json")
    try:
        with open(path) as f:
            data = json.load(f)
        ent = data[kernel_key]
        if ent.get("source_digest") != kernel_source_digest():
            return None
        return float(ent["dram_bytes_per_launch"])
    except Exception:
        return None


def slowest_rank_ms(step_ms, dist=None, device=None):
    """Max of a per-rank step time over all ranks (the job is as fast as its
    slowest rank). With no process group, the value itself."""
    if dist is None:
        return float(step_ms)
    import torch
    t = torch.tensor([float(step_ms)], dtype=torch.float64, device=device)
    dist.all_reduce(t, op=dist.ReduceOp.MAX)
    return float(t.item())


def job_throughput(world, elems_per_rank, step_ms):
    """Whole-job Gelem/s: every rank merges its own problem of elems_per_rank
    elements per step (replicas, weak scaling)."""
    return world * elems_per_rank / (step_ms * 1e-3) / 1e9


# ---------------------------------------------------------------------------
# the reference arm: the CPU oracle as it stands, on bounded samples
# ---------------------------------------------------------------------------
def run_reference(args):
    world, rank, _ = dist_env()
    if rank != 0:
        return
    import oracle
    mi = synth.merge_u64()
    m, n = len(mi.A), len(mi.B)
    # calibrate, then size each step so that warmup + steps stay near 90 s
    x = 1 << 20
    t0 = time.perf_counter()
    oracle.merge(mi.A[:x], mi.B[:x], mi.Apay[:x], mi.Bpay[:x])
    rate = 2 * x / max(time.perf_counter() - t0, 1e-6)
    budget = 90.0 / max(args.steps + args.warmup, 1)
    half = int(min(m, max(1 << 16, rate * budget / 2)))
    times = []
    for s in range(args.warmup + args.steps):
        off = (s * 7919 * 64) % max(m - half + 1, 1)
        a, b = mi.A[off:off + half], mi.B[off:off + half]
        pa, pb = mi.Apay[off:off + half], mi.Bpay[off:off + half]
        t0 = time.perf_counter()
        oracle.merge(a, b, pa, pb)
        dt = time.perf_counter() - t0
        if s >= args.warmup:
            times.append(dt)
    total = sum(times)
    elems = 2 * half * len(times)
    value = elems / total / 1e9
    sample = ("two-pointer oracle merge of %d + %d contiguous elements per step (slices of the "
              "2^26 + 2^26 uint64 + uint32-payload workload)" % (half, half))
    line = {
        "impl": "reference", "metric": METRIC, "value": value, "unit": UNIT,
        "n_gpus": args.gpus, "steps": args.steps, "warmup": args.warmup,
        "ms_per_step": 1e3 * total / len(times), "higher_is_better": True,
        "scaling": "weak", "vs_baseline": None, "dtype": "u64+u32", "data": "synthetic",
        "config": headline_config(m, n),
        "cpu_baseline": {"value": value, "unit": UNIT, "cores": 1, "kind": "oracle",
                         "sample": sample, "host_cores": os.cpu_count(),
                         "cpu_model": host_info()["cpu_model"]},
        "e2e": {"value": value, "unit": UNIT, "h2d_bytes_per_step": 0, "d2h_bytes_per_step": 0},
    }
    print(json.dumps(line), flush=True)


def headline_config(m, n):
    """The workload alone (the same for both arms); the kernel's tile shape
    goes in the line's `kernel_config`."""
    return {"workload": "stable merge, sorted uint64 keys with uint32 payload, m = n = 2^%d"
                        % (m.bit_length() - 1),
            "m": m, "n": n, "key": "u64", "payload": "u32",
            "l2": "inputs and outputs (3 GiB) exceed the 129 MB L2; no flush needed",
            "parallelism": "replicas"}


# ---------------------------------------------------------------------------
# our arm
# ---------------------------------------------------------------------------
def main():
    args = parse_args()
    if args.impl == "reference":
        run_reference(args)
        return
    world, rank, local = dist_env()
    import torch
    torch.cuda.set_device(local)
    dev = torch.device("cuda", local)
    pg = None
    if world > 1:
        import torch.distributed as dist
        dist.init_process_group("nccl", device_id=dev)
        pg = dist
    import lsm_replacement_merge_gb300 as lsm
    lsm.lib()
    if args.only:
        peak, _ = hbm_peak()
        print(json.dumps({"only": args.only,
                          "workloads": extra_workloads(lsm, torch, dev, peak, args, only=args.only)}))
        return
    mcfg = tuple(int(x) for x in args.merge_config.split(","))
    lsm.tune_merge(lsm.LSM_KEY_U64, *mcfg)
    items = mcfg[0]
    peak, peak_kind = hbm_peak()

    # ---------------- headline: 2^26 + 2^26 uint64 merge with payload ----------------
    mi = synth.merge_u64(seed=2 + rank, m=1 << args.log2, n=1 << args.log2)
    m, n = len(mi.A), len(mi.B)
    A = torch.from_numpy(mi.A).to(dev)
    B = torch.from_numpy(mi.B).to(dev)
    Ap = torch.from_numpy(mi.Apay).to(dev)
    Bp = torch.from_numpy(mi.Bpay).to(dev)
    out_k = torch.empty(m + n, dtype=torch.uint64, device=dev)
    out_p = torch.empty(m + n, dtype=torch.uint32, device=dev)
    ws = lsm.workspace(lsm.LSM_OP_MERGE_STABLE, m, n, dev)
    stream = torch.cuda.current_stream()

    def step():
        lsm.merge_stable(A, B, Ap, Bp, out_keys=out_k, out_pay=out_p, ws=ws)

    for _ in range(max(args.warmup, 3)):
        step()
    torch.cuda.synchronize()
    sampler = ClockSampler(local).start()
    # keep the GPU busy until the sampler has produced its first sample
    t_end_warm = time.time() + 3.0
    while not sampler.lines and time.time() < t_end_warm:
        step()
        torch.cuda.synchronize()
    K = args.steps
    k_start = [torch.cuda.Event(enable_timing=True) for _ in range(K)]
    k_stop = [torch.cuda.Event(enable_timing=True) for _ in range(K)]
    ev0 = torch.cuda.Event(enable_timing=True)
    ev1 = torch.cuda.Event(enable_timing=True)
    for e in k_start + k_stop:
        e.record(stream)  # create the CUDA events before the timed region
    if pg:
        pg.barrier()
    torch.cuda.synchronize()
    t_begin = time.time()
    # The tile kernel of every PROFILE_EVERY-th step is bracketed by events
    # (its duration is the roofline's); the other steps run with nothing
    # between their launches, so each kernel may launch while the one before
    # it finishes (programmatic dependent launch).
    profiled = list(range(0, K, PROFILE_EVERY))
    ev0.record(stream)
    for s in range(K):
        if s % PROFILE_EVERY == 0:
            lsm.set_profile_events(k_start[s], k_stop[s])
        step()
    ev1.record(stream)
    torch.cuda.synchronize()
    t_end = time.time()
    if pg:
        pg.barrier()
    sampler.stop()
    clocks = sampler.summary(t_begin, t_end)
    step_ms = ev0.elapsed_time(ev1) / K
    kern_ms = statistics.mean(k_start[s].elapsed_time(k_stop[s]) for s in profiled)
    step_ms = slowest_rank_ms(step_ms, pg, dev)
    value = job_throughput(world, m + n, step_ms)
    alg_bytes = (m + n) * (8 + 4) * 2
    achieved = alg_bytes / (kern_ms * 1e-3) / 1e9
    traffic = ncu_traffic("merge_tile_kernel<u64,payload,%d,%d,%d>" % mcfg)

    # the partition step alone (the same co-ranks the merge computes first)
    D = 256 * mcfg[0]
    part_out = torch.empty(2 * ((m + n + D - 1) // D + 1), dtype=torch.int64, device=dev)
    p0 = [torch.cuda.Event(enable_timing=True) for _ in range(20)]
    p1 = [torch.cuda.Event(enable_timing=True) for _ in range(20)]
    for q in range(20):
        p0[q].record(stream)
        lsm.merge_path_partition(A, B, D, out_ij=part_out)
        p1[q].record(stream)
    torch.cuda.synchronize()
    partition_ms = statistics.mean(p0[q].elapsed_time(p1[q]) for q in range(5, 20))
    del part_out

    # sanity: the timed output is the merge (spot-check against a numpy merge of samples)
    stride = max((m + n) // 4096, 1)
    got = out_k.view(torch.int64)[::stride].cpu().numpy().view(np.uint64)
    ref = np.sort(np.concatenate([mi.A, mi.B]))[::stride]
    assert np.array_equal(got, ref), "timed merge output differs from the sorted inputs"

    # ---------------- e2e: pinned host buffers through the public API -------------------
    e2e = None
    if rank == 0 or world > 1:
        hA = torch.from_numpy(mi.A).pin_memory()
        hB = torch.from_numpy(mi.B).pin_memory()
        hAp = torch.from_numpy(mi.Apay).pin_memory()
        hBp = torch.from_numpy(mi.Bpay).pin_memory()
        hK = torch.empty(m + n, dtype=torch.uint64).pin_memory()
        hP = torch.empty(m + n, dtype=torch.uint32).pin_memory()
        # Two device buffer sets and three streams: the H2D copies of step s + 1
        # run while step s merges and while the D2H copies of step s - 1 run.
        # Every step copies its own inputs in and its result out; a buffer set
        # is reused only after the step that last used it has been copied out.
        sets = [dict(A=torch.empty_like(A), B=torch.empty_like(B), Ap=torch.empty_like(Ap),
                     Bp=torch.empty_like(Bp), K=torch.empty_like(out_k), P=torch.empty_like(out_p),
                     ws=lsm.workspace(lsm.LSM_OP_MERGE_STABLE, m, n, dev))
                for _ in range(2)]
        s_in, s_mg, s_out = torch.cuda.Stream(), torch.cuda.Stream(), torch.cuda.Stream()
        ev_in = [torch.cuda.Event() for _ in range(2)]
        ev_mg = [torch.cuda.Event() for _ in range(2)]
        ev_out = [torch.cuda.Event() for _ in range(2)]
        used = [False, False]

        def e2e_step(q):
            b = q % 2
            d = sets[b]
            with torch.cuda.stream(s_in):
                if used[b]:
                    s_in.wait_event(ev_mg[b])  # the merge that read these inputs is done
                d["A"].copy_(hA, non_blocking=True)
                d["B"].copy_(hB, non_blocking=True)
                d["Ap"].copy_(hAp, non_blocking=True)
                d["Bp"].copy_(hBp, non_blocking=True)
                ev_in[b].record(s_in)
            with torch.cuda.stream(s_mg):
                s_mg.wait_event(ev_in[b])
                if used[b]:
                    s_mg.wait_event(ev_out[b])  # the result held here was copied out
                lsm.merge_stable(d["A"], d["B"], d["Ap"], d["Bp"], out_keys=d["K"], out_pay=d["P"],
                                 ws=d["ws"], stream=s_mg)
                ev_mg[b].record(s_mg)
            with torch.cuda.stream(s_out):
                s_out.wait_event(ev_mg[b])
                hK.copy_(d["K"], non_blocking=True)
                hP.copy_(d["P"], non_blocking=True)
                ev_out[b].record(s_out)
            used[b] = True

        for q in range(2):
            e2e_step(q)
        torch.cuda.synchronize()
        E = max(4, min(K, 12))
        e0 = torch.cuda.Event(enable_timing=True)
        e1 = torch.cuda.Event(enable_timing=True)
        e0.record(s_in)
        s_in.wait_event(ev_out[0])
        s_in.wait_event(ev_out[1])
        for q in range(E):
            e2e_step(q)
        s_out.record_event(e1)
        torch.cuda.synchronize()
        e2e_ms = e0.elapsed_time(e1) / E
        assert np.array_equal(hK.view(torch.int64).numpy().view(np.uint64)[::stride], ref)
        e2e = {"value": world * (m + n) / (e2e_ms * 1e-3) / 1e9, "unit": UNIT,
               "h2d_bytes_per_step": (m + n) * 12, "d2h_bytes_per_step": (m + n) * 12,
               "ms_per_step": e2e_ms, "steps": E,
               "pipeline": "H2D of step s+1, merge of step s and D2H of step s-1 overlap "
                           "(three streams, two device buffer sets)"}
        del hA, hB, hAp, hBp, hK, hP, sets

    # ---------------- CPU baseline: the oracle on the host cores (rank 0) ---------------
    cpu = None
    if rank == 0:
        import oracle
        reps, t_cpu = 0, 0.0
        while reps < 1 or (t_cpu < 3.0 and reps < 10):
            t0 = time.perf_counter()
            oracle.merge(mi.A, mi.B, mi.Apay, mi.Bpay)
            t_cpu += time.perf_counter() - t0
            reps += 1
        hi = host_info()
        cpu = {"value": reps * (m + n) / t_cpu / 1e9, "unit": UNIT, "cores": 1, "kind": "oracle",
               "sample": "the whole 2^26 + 2^26 merge with payload, %d run(s)" % reps,
               "host_cores": hi["cpu_count"], "cpu_model": hi["cpu_model"]}

    sweep = None
    if args.sweep and rank == 0:
        sweep = {}
        for cfg_e in lsm.MERGE_CONFIGS:
            lsm.tune_merge(lsm.LSM_KEY_U64, *cfg_e)
            for _ in range(3):
                step()
            s0 = [torch.cuda.Event(enable_timing=True) for _ in range(50)]
            s1 = [torch.cuda.Event(enable_timing=True) for _ in range(50)]
            for ev in s0 + s1:
                ev.record(stream)
            for q in range(50):
                lsm.set_profile_events(s0[q], s1[q])
                step()
            torch.cuda.synchronize()
            kms = statistics.mean(s0[q].elapsed_time(s1[q]) for q in range(50))
            sweep["%d,%d,%d" % cfg_e] = {"kernel_ms": kms, "gbs": alg_bytes / (kms * 1e-3) / 1e9}
        lsm.tune_merge(lsm.LSM_KEY_U64, *mcfg)

    ws_bytes = ws.numel()
    del A, B, Ap, Bp, out_k, out_p, ws
    torch.cuda.empty_cache()

    workloads = {}
    if not args.no_extra and rank == 0:
        workloads = extra_workloads(lsm, torch, dev, peak, args)

    launches = 2 * K  # partition + tile kernel per step
    rep_roof = None
    summary = {}
    for name, w in workloads.items():
        if isinstance(w, dict) and "ms_per_step" in w:
            summary[name] = {k: w[k] for k in ("ms_per_step", "gelem_s", "gbs", "frac",
                                               "frac_of_8TBs_nominal") if k in w}
    rw = workloads.get("replace_u64_12M_4M")
    if rw:
        rep_roof = {"workload": "replacement merge, |A| = 12,000,000 + |B| = 4,000,000 uint64 "
                                "keys, 25 % of B in A (refs-only outputs)",
                    "call": rw.get("call"), "bound": "hbm", "ms_per_step": rw["ms_per_step"],
                    "algorithmic_bytes": rw["algorithmic_bytes"], "achieved": rw["gbs"],
                    "peak": peak, "unit": "GB/s", "frac": rw["frac"], "peak_source": peak_kind,
                    "frac_of_8TBs_nominal": rw["frac_of_8TBs_nominal"],
                    "target_frac_of_8TBs_nominal": 0.60,
                    "kernel_ms_in_separate_calls": rw["separate_calls"]["kernel_ms"],
                    "workspace_bytes": rw.get("workspace_bytes"), "traffic": None,
                    "l2": rw.get("l2")}
    if rank == 0 and workloads:
        # the full per-workload record on its own line, before the result line
        print(json.dumps({"workloads": workloads}), flush=True)
    line = {
        "metric": METRIC, "value": value, "unit": UNIT, "n_gpus": world, "steps": K,
        "warmup": args.warmup, "ms_per_step": step_ms, "higher_is_better": True,
        "scaling": "weak", "vs_baseline": None, "dtype": "u64+u32", "data": "synthetic",
        "config": headline_config(m, n),
        "kernel_config": {"items_per_thread": mcfg[0], "stages": mcfg[1], "out_tiles": mcfg[2],
                          "tile": 256 * mcfg[0]},
        "roofline": {"bound": "hbm", "kernel": "merge_tile_kernel", "achieved": achieved,
                     "peak": peak, "unit": "GB/s", "frac": achieved / peak,
                     "peak_source": peak_kind, "traffic": traffic,
                     "algorithmic_bytes_per_launch": alg_bytes, "kernel_ms": kern_ms,
                     "kernel_launches_timed": len(profiled),
                     "partition_ms": partition_ms,
                     "frac_of_8TBs_nominal": achieved / 8000.0},
        "roofline_replacement": rep_roof,
        "cpu_baseline": cpu,
        "e2e": e2e,
        "gpu_launches": launches,
        "clocks": clocks,
        "workloads_summary": summary,
        "workspace_bytes": {"merge_stable": ws_bytes},
        "host": host_info(),
        "build": build_info(),
    }
    if sweep:
        line["items_sweep"] = sweep
    if rank == 0:
        print(json.dumps(line), flush=True)
    if pg:
        pg.barrier()
        pg.destroy_process_group()


# ---------------------------------------------------------------------------
# the other pipelines
# ---------------------------------------------------------------------------
class Flusher:
    """Writes a buffer larger than L2 between timed iterations."""

    def __init__(self, torch, dev):
        self.buf = torch.empty(2 * L2_BYTES // 4, dtype=torch.int32, device=dev)

    def __call__(self):
        self.buf.fill_(1)


def time_pipeline(torch, stages, steps, flush, warmup=3):
    """stages: list of (name, fn). Returns (mean ms per step, {name: mean kernel ms})."""
    import lsm_replacement_merge_gb300 as lsm
    for _ in range(warmup):
        for _, fn in stages:
            fn()
    torch.cuda.synchronize()
    stream = torch.cuda.current_stream()
    tot, per = [], {name: [] for name, _ in stages}
    # Whole steps first, with nothing between the launches (an event recorded
    # between two kernels would keep the second from launching early), then
    # the same steps again with each stage's main kernel bracketed by events.
    for _ in range(steps):
        flush()
        e0 = torch.cuda.Event(enable_timing=True)
        e1 = torch.cuda.Event(enable_timing=True)
        e0.record(stream)
        for _, fn in stages:
            fn()
        e1.record(stream)
        torch.cuda.synchronize()
        tot.append(e0.elapsed_time(e1))
    for _ in range(steps):
        flush()
        ks = [(torch.cuda.Event(enable_timing=True), torch.cuda.Event(enable_timing=True))
              for _ in stages]
        for a, b in ks:
            a.record(stream)
            b.record(stream)
        for (name, fn), (a, b) in zip(stages, ks):
            lsm.set_profile_events(a, b)
            fn()
        torch.cuda.synchronize()
        for (name, _), (a, b) in zip(stages, ks):
            per[name].append(a.elapsed_time(b))
    return statistics.mean(tot), {k: statistics.mean(v) for k, v in per.items()}


def extra_workloads(lsm, torch, dev, peak, args, only=""):
    out = {}
    flush = Flusher(torch, dev)
    steps = max(5, min(args.steps, 30))

    def wanted(name):
        return not only or only == name

    # int32 4096 + 4096 with payload
    if wanted("merge_i32_4096"):
        extra_merge_i32(lsm, torch, dev, steps, out)
    for name, gen in (("replace_u64_12M_4M", synth.replace_u64),
                      ("replace_skewed_2pow24_65536", synth.replace_skewed)):
        if wanted(name):
            extra_replace(lsm, torch, dev, peak, steps, flush, name, gen, out, args.sweep)
    if wanted("merge_sort_u64_2pow27"):
        extra_merge_sort(lsm, torch, dev, peak, steps, flush, out)
    if args.no_strings or not wanted("strings_fc_4M_4M"):
        return out
    extra_strings(lsm, torch, dev, peak, steps, flush, out)
    return out


def extra_merge_sort(lsm, torch, dev, peak, steps, flush, out):
    """Bottom-up merge sort of 2^27 uniform uint64 keys with uint32 payloads:
    the block sort to runs of 2816, then one partition + tile launch per pass."""
    si = synth.sort_u64()
    N = len(si.keys)
    keys, pay = torch.from_numpy(si.keys).to(dev), torch.from_numpy(si.pay).to(dev)
    ok = torch.empty_like(keys)
    op = torch.empty_like(pay)
    ws = lsm.workspace(lsm.LSM_OP_MERGE_SORT, N, 0, dev, lsm.LSM_KEY_U64)
    ms, per = time_pipeline(torch, [("merge_sort", lambda: lsm.merge_sort(
        keys, pay, out_keys=ok, out_pay=op, ws=ws))], steps, flush)
    tile = 256 * 11
    passes = 0
    w = tile
    while w < N:
        passes += 1
        w *= 2
    pass_bytes = 2 * 12 * N  # one pass reads and writes every key and payload
    last = per["merge_sort"]
    out["merge_sort_u64_2pow27"] = {
        "N": N, "ms_per_step": ms, "gelem_s": N / (ms * 1e-3) / 1e9,
        "passes": {"block_sort": 1, "global": passes},
        "algorithmic_bytes": (1 + passes) * pass_bytes,
        "gbs": (1 + passes) * pass_bytes / (ms * 1e-3) / 1e9,
        "frac": (1 + passes) * pass_bytes / (ms * 1e-3) / 1e9 / peak,
        "last_pass_tile_kernel_ms": last,
        "last_pass_tile_kernel_gbs": pass_bytes / (last * 1e-3) / 1e9,
        "last_pass_tile_kernel_frac": pass_bytes / (last * 1e-3) / 1e9 / peak,
        "gpu_launches_per_step": 1 + 2 * passes,
        "workspace_bytes": {"merge_sort": ws.numel()},
        "l2": "flushed (256 MiB write) before every step; inputs 1.5 GiB"}
    del keys, pay, ok, op, ws
    torch.cuda.empty_cache()


def extra_merge_i32(lsm, torch, dev, steps, out):
    mi = synth.merge_i32()
    A, B = torch.from_numpy(mi.A).to(dev), torch.from_numpy(mi.B).to(dev)
    Ap, Bp = torch.from_numpy(mi.Apay).to(dev), torch.from_numpy(mi.Bpay).to(dev)
    ok = torch.empty(8192, dtype=torch.int32, device=dev)
    op = torch.empty(8192, dtype=torch.uint32, device=dev)
    ws = lsm.workspace(lsm.LSM_OP_MERGE_STABLE, 4096, 4096, dev, lsm.LSM_KEY_I32)
    ms, per = time_pipeline(torch, [("merge_stable", lambda: lsm.merge_stable(
        A, B, Ap, Bp, out_keys=ok, out_pay=op, ws=ws))], max(steps, 20), lambda: None)
    out["merge_i32_4096"] = {"ms_per_step": ms, "gelem_s": 8192 / (ms * 1e-3) / 1e9,
                             "kernel_ms": per, "note": "latency-bound (two launches)"}


def extra_replace(lsm, torch, dev, peak, steps, flush, name, gen, out, sweep=False):
    ri = gen()
    m, n = len(ri.A), len(ri.B)
    A, B = torch.from_numpy(ri.A).to(dev), torch.from_numpy(ri.B).to(dev)
    C = torch.empty((m + 31) // 32, dtype=torch.uint32, device=dev)
    lb = torch.empty(n, dtype=torch.uint32, device=dev)
    dir_ = torch.empty(3 * (m // 512 + 1), dtype=torch.uint32, device=dev)
    tot = torch.empty(1, dtype=torch.int64, device=dev)
    refs = torch.empty(m + n, dtype=torch.uint32, device=dev)
    oa = torch.empty(m, dtype=torch.uint32, device=dev)
    ob = torch.empty(n, dtype=torch.uint32, device=dev)
    cnt = torch.empty(1, dtype=torch.int64, device=dev)
    w1 = lsm.workspace(lsm.LSM_OP_COLLISION_MARK, m, n, dev)
    w2 = lsm.workspace(lsm.LSM_OP_RANK_BUILD, m, 0, dev)
    w3 = lsm.workspace(lsm.LSM_OP_REPLACEMENT_COMPACT, m, n, dev)
    w6 = lsm.workspace(lsm.LSM_OP_REPLACEMENT_MERGE, m, n, dev)
    stages = [("collision_mark", lambda: lsm.collision_mark(A, B, C, lb, w1)),
              ("rank_build", lambda: lsm.rank_build(C, m, dir_, tot, w2)),
              ("replacement_merge_compact", lambda: lsm.replacement_merge_compact(
                  m, n, C, dir_, lb, refs, oa, ob, cnt, w3))]
    # The step: the whole path in one call (partition + mark, rank512 build,
    # compaction on the mark's diagonals): C, dir, R(m), refs, ordinals and
    # the count; the lower bounds are scratch on this path and not written.
    whole = [("replacement_merge", lambda: lsm.replacement_merge(
        A, B, C, None, dir_, tot, refs, oa, ob, cnt, w6, want_lb=False))]
    ms, per_whole = time_pipeline(torch, whole, steps, flush)
    N = int(cnt.item())
    # the same call also writing lb_B (every output of the three calls)
    whole_lb = [("replacement_merge", lambda: lsm.replacement_merge(
        A, B, C, lb, dir_, tot, refs, oa, ob, cnt, w6))]
    ms_lb, _ = time_pipeline(torch, whole_lb, steps, flush)
    # the same call in its other form: the mark and the compaction of each
    # tile in one persistent kernel (R from the mark warps' published counts)
    lsm.tune_replacement_merge(1)
    try:
        ms_one, _ = time_pipeline(torch, whole, steps, flush)
    finally:
        lsm.tune_replacement_merge(lsm.DEFAULT_REPLACEMENT_MERGE_MODE)
    # the same work as three separate calls: per-kernel times (each call's
    # main pipeline bracketed by events) and the step with one more partition
    ms_sep, per = time_pipeline(torch, stages, steps, flush)
    alg = (8 * (m + n)                      # read keys
           + 4 * ((m + 31) // 32)           # write C
           + 12 * (m // 512 + 1)            # write dir
           + 4 * N + 4 * (m + n))           # write refs, ord_A, ord_B
    out[name] = {"m": m, "n": n, "survivors": N, "ms_per_step": ms,
                 "gelem_s": (m + n) / (ms * 1e-3) / 1e9,
                 "algorithmic_bytes": alg, "gbs": alg / (ms * 1e-3) / 1e9,
                 "frac": alg / (ms * 1e-3) / 1e9 / peak,
                 "frac_of_8TBs_nominal": alg / (ms * 1e-3) / 1e9 / 8000.0,
                 "call": "lsm_replacement_merge", "gpu_launches_per_step": 4,
                 "mark_pipeline_ms": per_whole["replacement_merge"],
                 "lb_B": "scratch, not written",
                 "with_lb_B_written": {"ms_per_step": ms_lb},
                 "form": "two tile pipelines (mark, rank512 build, compaction)",
                 "one_kernel": {"ms_per_step": ms_one, "gpu_launches_per_step": 3},
                 "workspace_bytes": {"replacement_merge": w6.numel()},
                 "separate_calls": {"ms_per_step": ms_sep, "kernel_ms": per,
                                    # mark: partition + pipeline; rank build;
                                    # compaction from lb_B: its partition, the
                                    # merge bitmap and the pipeline
                                    "gpu_launches_per_step": 6,
                                    "workspace_bytes": {"collision_mark": w1.numel(),
                                                        "rank_build": w2.numel(),
                                                        "replacement_merge_compact": w3.numel()}},
                 "l2": "flushed (256 MiB write) before every step"}
    # The materialized row: the same step plus the survivors' keys, values
    # and tombstone bits gathered in merged order.
    vA, vB = torch.from_numpy(ri.valA).to(dev), torch.from_numpy(ri.valB).to(dev)
    tB = torch.from_numpy(ri.tombB).to(dev)
    ok = torch.empty(m + n, dtype=A.dtype, device=dev)
    ov = torch.empty(m + n, dtype=torch.uint32, device=dev)
    otb = torch.empty((m + n + 31) // 32, dtype=torch.uint32, device=dev)
    stages_mat = stages + [("replacement_materialize", lambda: lsm.replacement_materialize(
        A, B, refs, cnt, valA=vA, valB=vB, tombB=tB, out_keys=ok, out_vals=ov, out_tomb=otb))]
    ms_mat, per_mat = time_pipeline(torch, stages_mat, steps, flush)
    alg_mat = (alg + 4 * (m + n) + 4 * len(ri.tombB)   # read values and B's tombstone bits
               + 8 * N + 4 * N + 4 * ((N + 31) // 32))  # write keys, values, tombstone bits
    out[name]["materialized"] = {
        "ms_per_step": ms_mat, "gelem_s": (m + n) / (ms_mat * 1e-3) / 1e9,
        "algorithmic_bytes": alg_mat, "gbs": alg_mat / (ms_mat * 1e-3) / 1e9,
        "frac": alg_mat / (ms_mat * 1e-3) / 1e9 / peak,
        "kernel_ms": {"replacement_materialize": per_mat["replacement_materialize"]},
        "gpu_launches_per_step": 7}
    del vA, vB, tB, ok, ov, otb
    # The same step with the rank2048 directory in place of rank512 ("Suggested
    # separate modes": collision512 against collision2048 in the whole pipeline).
    d2 = torch.empty(m // 2048 + 1, dtype=torch.uint64, device=dev)
    e2 = torch.empty(m // (1 << 32) + 1, dtype=torch.uint64, device=dev)
    w4 = lsm.workspace(lsm.LSM_OP_RANK2048_BUILD, m, 0, dev)
    stages_2048 = [stages[0],
                   ("rank2048_build", lambda: lsm.rank2048_build(C, m, d2, e2, tot, w4)),
                   ("replacement_merge_compact", lambda: lsm.replacement_merge_compact_rank2048(
                       m, n, C, d2, e2, lb, refs, oa, ob, cnt, w3))]
    ms_2048, per_2048 = time_pipeline(torch, stages_2048, steps, flush)
    alg_2048 = alg - 12 * (m // 512 + 1) + 8 * (m // 2048 + 1) + 8 * len(e2)
    out[name]["rank2048"] = {
        "ms_per_step": ms_2048, "gelem_s": (m + n) / (ms_2048 * 1e-3) / 1e9,
        "algorithmic_bytes": alg_2048, "gbs": alg_2048 / (ms_2048 * 1e-3) / 1e9,
        "frac": alg_2048 / (ms_2048 * 1e-3) / 1e9 / peak,
        "kernel_ms": per_2048, "gpu_launches_per_step": 6,
        "directory_bytes": {"rank512": 12 * (m // 512 + 1) + w2.numel(),
                            "rank2048": 8 * (m // 2048 + 1) + 8 * len(e2) + w4.numel()}}
    del d2, e2, w4
    # The fused pass: mark, ordinals and refs in one tile pipeline, then the
    # rank512 build over C (the same outputs as the three calls above).
    w5 = lsm.workspace(lsm.LSM_OP_REPLACEMENT_FUSED, m, n, dev)
    stages_fu = [("replacement_merge_fused", lambda: lsm.replacement_merge_fused(
        A, B, C, lb, dir_, tot, refs, oa, ob, cnt, w5))]
    ms_fu, per_fu = time_pipeline(torch, stages_fu, steps, flush)
    out[name]["fused"] = {
        "ms_per_step": ms_fu, "gelem_s": (m + n) / (ms_fu * 1e-3) / 1e9,
        "algorithmic_bytes": alg, "gbs": alg / (ms_fu * 1e-3) / 1e9,
        "frac": alg / (ms_fu * 1e-3) / 1e9 / peak,
        "frac_of_8TBs_nominal": alg / (ms_fu * 1e-3) / 1e9 / 8000.0,
        "kernel_ms": {"fused_tile_kernel": per_fu["replacement_merge_fused"]},
        "gpu_launches_per_step": 3}
    del w5
    # The tiled direct scatter in place of the compaction ("The three
    # experimental paths", second path): the same outputs, the keys read again.
    stages_sc = stages[:2] + [("replacement_direct_scatter", lambda: lsm.replacement_direct_scatter(
        A, B, C, dir_, lb, refs, oa, ob, cnt))]
    ms_sc, per_sc = time_pipeline(torch, stages_sc, steps, flush)
    alg_sc = alg + 8 * (m + n) + 4 * n  # keys read again, lb_B read
    out[name]["direct_scatter"] = {
        "ms_per_step": ms_sc, "gelem_s": (m + n) / (ms_sc * 1e-3) / 1e9,
        "algorithmic_bytes": alg_sc, "gbs": alg_sc / (ms_sc * 1e-3) / 1e9,
        "frac": alg_sc / (ms_sc * 1e-3) / 1e9 / peak,
        "kernel_ms": per_sc, "gpu_launches_per_step": 4}
    if sweep:
        res = {}
        for kernel, label in ((0, "collision_mark"), (1, "replacement_merge_compact")):
            for v in lsm.REPLACE_VARIANTS:
                lsm.tune_replace(kernel, *v)
                _, per_v = time_pipeline(torch, stages, steps, flush)
                res["%s %d,%d" % (label, v[0], v[1])] = per_v[label]
            lsm.tune_replace(kernel, *lsm.DEFAULT_REPLACE_VARIANT[kernel])
        out[name]["variant_sweep_ms"] = res
    del A, B, C, lb, dir_, tot, refs, oa, ob, cnt, w1, w2, w3
    torch.cuda.empty_cache()


def extra_strings(lsm, torch, dev, peak, steps, flush, out):
    s = synth.strings()
    Ak = lsm.Bytes.from_numpy(s.A.key_arena, s.A.key_off, dev)
    Bk = lsm.Bytes.from_numpy(s.B.key_arena, s.B.key_off, dev)
    fc = lsm.FcInput(Ak, lsm.Bytes.from_numpy(s.A.val_arena, s.A.val_off, dev),
                     torch.from_numpy(s.A.tomb).to(dev), Bk,
                     lsm.Bytes.from_numpy(s.B.val_arena, s.B.val_off, dev),
                     torch.from_numpy(s.B.tomb).to(dev))
    m, n = Ak.count, Bk.count
    C = torch.empty((m + 31) // 32, dtype=torch.uint32, device=dev)
    lb = torch.empty(n, dtype=torch.uint32, device=dev)
    dir_ = torch.empty(3 * (m // 512 + 1), dtype=torch.uint32, device=dev)
    tot = torch.empty(1, dtype=torch.int64, device=dev)
    refs = torch.empty(m + n, dtype=torch.uint32, device=dev)
    oa = torch.empty(m, dtype=torch.uint32, device=dev)
    ob = torch.empty(n, dtype=torch.uint32, device=dev)
    cnt = torch.empty(1, dtype=torch.int64, device=dev)
    w1 = lsm.workspace(lsm.LSM_OP_COLLISION_MARK_STR, m, n, dev)
    w2 = lsm.workspace(lsm.LSM_OP_RANK_BUILD, m, 0, dev)
    w3 = lsm.workspace(lsm.LSM_OP_REPLACEMENT_COMPACT, m, n, dev)
    # the mark also writes the key prefix tables the lengths pass reads
    pA = torch.empty(2 * m, dtype=torch.uint64, device=dev)
    pB = torch.empty(2 * n, dtype=torch.uint64, device=dev)
    fc.prefixA, fc.prefixB = pA, pB
    lsm.collision_mark_str_prefix(Ak, Bk, C, lb, pA, pB, w1)
    lsm.rank_build(C, m, dir_, tot, w2)
    lsm.replacement_merge_compact(m, n, C, dir_, lb, refs, oa, ob, cnt, w3)
    N = int(cnt.item())
    lcp = torch.empty(N, dtype=torch.uint32, device=dev)
    ctrl = torch.empty(N, dtype=torch.uint32, device=dev)
    rec = torch.empty(N, dtype=torch.uint32, device=dev)
    off = torch.empty(N + 1, dtype=torch.uint64, device=dev)
    w4 = lsm.workspace(lsm.LSM_OP_FC_LENGTHS_SCAN, N, 0, dev)
    lsm.fc_lengths_scan(fc, refs, N, lcp, ctrl, rec, off, w4)
    total_bits = int(off[N:].cpu().numpy()[0])
    nwords = (total_bits + 31) // 32
    payload = torch.empty(max(nwords, 4), dtype=torch.uint32, device=dev)
    # The step: the string replacement merge in one call (partition, mark,
    # which also writes the merge bitmap, the compaction's co-ranks and the
    # key prefix tables, rank512 build, compaction), then the FC lengths
    # scan and emit. lb_B is scratch on this path and not written.
    w5 = lsm.workspace(lsm.LSM_OP_REPLACEMENT_MERGE_STR, m, n, dev)
    stages = [("replacement_merge_str", lambda: lsm.replacement_merge_str(
                  Ak, Bk, C, None, pA, pB, dir_, tot, refs, oa, ob, cnt, w5, want_lb=False)),
              ("fc_lengths_scan", lambda: lsm.fc_lengths_scan(fc, refs, N, lcp, ctrl, rec, off, w4)),
              ("fc_emit", lambda: lsm.fc_emit(fc, refs, N, lcp, ctrl, off, nwords, payload))]
    ms, per = time_pipeline(torch, stages, steps, flush)
    # the same step with the mark, the rank build and the compaction as
    # separate calls (the compaction then rebuilds the merge bitmap and its
    # co-ranks from lb_B)
    stages_sep = [("collision_mark_str", lambda: lsm.collision_mark_str_prefix(
                      Ak, Bk, C, lb, pA, pB, w1)),
                  ("rank_build", lambda: lsm.rank_build(C, m, dir_, tot, w2)),
                  ("replacement_merge_compact", lambda: lsm.replacement_merge_compact(
                      m, n, C, dir_, lb, refs, oa, ob, cnt, w3))] + stages[1:]
    ms_sep, per_sep = time_pipeline(torch, stages_sep, steps, flush)
    key_bytes = len(s.A.key_arena) + len(s.B.key_arena) + 8 * (m + n + 2)
    val_bytes = len(s.A.val_arena) + len(s.B.val_arena) + 8 * (m + n + 2) + 4 * (len(s.A.tomb) + len(s.B.tomb))
    alg = (key_bytes + val_bytes                      # keys and values read once
           + 4 * ((m + 31) // 32) + 12 * (m // 512 + 1) + 4 * N + 4 * (m + n)  # C, dir, refs, ords
           + 12 * N + 8 * (N + 1) + 4 * nwords)      # lcp, ctrl, rec_bits, bit_off, payload
    out["strings_fc_4M_4M"] = {"m": m, "n": n, "survivors": N, "payload_bits": total_bits,
                               "ms_per_step": ms, "gelem_s": (m + n) / (ms * 1e-3) / 1e9,
                               "algorithmic_bytes": alg, "gbs": alg / (ms * 1e-3) / 1e9,
                               "frac": alg / (ms * 1e-3) / 1e9 / peak, "kernel_ms": per,
                               "kernel_ms_note": "replacement_merge_str: its string mark kernel",
                               "gpu_launches_per_step": 8,
                               "workspace_bytes": {"replacement_merge_str": w5.numel(),
                                                   "fc_lengths_scan": w4.numel(),
                                                   "prefix_tables": 8 * (pA.numel() + pB.numel())},
                               "separate_calls": {
                                   "ms_per_step": ms_sep, "kernel_ms": per_sep,
                                   "gpu_launches_per_step": 10,
                                   "workspace_bytes": {"collision_mark_str": w1.numel(),
                                                       "rank_build": w2.numel(),
                                                       "replacement_merge_compact": w3.numel()}},
                               "l2": "flushed (256 MiB write) before every step"}
    # The byte profile in place of the bit profile: the same step with the
    # byte-FC lengths scan and emit.
    lcpb = torch.empty(N, dtype=torch.uint32, device=dev)
    ctrlb = torch.empty(N, dtype=torch.uint32, device=dev)
    recb = torch.empty(N, dtype=torch.uint32, device=dev)
    offb = torch.empty(N + 1, dtype=torch.uint64, device=dev)
    lsm.bytefc_lengths_scan(fc, refs, N, 0, lcpb, ctrlb, recb, offb, w4)
    total_bytes = int(offb[N:].cpu().numpy()[0])
    payb = torch.empty(max(total_bytes, 16), dtype=torch.uint8, device=dev)
    stages_b = stages[:1] + [
        ("bytefc_lengths_scan", lambda: lsm.bytefc_lengths_scan(fc, refs, N, 0, lcpb, ctrlb, recb,
                                                                offb, w4)),
        ("bytefc_emit", lambda: lsm.bytefc_emit(fc, refs, N, lcpb, ctrlb, offb, total_bytes, 0,
                                                payb))]
    ms_b, per_b = time_pipeline(torch, stages_b, steps, flush)
    alg_b = alg - 4 * nwords + total_bytes
    out["strings_fc_4M_4M"]["byte_profile"] = {
        "ms_per_step": ms_b, "payload_bytes": total_bytes,
        "gelem_s": (m + n) / (ms_b * 1e-3) / 1e9, "algorithmic_bytes": alg_b,
        "gbs": alg_b / (ms_b * 1e-3) / 1e9, "frac": alg_b / (ms_b * 1e-3) / 1e9 / peak,
        "kernel_ms": {k: per_b[k] for k in ("bytefc_lengths_scan", "bytefc_emit")},
        # the string call's four, the byte lengths with the offset scan (three), the emit
        "gpu_launches_per_step": 8}
    del lcpb, ctrlb, recb, offb, payb
    # The same step followed by the Elias-Fano navigation over bit_off.
    n_ef, L, nl, nh, G = lsm.ef_sizes(N, total_bits)
    lows = torch.empty(max(nl, 1), dtype=torch.uint64, device=dev)
    highs = torch.empty(nh, dtype=torch.uint64, device=dev)
    samples = torch.empty(2 * G, dtype=torch.uint64, device=dev)
    sparse = torch.empty(n_ef, dtype=torch.uint64, device=dev)
    nsp = torch.empty(1, dtype=torch.int64, device=dev)
    stages_ef = stages + [("fc_ef_build", lambda: lsm.fc_ef_build(
        off, N, total_bits, 0, lows, highs, samples, sparse, nsp))]
    ms_ef, per_ef = time_pipeline(torch, stages_ef, steps, flush)
    ef_bytes = 8 * n_ef + 8 * (nl + nh + 2 * G) + 8 * int(nsp.item())
    out["strings_fc_4M_4M"]["with_ef"] = {
        "ms_per_step": ms_ef, "ef_entries": n_ef, "ef_L": L,
        "ef_sparse_entries": int(nsp.item()), "ef_algorithmic_bytes": ef_bytes,
        "kernel_ms": {"fc_ef_build": per_ef["fc_ef_build"]},
        "gpu_launches_per_step": 10}


if __name__ == "__main__":
    main()
