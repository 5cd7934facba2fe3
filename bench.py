"""Benchmark of the zonal-scatter hot path on GB300.

One step = stable destination CSR build + forward + backward (every step of
the path) over one synthetic graph shaped like the 4096-atom diamond frame
of the deepmd-kit pull request "fused Triton zonal scatter for the GIE head"
(section "Numbers": N=4096, E=647170, C=32, fp32).

    python bench.py [--gpus N] [--steps K] [--warmup W] [--config n4096]
                    [--impl zs|reference] [--no-cpu-baseline] [--no-e2e]

Prints one JSON line on rank 0.  ``--impl reference`` times the fp64 CPU
oracle on the host cores instead (the only other place this file runs it).
Under torchrun every rank runs an independent replica (the path needs no
exchange between GPUs); ``value`` is the total over ranks divided by the
slowest rank's time.
"""
from __future__ import annotations

import argparse
import hashlib
import json
import os
import statistics
import subprocess
import sys
import time
from types import SimpleNamespace

import numpy as np

ROOT = os.path.dirname(os.path.abspath(__file__))
sys.path.insert(0, ROOT)

METRIC = "zonal-scatter fwd+bwd edges/s at N=4096,E=647170,C=32; % of HBM roofline"
FALLBACK_HBM_GBS = 6800.0
NOMINAL_HBM_GBS = 8000.0     # nominal HBM3e rate of the part (about 8 TB/s), reported beside the peak in use
L2_BYTES = 129 * 10 ** 6
KERNEL_SOURCES = {
    "fwd": "equivariant_interatomic_potential_gb300/csrc/zs_forward.cu",
    "bwd_csr": "equivariant_interatomic_potential_gb300/csrc/zs_backward.cu",
    "bwd_edge": "equivariant_interatomic_potential_gb300/csrc/zs_backward.cu",
    "csr": "equivariant_interatomic_potential_gb300/csrc/zs_csr.cu",
}


# ---------------------------------------------------------------- byte models

def algorithmic_bytes(N: int, E: int, C: int, lmax: int = 3) -> dict:
    """Bytes each step must move at least (fp32 data, int32 indices); ladder of
    degree lmax: R = (lmax+1)^2 - 1 coupling rows, lmax radial slots, D = R + 1
    node rows (R = 15, D = 16 at lmax = 3)."""
    D = (lmax + 1) ** 2
    R = D - 1
    fwd = E * (4 + 4 * R + 4 * lmax * C) + 4 * (N + 1) + 4 * D * N * C
    bwd = E * (4 + 4 * R + 4 * lmax * C + 4 * R + 4 * lmax * C) + 4 * D * N * C
    csr = E * (4 + 4) + 4 * (N + 1)
    return {"fwd": fwd, "bwd": bwd, "csr": csr}


def kernel_figures(ab: dict, b2b: dict, per: dict, E: int, peak: float, peak_kind: str, names,
                   marginal: dict | None = None) -> dict:
    """Per entry point: the roofline figures from the back-to-back launches
    (b2b: mean microseconds per launch) and, alongside, the launches
    bracketed inside a step (per: microseconds of each; launch latency and
    the previous kernel's L2 write-backs included) and, where given, the
    marginal cost in the step (marginal: the whole step's microseconds minus
    those of the same step without that entry point, events only at the ends
    of both loops, so programmatic overlap is kept).  Fractions of the peak
    in use and of the nominal 8 TB/s HBM3e rate."""
    kernels = {}
    for k in names:
        us = b2b[k]
        us_step = statistics.mean(per[k])
        gbs = ab[k] / (us * 1e-6) / 1e9
        kernels[k] = {"us_back_to_back": us, "algorithmic_bytes": ab[k],
                      "GBs": gbs, "frac_of_" + peak_kind: gbs / peak, "frac_of_nominal_8000": gbs / NOMINAL_HBM_GBS,
                      "edges_per_s": E / (us * 1e-6),
                      "us_in_step_mean": us_step, "us_in_step_median": statistics.median(per[k]),
                      "frac_in_step": ab[k] / (us_step * 1e-6) / 1e9 / peak}
        if marginal and k in marginal:
            kernels[k]["us_marginal_in_step"] = marginal[k]
            kernels[k]["frac_marginal_in_step"] = ab[k] / (marginal[k] * 1e-6) / 1e9 / peak
    return kernels


def metric_for(lmax: int, scaled: bool = False) -> str:
    m = METRIC if lmax == 3 else METRIC.replace("C=32;", f"C=32,lmax={lmax};")
    return m.replace("zonal-scatter", "degree-normalised zonal-scatter") if scaled else m


def scaled_extra_bytes(N: int, C: int, lmax: int) -> dict:
    """What fusing the per-node factor adds: the factor (4 B per node) and the
    unscaled output the scale's gradient needs (written by the forward, read
    with g again by the backward)."""
    node = 4 * (lmax + 1) ** 2 * C
    return {"fwd": 4 * N + node * N, "bwd": 4 * N + 2 * node * N + 4 * N}


def measured_peaks() -> tuple[float, str]:
    path = os.path.join(ROOT, "MEASURED_PEAKS.json")
    try:
        with open(path) as f:
            d = json.load(f)
        for key in ("hbm_gbs", "hbm_GBs", "copy_gbs"):
            if key in d:
                return float(d[key]), "measured"
        for v in d.values():
            if isinstance(v, dict) and "hbm_gbs" in v:
                return float(v["hbm_gbs"]), "measured"
    except (OSError, ValueError):
        pass
    return FALLBACK_HBM_GBS, "fallback"


def source_hash(rel: str) -> str:
    with open(os.path.join(ROOT, rel), "rb") as f:
        return hashlib.sha256(f.read()).hexdigest()[:16]


def ncu_traffic(kernel_key: str, workload: str):
    """DRAM bytes per launch from the committed ncu summary, if the kernel
    source is unchanged since the counters were taken."""
    path = os.path.join(ROOT, "profiles", "ncu_traffic.json")
    try:
        with open(path) as f:
            d = json.load(f)
        e = d[workload][kernel_key]
        if e.get("source_sha256_16") != source_hash(KERNEL_SOURCES[kernel_key]):
            return None
        return int(e["dram_bytes_per_launch"])
    except (OSError, KeyError, ValueError):
        return None


def make_graph(config: str, lmax: int = 3):
    """One of the named configurations, or "uniform:N:E" (a seeded graph of E
    edges with uniform destinations over N nodes, C = 32: extra sizes for
    profiling, not a headline workload)."""
    from equivariant_interatomic_potential_gb300 import workloads
    if config.startswith("uniform:"):
        _, n, e = config.split(":")
        return workloads.make_random(int(n), int(e), 32, seed=int(n) + int(e), lmax=lmax)
    return workloads.make_workload(config, lmax=lmax)


# ---------------------------------------------------------------- ranks

def reduce_max(value: float, world: int, device) -> float:
    """Maximum of a per-rank scalar over all ranks (the slowest rank's time)."""
    if world <= 1:
        return float(value)
    import torch
    import torch.distributed as dist
    t = torch.tensor([float(value)], dtype=torch.float64, device=device)
    dist.all_reduce(t, op=dist.ReduceOp.MAX)
    return float(t.item())


def job_throughput(units_per_rank: int, steps: int, max_ms: float, world: int) -> float:
    """Whole-job units per second: every rank's units over the slowest rank's time."""
    return world * units_per_rank * steps / (max_ms / 1e3)


def workload_config(w, backward: str, scaled: bool = False) -> dict:
    entry = "zs_backward_csr" if backward == "csr" else "zs_backward"
    if scaled:
        entry = "zs_backward_scaled"
    lmax = w.rad.shape[1]
    rows = "/".join(str(2 * l + 1) for l in range(1, lmax + 1))
    return {"workload": f"{w.name}: N={w.N}, E={w.E}, C={w.C}, lmax={lmax} (rows {rows}), fp32, seed {w.seed}",
            "step": "zs_build_csr + " + ("zs_forward_scaled" if scaled else "zs_forward") + " + " + entry,
            "l2": ("inputs larger than L2" if w.coup.nbytes + w.rad.nbytes > L2_BYTES else
                   "inputs smaller than L2, no flush") + " (coup+rad = %.0f MB)" % ((w.coup.nbytes + w.rad.nbytes) / 1e6)}


# ---------------------------------------------------------------- clocks

class ClockSampler:
    """nvidia-smi sampling of SM clock and throttle reasons during the timed region."""
    FIELDS = ("index,clocks.sm,clocks.max.sm,power.draw,clocks_event_reasons.active,"
              "clocks_event_reasons.hw_slowdown,clocks_event_reasons.hw_thermal_slowdown,"
              "clocks_event_reasons.sw_thermal_slowdown,clocks_event_reasons.sw_power_cap")

    def __init__(self, gpu_index: int):
        self.gpu = gpu_index
        self.proc = None
        self.path = os.path.join("/tmp", f"zs_clocks_{os.getpid()}.csv")

    def __enter__(self):
        try:
            self.fh = open(self.path, "w")
            self.proc = subprocess.Popen(["nvidia-smi", f"--id={self.gpu}", f"--query-gpu={self.FIELDS}",
                                          "--format=csv,noheader,nounits", "-lms", "100"],
                                         stdout=self.fh, stderr=subprocess.DEVNULL)
        except (OSError, ValueError):
            self.proc = None
        time.sleep(0.3)
        return self

    def __exit__(self, *exc):
        if self.proc is not None:
            time.sleep(0.15)
            self.proc.terminate()
            try:
                self.proc.wait(timeout=5)
            except subprocess.TimeoutExpired:
                self.proc.kill()
            self.fh.close()

    def summary(self) -> dict:
        if self.proc is None:
            return {"sm_mhz": None, "sm_max_mhz": None, "reasons": ["nvidia-smi unavailable"]}
        sm, smax, reasons = [], [], set()
        names = ["hw_slowdown", "hw_thermal_slowdown", "sw_thermal_slowdown", "sw_power_cap"]
        with open(self.path) as f:
            for line in f:
                p = [x.strip() for x in line.split(",")]
                if len(p) < 9:
                    continue
                try:
                    sm.append(float(p[1]))
                    smax.append(float(p[2]))
                except ValueError:
                    continue
                for n, v in zip(names, p[5:9]):
                    if v.lower() == "active":
                        reasons.add(n)
        try:
            os.remove(self.path)
        except OSError:
            pass
        if not sm:
            return {"sm_mhz": None, "sm_max_mhz": None, "reasons": ["no samples"]}
        return {"sm_mhz": statistics.median(sm), "sm_max_mhz": max(smax), "reasons": sorted(reasons),
                "samples": len(sm)}


# ---------------------------------------------------------------- GPU arm

def run_gpu_arm(args, rank: int, world: int) -> dict | None:
    import torch
    import torch.distributed as dist

    from equivariant_interatomic_potential_gb300 import workloads, zs

    local = int(os.environ.get("LOCAL_RANK", "0"))
    torch.cuda.set_device(local)
    w = make_graph(args.config, lmax=args.lmax)
    N, E, C, L = w.N, w.E, w.C, args.lmax
    D, R = (L + 1) ** 2, (L + 1) ** 2 - 1
    dev = torch.device("cuda", local)
    lib = zs.load()

    # Resident input/output sets, rotated step by step, so that no step finds
    # lines an earlier step left in L2 (a new batch every step, as in training):
    # enough sets that their arrays exceed L2 several times over.
    def make_set(src=None):
        b = SimpleNamespace()
        if src is None:
            b.dst = torch.from_numpy(w.dst).to(dev)
            b.coup = torch.from_numpy(w.coup).to(dev)
            b.rad = torch.from_numpy(w.rad).to(dev)
            b.g = torch.from_numpy(w.grad_out).to(dev)
        else:
            b.dst, b.coup, b.rad, b.g = (t.clone() for t in (src.dst, src.coup, src.rad, src.g))
        b.row_ptr = torch.empty(N + 1, dtype=torch.int32, device=dev)
        b.perm = torch.empty(E, dtype=torch.int32, device=dev)
        b.bad = torch.empty(1, dtype=torch.int32, device=dev)
        b.ws_csr = torch.empty(max(1, zs.zs_build_csr_workspace_bytes(E, N)), dtype=torch.uint8, device=dev)
        b.ws_fwd = torch.empty(max(1, zs.zs_forward_workspace_bytes(E, N, C, L)), dtype=torch.uint8, device=dev)
        b.out = torch.empty((N, D, C), dtype=torch.float32, device=dev)
        b.d_coup = torch.empty((E, R), dtype=torch.float32, device=dev)
        b.d_rad = torch.empty((E, L, C), dtype=torch.float32, device=dev)
        if args.scaled:
            b.out_raw = torch.empty_like(b.out)
            b.d_scale = torch.empty(N, dtype=torch.float32, device=dev)
        return b

    first = make_set()
    set_bytes = sum(t.numel() * t.element_size() for t in vars(first).values())
    n_sets = args.sets or max(3, min(64, -(-4 * L2_BYTES // max(1, set_bytes))))
    sets = [first] + [make_set(first) for _ in range(n_sets - 1)]
    stream = torch.cuda.current_stream(dev)
    sp = stream.cuda_stream

    P = lambda t: t.data_ptr()  # noqa: E731
    csr_ws_bytes, fwd_ws_bytes = first.ws_csr.numel(), first.ws_fwd.numel()

    def csr(b):
        st = lib.zs_build_csr(P(b.dst), E, N, P(b.row_ptr), P(b.perm), P(b.bad), P(b.ws_csr), csr_ws_bytes, sp)
        assert st == 0, lib.zs_last_error()

    def fwd(b):
        st = lib.zs_forward(P(b.coup), P(b.rad), P(b.row_ptr), P(b.perm), E, N, C, L, P(b.out), P(b.ws_fwd),
                            fwd_ws_bytes, sp)
        assert st == 0, lib.zs_last_error()

    def bwd_edge(b):
        st = lib.zs_backward(P(b.g), P(b.coup), P(b.rad), P(b.dst), E, N, C, L, P(b.d_coup), P(b.d_rad), sp)
        assert st == 0, lib.zs_last_error()

    def bwd_csr(b):
        st = lib.zs_backward_csr(P(b.g), P(b.coup), P(b.rad), P(b.row_ptr), P(b.perm), E, N, C, L, P(b.d_coup),
                                 P(b.d_rad), sp)
        assert st == 0, lib.zs_last_error()

    bwd, bwd_other, other_name = (bwd_csr, bwd_edge, "bwd_edge") if args.backward == "csr" else \
        (bwd_edge, bwd_csr, "bwd_csr")

    if args.scaled:
        # the degree normalisation fused in: s[n] = 1/sqrt(in-degree), 0 without edges
        indeg = np.bincount(w.dst[(w.dst >= 0) & (w.dst < N)], minlength=N)
        s_host = np.where(indeg > 0, 1.0 / np.sqrt(np.maximum(indeg, 1)), 0.0).astype(np.float32)
        node_scale = torch.from_numpy(s_host).to(dev)

        def fwd(b):
            st = lib.zs_forward_scaled(P(b.coup), P(b.rad), P(b.row_ptr), P(b.perm), P(node_scale), E, N, C, L,
                                       P(b.out), P(b.out_raw), P(b.ws_fwd), fwd_ws_bytes, sp)
            assert st == 0, lib.zs_last_error()

        def bwd(b):
            st = lib.zs_backward_scaled(P(b.g), P(b.coup), P(b.rad), P(b.dst), P(node_scale), P(b.out_raw), E, N,
                                        C, L, P(b.d_coup), P(b.d_rad), P(b.d_scale), sp)
            assert st == 0, lib.zs_last_error()

        def fwd_unfused(b):
            plain_fwd(b)
            torch.mul(b.out_raw, node_scale[:, None, None], out=b.out)

        def bwd_unfused(b):
            gs = b.g * node_scale[:, None, None]
            st = lib.zs_backward(P(gs), P(b.coup), P(b.rad), P(b.dst), E, N, C, L, P(b.d_coup), P(b.d_rad), sp)
            assert st == 0, lib.zs_last_error()
            torch.sum(b.g[:, 1:] * b.out_raw[:, 1:], dim=(1, 2), out=b.d_scale)

        def plain_fwd(b):
            st = lib.zs_forward(P(b.coup), P(b.rad), P(b.row_ptr), P(b.perm), E, N, C, L, P(b.out_raw),
                                P(b.ws_fwd), fwd_ws_bytes, sp)
            assert st == 0, lib.zs_last_error()

    # zs_build_csr: three launches on its one-pass counting path (N + 1 <= 5120; one for E <= 8192),
    # else three per 8-bit radix pass plus the row_ptr pass (one launch for E = 0);
    # zs_forward: one kernel at C = 32 (aligned tensors), else main kernel and
    # fix-up; the backward: one kernel (none for E = 0)
    if E == 0:
        csr_launches = 1
    elif N + 1 <= 5120:
        csr_launches = 1 if E <= 8192 else 3   # one CTA, one launch for up to 8192 edges
    else:
        csr_launches = 3 * max(1, (max(N, 1).bit_length() + 7) // 8) + 1
    launches_per_step = csr_launches + (1 if C == 32 else 2) + (1 if E > 0 else 0)
    if args.scaled:
        launches_per_step += 1   # the scale's gradient

    for i in range(max(args.warmup, n_sets)):
        b = sets[i % n_sets]
        csr(b); fwd(b); bwd(b)
    torch.cuda.synchronize()

    def barrier():
        if world > 1:
            dist.barrier()

    # the timed region: K whole steps back to back, events only at its ends
    # (an event between two kernels would break their programmatic overlap)
    t0 = torch.cuda.Event(enable_timing=True)
    t1 = torch.cuda.Event(enable_timing=True)
    with ClockSampler(local) as clocks:
        barrier()
        torch.cuda.synchronize()
        t0.record(stream)
        for i in range(args.steps):
            b = sets[i % n_sets]
            csr(b)
            fwd(b)
            bwd(b)
        t1.record(stream)
        torch.cuda.synchronize()
        barrier()
    total_ms = t0.elapsed_time(t1)
    clock = clocks.summary()
    # per-kernel durations (1): each launch of a step bracketed by events on the same stream
    ev = {k: [(torch.cuda.Event(enable_timing=True), torch.cuda.Event(enable_timing=True))
              for _ in range(args.steps)] for k in ("csr", "fwd", "bwd")}
    for i in range(args.steps):
        b = sets[i % n_sets]
        for k, fn in (("csr", csr), ("fwd", fwd), ("bwd", bwd)):
            ev[k][i][0].record(stream)
            fn(b)
            ev[k][i][1].record(stream)
    torch.cuda.synchronize()
    per = {k: [a.elapsed_time(b) * 1e3 for a, b in ev[k]] for k in ev}   # microseconds
    # the other backward entry point, timed on its own for comparison
    oth = [(torch.cuda.Event(enable_timing=True), torch.cuda.Event(enable_timing=True)) for _ in range(args.steps)]
    for i, (a, b) in enumerate(oth):
        a.record(stream)
        bwd_other(sets[i % n_sets])
        b.record(stream)
    torch.cuda.synchronize()
    per[other_name] = [a.elapsed_time(b) * 1e3 for a, b in oth]

    # per-kernel durations (3): the step's time minus that of the same step
    # without one entry point (its inputs are still valid: each set's CSR was
    # built in the warm-up), K steps between two events each
    def loop_us(fns):
        for i in range(3):
            for fn in fns:
                fn(sets[i % n_sets])
        a = torch.cuda.Event(enable_timing=True)
        z = torch.cuda.Event(enable_timing=True)
        torch.cuda.synchronize()
        a.record(stream)
        for i in range(args.steps):
            for fn in fns:
                fn(sets[i % n_sets])
        z.record(stream)
        torch.cuda.synchronize()
        return a.elapsed_time(z) * 1e3 / args.steps
    step_us = loop_us((csr, fwd, bwd))
    marginal = {"csr": step_us - loop_us((fwd, bwd)), "fwd": step_us - loop_us((csr, bwd)),
                "bwd": step_us - loop_us((csr, fwd))}
    # per-kernel durations (2): K launches of one entry point back to back over
    # the rotating sets, events at the ends: the steady-state cost of a launch,
    # its own write-backs included and its launch latency overlapped
    b2b = {}
    for k, fn in (("csr", csr), ("fwd", fwd), ("bwd", bwd), (other_name, bwd_other)):
        for i in range(3):
            fn(sets[i % n_sets])
        a = torch.cuda.Event(enable_timing=True)
        z = torch.cuda.Event(enable_timing=True)
        torch.cuda.synchronize()
        a.record(stream)
        for i in range(args.steps):
            fn(sets[i % n_sets])
        z.record(stream)
        torch.cuda.synchronize()
        b2b[k] = a.elapsed_time(z) * 1e3 / args.steps
    unfused = None
    if args.scaled:
        # the same step with the factor applied by separate torch ops
        ev_u = {k: [(torch.cuda.Event(enable_timing=True), torch.cuda.Event(enable_timing=True))
                    for _ in range(args.steps)] for k in ("fwd", "bwd")}
        for i in range(args.warmup):
            b = sets[i % n_sets]
            csr(b); fwd_unfused(b); bwd_unfused(b)
        torch.cuda.synchronize()
        for i in range(args.steps):
            b = sets[i % n_sets]
            csr(b)
            for k, fn in (("fwd", fwd_unfused), ("bwd", bwd_unfused)):
                ev_u[k][i][0].record(stream)
                fn(b)
                ev_u[k][i][1].record(stream)
        torch.cuda.synchronize()
        unfused = {k + "_us": statistics.median(a.elapsed_time(b) * 1e3 for a, b in ev_u[k]) for k in ev_u}
        unfused["how"] = "zs_forward + torch.mul; g*s in torch, zs_backward, torch sum for d_scale"
        unfused["fused_us_same_protocol"] = {k: statistics.median(per[k]) for k in ("fwd", "bwd")}
    zs.zs_check_timeouts()

    # end to end through the public API: pinned host buffers in, results out
    e2e = None
    if not args.no_e2e:
        h_dst = torch.from_numpy(w.dst).pin_memory()
        h_coup = torch.from_numpy(w.coup).pin_memory()
        h_rad = torch.from_numpy(w.rad).pin_memory()
        h_g = torch.from_numpy(w.grad_out).pin_memory()
        h_out = torch.empty_like(first.out, device="cpu").pin_memory()
        h_dc = torch.empty_like(first.d_coup, device="cpu").pin_memory()
        h_dr = torch.empty_like(first.d_rad, device="cpu").pin_memory()

        # Two sets of device buffers: step i+1's inputs arrive (copy stream in) while
        # step i computes and step i-1's results leave (copy stream out).
        def buffers():
            return {k: torch.empty_like(v) for k, v in vars(first).items()}

        del sets[1:]
        bufs = [buffers(), buffers()]
        n_copy = max(1, args.copy_streams)
        s_in = [torch.cuda.Stream(dev) for _ in range(n_copy)]
        s_out = [torch.cuda.Stream(dev) for _ in range(n_copy)]
        s_comp = torch.cuda.Stream(dev)
        ev_in = [[torch.cuda.Event() for _ in range(n_copy)] for _ in range(2)]
        ev_comp = [torch.cuda.Event() for _ in range(2)]
        ev_out = [[torch.cuda.Event() for _ in range(n_copy)] for _ in range(2)]
        used = [False, False]

        def chunked(pairs):
            # (dst, src) copies split into n_copy slices along dim 0, one slice per copy stream
            for d, src in pairs:
                rows = d.shape[0]
                for c in range(n_copy):
                    lo, hi = rows * c // n_copy, rows * (c + 1) // n_copy
                    if hi > lo:
                        yield c, d[lo:hi], src[lo:hi]

        def e2e_step(i):
            k = i % 2
            B = bufs[k]
            for c in range(n_copy):
                if used[k]:
                    s_in[c].wait_event(ev_comp[k])     # step i-2 is done with these inputs
            for c, d, src in chunked(((B["dst"], h_dst), (B["coup"], h_coup), (B["rad"], h_rad), (B["g"], h_g))):
                with torch.cuda.stream(s_in[c]):
                    d.copy_(src, non_blocking=True)
            for c in range(n_copy):
                ev_in[k][c].record(s_in[c])
            with torch.cuda.stream(s_comp):
                for c in range(n_copy):
                    s_comp.wait_event(ev_in[k][c])
                if used[k]:
                    for c in range(n_copy):
                        s_comp.wait_event(ev_out[k][c])   # step i-2's results have left
                zs.zs_build_csr(B["dst"], N, row_ptr=B["row_ptr"], perm=B["perm"], bad_dst_count=B["bad"],
                                workspace=B["ws_csr"])
                if args.scaled:
                    zs.zs_forward_scaled(B["coup"], B["rad"], B["row_ptr"], B["perm"], node_scale, N, out=B["out"],
                                         out_raw=B["out_raw"], workspace=B["ws_fwd"])
                    zs.zs_backward_scaled(B["g"], B["coup"], B["rad"], B["dst"], node_scale, N, out_raw=B["out_raw"],
                                          d_coup=B["d_coup"], d_rad=B["d_rad"], d_scale=B["d_scale"])
                elif args.backward == "csr":
                    zs.zs_forward(B["coup"], B["rad"], B["row_ptr"], B["perm"], N, out=B["out"], workspace=B["ws_fwd"])
                    zs.zs_backward_csr(B["g"], B["coup"], B["rad"], B["row_ptr"], B["perm"], N, d_coup=B["d_coup"],
                                       d_rad=B["d_rad"])
                else:
                    zs.zs_forward(B["coup"], B["rad"], B["row_ptr"], B["perm"], N, out=B["out"], workspace=B["ws_fwd"])
                    zs.zs_backward(B["g"], B["coup"], B["rad"], B["dst"], N, d_coup=B["d_coup"], d_rad=B["d_rad"])
                ev_comp[k].record(s_comp)
            for c in range(n_copy):
                s_out[c].wait_event(ev_comp[k])
            for c, d, src in chunked(((h_out, B["out"]), (h_dc, B["d_coup"]), (h_dr, B["d_rad"]))):
                with torch.cuda.stream(s_out[c]):
                    d.copy_(src, non_blocking=True)
            for c in range(n_copy):
                ev_out[k][c].record(s_out[c])
            used[k] = True

        for i in range(max(2, args.warmup)):
            e2e_step(i)
        torch.cuda.synchronize()
        barrier()
        a = torch.cuda.Event(enable_timing=True)
        b = torch.cuda.Event(enable_timing=True)
        a.record(s_in[0])
        for c in range(1, n_copy):
            s_in[c].wait_event(a)
        for i in range(args.steps):
            e2e_step(i)
        for c in range(1, n_copy):
            s_out[0].wait_stream(s_out[c])
        b.record(s_out[0])
        torch.cuda.synchronize()
        barrier()
        e2e_ms = reduce_max(a.elapsed_time(b), world, dev)
        h2d = sum(t.numel() * t.element_size() for t in (h_dst, h_coup, h_rad, h_g))
        d2h = sum(t.numel() * t.element_size() for t in (h_out, h_dc, h_dr))
        # what the host link allows: the same copies, both directions at once, no kernels
        a2 = torch.cuda.Event(enable_timing=True)
        b2 = torch.cuda.Event(enable_timing=True)
        torch.cuda.synchronize()
        a2.record(s_in[0])
        s_out[0].wait_event(a2)
        for i in range(args.steps):
            B = bufs[i % 2]
            with torch.cuda.stream(s_in[0]):
                for d, src in ((B["dst"], h_dst), (B["coup"], h_coup), (B["rad"], h_rad), (B["g"], h_g)):
                    d.copy_(src, non_blocking=True)
            with torch.cuda.stream(s_out[0]):
                for d, src in ((h_out, B["out"]), (h_dc, B["d_coup"]), (h_dr, B["d_rad"])):
                    d.copy_(src, non_blocking=True)
        s_in[0].wait_stream(s_out[0])
        b2.record(s_in[0])
        torch.cuda.synchronize()
        link_ms = a2.elapsed_time(b2) / args.steps
        e2e = {"value": job_throughput(E, args.steps, e2e_ms, world), "unit": "edges/s",
               "h2d_bytes_per_step": h2d, "d2h_bytes_per_step": d2h,
               "ms_per_step": e2e_ms / args.steps,
               "pipeline": f"two buffer sets: step i+1's host-to-device copies and step i-1's device-to-host "
                           f"copies overlap step i; each copy split over {n_copy} stream(s) per direction",
               "host_link": {"ms_per_step": link_ms, "GBs": (h2d + d2h) / (link_ms * 1e-3) / 1e9,
                             "how": "the same copies alone, host to device and device to host at once"}}

    total_ms = reduce_max(total_ms, world, dev)
    if rank != 0:
        return None

    ab = algorithmic_bytes(N, E, C, L)
    if args.scaled:
        extra = scaled_extra_bytes(N, C, L)
        ab["fwd"] += extra["fwd"]
        ab["bwd"] += extra["bwd"]
    peak, peak_kind = measured_peaks()
    ab["bwd_edge"] = ab["bwd_csr"] = ab["bwd"]
    kernels = kernel_figures(ab, b2b, per, E, peak, peak_kind, ("csr", "fwd", "bwd", other_name), marginal)
    dom = max(("fwd", "bwd"), key=lambda k: kernels[k]["us_back_to_back"])
    bwd_entry = "zs_backward_csr" if args.backward == "csr" else "zs_backward"
    roof = {"kernel": {"fwd": "zs_forward", "bwd": bwd_entry}[dom], "bound": "hbm",
            "achieved": kernels[dom]["GBs"], "peak": peak, "unit": "GB/s",
            "frac": kernels[dom]["GBs"] / peak, "peak_kind": peak_kind,
            "frac_of_nominal_8000": kernels[dom]["GBs"] / NOMINAL_HBM_GBS,
            "traffic": ncu_traffic(dom if dom == "fwd" else "bwd_" + args.backward,
                                   args.config if L == 3 else f"{args.config}@lmax{L}") if not args.scaled else None,
            "algorithmic_bytes_per_launch": ab[dom]}
    ms_per_step = total_ms / args.steps
    fwd_bwd_us = kernels["fwd"]["us_back_to_back"] + kernels["bwd"]["us_back_to_back"]
    res = {
        "metric": metric_for(L, args.scaled),
        "value": job_throughput(E, args.steps, total_ms, world),
        "unit": "edges/s",
        "n_gpus": world,
        "steps": args.steps,
        "warmup": args.warmup,
        "ms_per_step": ms_per_step,
        "higher_is_better": True,
        "scaling": "weak",
        "vs_baseline": None,
        "dtype": "f32",
        "data": "synthetic",
        "config": dict(workload_config(w, args.backward, args.scaled),
                       parallelism="replicas" if world > 1 else "single GPU",
                       l2=f"{n_sets} resident input/output sets of {set_bytes / 1e6:.0f} MB rotated step by step "
                          f"({n_sets * set_bytes / 1e6:.0f} MB against a {L2_BYTES / 1e6:.0f} MB L2); no flush"),
        "fwd_bwd_edges_per_s": E / (fwd_bwd_us * 1e-6),
        "kernels": kernels,
        "roofline": roof,
        "clocks": clock,
        "e2e": e2e,
        "gpu_launches": launches_per_step * args.steps,
    }
    if unfused is not None:
        res["unfused"] = unfused
    return res


# ---------------------------------------------------------------- CPU oracle

def run_oracle(config: str, min_seconds: float, w=None, lmax: int = 3, threads: int = 1) -> dict:
    """The fp64 oracle (C; its node and edge loops on `threads` host threads) on
    the full graph, repeated until min_seconds of CPU work has been timed."""
    import oracle
    from equivariant_interatomic_potential_gb300 import workloads

    w = make_graph(config, lmax=lmax) if w is None else w
    oracle.build()
    oracle.set_threads(threads)
    reps, t_csr, t_fwd, t_bwd = 0, 0.0, 0.0, 0.0
    while reps == 0 or (t_csr + t_fwd + t_bwd) < min_seconds:
        a = time.perf_counter()
        row_ptr, perm, _ = oracle.build_csr(w.dst, w.N)
        b = time.perf_counter()
        oracle.forward(w.coup, w.rad, row_ptr, perm, w.N)
        c = time.perf_counter()
        oracle.backward(w.grad_out, w.coup, w.rad, w.dst, w.N)
        d = time.perf_counter()
        t_csr += b - a
        t_fwd += c - b
        t_bwd += d - c
        reps += 1
    tot = t_csr + t_fwd + t_bwd
    oracle.set_threads(1)
    how = "fp64 C, one thread" if threads == 1 else f"fp64 C, node and edge loops over {threads} threads (OpenMP)"
    return {"value": w.E * reps / tot, "unit": "edges/s", "cores": threads, "kind": "oracle",
            "sample": f"full {config} graph (N={w.N}, E={w.E}, C={w.C}), csr+forward+backward, "
                      f"{reps} repetition(s), {tot:.1f} s, {how}",
            "ms_per_step": tot / reps * 1e3,
            "fwd_bwd_edges_per_s": w.E * reps / (t_fwd + t_bwd)}


# ---------------------------------------------------------------- main

def main():
    ap = argparse.ArgumentParser()
    ap.add_argument("--gpus", type=int, default=1)
    ap.add_argument("--steps", type=int, default=30)
    ap.add_argument("--warmup", type=int, default=8)
    ap.add_argument("--config", default="n4096")
    ap.add_argument("--impl", default="zs", choices=["zs", "reference"])
    ap.add_argument("--backward", default="edge", choices=["csr", "edge"],
                    help="backward entry point timed in the step (the other is timed alongside)")
    ap.add_argument("--no-cpu-baseline", action="store_true")
    ap.add_argument("--no-e2e", action="store_true")
    ap.add_argument("--cpu-seconds", type=float, default=10.0)
    ap.add_argument("--copy-streams", type=int, default=1,
                    help="streams per copy direction in the end-to-end measurement")
    ap.add_argument("--scaled", action="store_true",
                    help="step with the degree normalisation fused in (zs_forward_scaled, zs_backward_scaled)")
    ap.add_argument("--sets", type=int, default=0,
                    help="resident input/output sets the timed loops rotate through (0: enough to exceed 4x L2)")
    ap.add_argument("--lmax", type=int, default=3, choices=[1, 2, 3, 4, 5],
                    help="ladder degree of the operands (3: the 3/5/7 rows of the headline workload)")
    args = ap.parse_args()
    if args.warmup < 3:
        args.warmup = 3

    world = int(os.environ.get("WORLD_SIZE", "1"))
    rank = int(os.environ.get("RANK", "0"))

    if args.impl == "reference":
        # the oracle on the host cores, rank 0 only
        if rank != 0:
            return
        from equivariant_interatomic_potential_gb300 import workloads
        w = make_graph(args.config, lmax=args.lmax)
        cores = os.cpu_count() or 1
        t0 = time.perf_counter()
        steps = []
        for i in range(args.warmup + args.steps):
            r = run_oracle(args.config, 0.0, w, threads=cores)
            if i >= args.warmup:
                steps.append(r["ms_per_step"])
        ms = statistics.mean(steps)
        val = w.E / (ms / 1e3)
        sample = (f"full {w.name} graph (N={w.N}, E={w.E}, C={w.C}) per step: csr build, forward, backward, "
                  f"fp64 C over {cores} host threads, {args.steps} timed steps after {args.warmup} warm-up")
        res = {"impl": "reference", "metric": metric_for(args.lmax), "value": val, "unit": "edges/s", "n_gpus": world,
               "steps": args.steps, "warmup": args.warmup, "ms_per_step": ms, "higher_is_better": True,
               "scaling": "weak", "vs_baseline": None, "dtype": "f64", "data": "synthetic",
               "config": dict(workload_config(w, args.backward), parallelism="replicas" if world > 1 else "single GPU"),
               "cpu_baseline": {"value": val, "unit": "edges/s", "cores": cores, "kind": "oracle", "sample": sample},
               "e2e": {"value": val, "unit": "edges/s", "h2d_bytes_per_step": 0, "d2h_bytes_per_step": 0},
               "wall_s": time.perf_counter() - t0}
        print(json.dumps(res))
        return

    import torch
    import torch.distributed as dist
    if world > 1:
        dist.init_process_group("nccl")
    try:
        res = run_gpu_arm(args, rank, world)
        if rank == 0 and res is not None:
            if not args.no_cpu_baseline:
                res["cpu_baseline"] = run_oracle(args.config, args.cpu_seconds, lmax=args.lmax)
                res["cpu_baseline_all_cores"] = run_oracle(args.config, args.cpu_seconds / 2, lmax=args.lmax,
                                                           threads=os.cpu_count() or 1)
            print(json.dumps(res))
    finally:
        if world > 1:
            dist.destroy_process_group()
    del torch


if __name__ == "__main__":
    main()
