"""Benchmark of the INT4 MatMulNBits decode GEMV (headline) and the other measured paths.

``python bench.py [--gpus N] [--steps K] [--warmup W] [--impl reference] [--quick]``

Headline (N = 1 and per rank under torchrun): the 7B-class attention-projection decode
GEMV (M = 1, K = N = 4096, block 32, fp16 scales, asymmetric zero points, fp16
activations ~N(0,1) clipped to +-4).  One step is one replay of a CUDA graph holding 1000
``mnb_gemv`` calls launched with programmatic dependent launch; the calls cycle through
enough weight copies (> 3 x L2) that every call streams its weights from HBM.  ``value``
is the effective bandwidth (algorithmic bytes: packed weights + scales + zero points +
A + Y) over all ranks.

Secondary lines in the same JSON record: the M = 2048 prefill GEMM (TFLOP/s, the
metric's second half), the fused gate/up SwiGLU GEMV, the down-projection GEMV and the
small-M verify GEMMs, each timed the same way with rotating copies.  ``--impl reference``
times the fp64 CPU oracle instead (the deliberately slow baseline arm).
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

import mnb_synth as syn  # noqa: E402

METRIC = "M=1 GEMV µs/call & GB/s (% of HBM peak); M=2048 GEMM TFLOP/s (% tensor peak)"
HEADLINE = "gemv_attnproj_k4096_n4096"
CALLS_PER_STEP = 1000
FALLBACK_PEAKS = {"hbm_gbs": 6800.0, "bf16_tflops": 1900.0, "bf16_tflops_sustained": 1700.0}


# ---------------------------------------------------------------------------------
# Algorithmic byte and flop counts
# ---------------------------------------------------------------------------------
def weight_bytes(wl: syn.Workload) -> int:
    s = 2 if wl.scales_dtype == "f16" else 4
    zp = wl.N * wl.zp_row_bytes if wl.has_zp else 0
    return wl.N * wl.K // 2 + wl.N * wl.k_blocks * s + zp


def call_bytes(wl: syn.Workload, n_weights: int = 1) -> int:
    return n_weights * weight_bytes(wl) + wl.M * wl.K * 2 + wl.M * wl.N * 2


def call_flops(wl: syn.Workload, n_weights: int = 1) -> int:
    return 2 * n_weights * wl.M * wl.N * wl.K


def load_peaks():
    path = os.path.join(ROOT, "MEASURED_PEAKS.json")
    if os.path.exists(path):
        with open(path) as f:
            d = json.load(f)
        return d, "measured"
    return dict(FALLBACK_PEAKS), "fallback"


def source_digest(files):
    h = hashlib.sha256()
    for f in files:
        with open(os.path.join(ROOT, f), "rb") as fh:
            h.update(fh.read())
    return h.hexdigest()[:16]


def profiled_traffic(kernel_key: str, files):
    """DRAM bytes per launch from the committed ncu summary, if it matches the source."""
    path = os.path.join(ROOT, "profiles", "dram_traffic.txt")
    if not os.path.exists(path):
        return None
    digest = source_digest(files)
    with open(path) as f:
        for line in f:
            parts = line.split()
            if len(parts) >= 3 and not line.startswith("#") and parts[0] == kernel_key:
                if parts[1] == digest:
                    return float(parts[2])
    return None


# ---------------------------------------------------------------------------------
# Clock sampling during the timed regions
# ---------------------------------------------------------------------------------
class ClockSampler:
    FIELDS = ("index,clocks.sm,clocks.max.sm,power.draw,clocks_event_reasons.active,"
              "clocks_event_reasons.hw_slowdown,clocks_event_reasons.hw_thermal_slowdown,"
              "clocks_event_reasons.sw_thermal_slowdown,clocks_event_reasons.sw_power_cap")

    def __init__(self, gpu_index: int, path: str | None):
        self.proc = None
        self.path = path
        self.gpu_index = gpu_index
        self.windows = []

    def start(self):
        if self.path is None:
            return
        try:
            self.fh = open(self.path, "w")
            self.proc = subprocess.Popen(
                ["nvidia-smi", "-i", str(self.gpu_index), f"--query-gpu={self.FIELDS}",
                 "--format=csv,noheader,nounits", "-lms", "100"],
                stdout=self.fh, stderr=subprocess.DEVNULL)
        except (OSError, FileNotFoundError):
            self.proc = None

    def mark(self, begin: bool):
        if begin:
            self.windows.append([time.time(), None])
        elif self.windows:
            self.windows[-1][1] = time.time()

    def stop(self):
        if self.proc is None:
            return {"sm_mhz": None, "sm_max_mhz": None, "reasons": ["clock sampling unavailable"]}
        time.sleep(0.25)
        self.proc.terminate()
        self.proc.wait(timeout=5)
        self.fh.close()
        sm, smax, reasons = [], None, set()
        with open(self.path) as f:
            rows = [r.strip().split(", ") for r in f if r.strip()]
        for r in rows:
            try:
                sm.append(float(r[1]))
                smax = float(r[2])
                names = ["hw_slowdown", "hw_thermal_slowdown", "sw_thermal_slowdown", "sw_power_cap"]
                for nm, v in zip(names, r[5:9]):
                    if v.strip().lower() == "active":
                        reasons.add(nm)
            except (ValueError, IndexError):
                continue
        loaded = sorted(sm)[len(sm) // 2:] if sm else []
        return {"sm_mhz": statistics.median(loaded) if loaded else None, "sm_max_mhz": smax,
                "reasons": sorted(reasons), "samples": len(sm)}


# ---------------------------------------------------------------------------------
# Device benchmarks
# ---------------------------------------------------------------------------------
class DeviceBench:
    def __init__(self, torch, mnb, dev, l2_bytes, rank):
        self.torch, self.mnb, self.dev, self.l2, self.rank = torch, mnb, dev, l2_bytes, rank
        self.launches = 0

    def copies_for(self, bytes_per_copy: int) -> int:
        return max(2, -(-3 * self.l2 // max(1, bytes_per_copy)))

    def upload_weights(self, wl, tag, copies):
        """`copies` device copies of one seeded weight (same values, distinct buffers)."""
        torch = self.torch
        w = syn.make_weight(wl, tag)
        base = [torch.from_numpy(np.ascontiguousarray(x)).to(self.dev) if x is not None else None
                for x in (w.packed, w.scales, w.zero_points)]
        out = [tuple(base)]
        for _ in range(copies - 1):
            out.append(tuple(None if x is None else x.clone() for x in base))
        return w, out

    def time_graph(self, record_calls, calls_per_replay, steps, warmup, sampler=None, pdl=True):
        """Captures `record_calls()` once into a graph; returns ms per replay."""
        torch, mnb = self.torch, self.mnb
        s = torch.cuda.Stream(device=self.dev)
        s.wait_stream(torch.cuda.current_stream())
        with torch.cuda.stream(s):
            record_calls()  # eager warm-up outside capture (same launches)
        torch.cuda.synchronize()
        g = torch.cuda.CUDAGraph()
        mnb.mnb_set_programmatic_launch(pdl)
        try:
            with torch.cuda.stream(s):
                with torch.cuda.graph(g, stream=s):
                    record_calls()
        finally:
            mnb.mnb_set_programmatic_launch(False)
        torch.cuda.current_stream().wait_stream(s)
        for _ in range(warmup):
            g.replay()
        torch.cuda.synchronize()
        barrier()
        # One event per replay boundary (no extra synchronisation): the bracketed total gives
        # the mean per replay, the per-replay differences its median.
        evs = [torch.cuda.Event(enable_timing=True) for _ in range(steps + 1)]
        if sampler:
            sampler.mark(True)
        evs[0].record()
        for i in range(steps):
            g.replay()
            evs[i + 1].record()
        torch.cuda.synchronize()
        if sampler:
            sampler.mark(False)
        barrier()
        self.launches += steps * calls_per_replay
        ms = evs[0].elapsed_time(evs[-1]) / steps
        self.last_median_ms = float(np.median([evs[i].elapsed_time(evs[i + 1]) for i in range(steps)]))
        return max_over_ranks(ms), g

    # -- the headline and friends ---------------------------------------------------
    def gemv(self, wl, steps, warmup, sampler, calls=CALLS_PER_STEP, copies=None):
        torch, mnb = self.torch, self.mnb
        ncopy = self.copies_for(weight_bytes(wl)) if copies is None else copies
        w, copies = self.upload_weights(wl, "B", ncopy)
        A = torch.from_numpy(syn.make_activation(wl).reshape(-1)).to(self.dev)
        Y = torch.empty(wl.N, dtype=torch.float16, device=self.dev)

        def rec():
            for i in range(calls):
                mnb.mnb_gemv(A, *copies[i % ncopy], wl.K, wl.N, wl.block_size, out=Y)

        ms, g = self.time_graph(rec, calls, steps, warmup, sampler)
        us = ms * 1e3 / calls
        # The graph holds raw pointers into `copies`, A and Y: keep them alive with it.
        return {"workload": wl.name, "us_per_call": us, "gbps": call_bytes(wl) / (us * 1e3),
                "us_per_call_median": self.last_median_ms * 1e3 / calls,
                "copies": ncopy, "calls_per_replay": calls, "ms_per_replay": ms,
                "variant": mnb.mnb_last_variant(), "graph": g, "A": A, "Y": Y, "w": w,
                "buffers": copies}

    def swiglu(self, wl, steps, warmup, sampler, calls=200):
        torch, mnb = self.torch, self.mnb
        ncopy = self.copies_for(2 * weight_bytes(wl))
        _, gates = self.upload_weights(wl, "gate", ncopy)
        _, ups = self.upload_weights(wl, "up", ncopy)
        A = torch.from_numpy(syn.make_activation(wl).reshape(-1)).to(self.dev)
        Y = torch.empty(wl.N, dtype=torch.float16, device=self.dev)

        def rec():
            for i in range(calls):
                mnb.mnb_gemv_gate_up_swiglu(A, gates[i % ncopy], ups[i % ncopy], wl.K, wl.N,
                                            wl.block_size, out=Y)

        ms, _ = self.time_graph(rec, calls, steps, warmup, sampler)
        us = ms * 1e3 / calls
        return {"workload": wl.name, "us_per_call": us, "gbps": call_bytes(wl, 2) / (us * 1e3),
                "copies": ncopy, "variant": mnb.mnb_last_variant()}

    def mlp_chain(self, steps, warmup, sampler, calls=100):
        """Decode MLP at M = 1: gate/up SwiGLU GEMV feeding the down GEMV, one graph segment."""
        torch, mnb = self.torch, self.mnb
        wg = syn.WORKLOADS["mlp_gate_up_k4096_n14336"]
        wd = syn.WORKLOADS["mlp_down_k14336_n4096"]
        per = 2 * weight_bytes(wg) + weight_bytes(wd)
        ncopy = self.copies_for(per)
        _, gates = self.upload_weights(wg, "gate", ncopy)
        _, ups = self.upload_weights(wg, "up", ncopy)
        _, downs = self.upload_weights(wd, "B", ncopy)
        x = torch.from_numpy(syn.make_activation(wg).reshape(-1)).to(self.dev)
        h = torch.empty(wg.N, dtype=torch.float16, device=self.dev)
        y = torch.empty(wd.N, dtype=torch.float16, device=self.dev)

        def rec():
            for i in range(calls):
                j = i % ncopy
                mnb.mnb_gemv_gate_up_swiglu(x, gates[j], ups[j], wg.K, wg.N, wg.block_size, out=h)
                mnb.mnb_gemv(h, *downs[j], wd.K, wd.N, wd.block_size, out=y)

        ms, _ = self.time_graph(rec, 2 * calls, steps, warmup, sampler)
        us = ms * 1e3 / calls
        nbytes = 2 * weight_bytes(wg) + weight_bytes(wd) + 2 * wg.K + 2 * wg.N + 2 * wd.N
        return {"workload": "mlp_chain_gate_up_k4096_n14336_down", "us_per_call": us,
                "gbps": nbytes / (us * 1e3), "copies": ncopy, "variant": "gate_up_swiglu + down gemv"}

    def act_order(self, wl, steps, warmup, sampler, calls=200, kind="act_order"):
        """M-row product of an act-order weight: the activation gather and the block kernel
        on the prepared weight, per call (two launches)."""
        torch, mnb = self.torch, self.mnb
        g_idx = syn.make_g_idx(wl, kind)
        kp, perm, bg = mnb.mnb_act_order_plan(g_idx, wl.K, wl.block_size)
        perm_d = torch.from_numpy(perm).to(self.dev)
        bg_d = torch.from_numpy(bg).to(self.dev)
        wlp = syn.custom(wl.name + "_prepared", wl.M, kp, wl.N, wl.block_size, wl.scales_dtype, wl.has_zp)
        ncopy = self.copies_for(weight_bytes(wlp))
        w, raw = self.upload_weights(wl, "B", 1)
        base = mnb.mnb_act_order_prepare(*raw[0], wl.K, wl.N, wl.block_size, perm_d, bg_d, kp)
        del raw
        copies = [base] + [tuple(None if x is None else x.clone() for x in base) for _ in range(ncopy - 1)]
        A = torch.from_numpy(syn.make_activation(wl)).to(self.dev)
        Y = torch.empty((wl.M, wl.N), dtype=torch.float16, device=self.dev)
        ws = torch.empty(mnb.mnb_act_order_workspace_bytes(wl.M, kp), dtype=torch.uint8, device=self.dev)

        def rec():
            for i in range(calls):
                mnb.mnb_gemm_act_order(A, *copies[i % ncopy], perm_d, wl.K, kp, wl.N, wl.block_size,
                                       workspace=ws, out=Y)

        # M = 1 (K' <= 8192): one launch per call, the GEMV gathers its own activations;
        # otherwise a gather pass and the block kernel.
        ms, _ = self.time_graph(rec, calls if wl.M == 1 else 2 * calls, steps, warmup, sampler)
        us = ms * 1e3 / calls
        variant = mnb.mnb_last_variant()
        return {"workload": f"{wl.name}_{kind}", "K_prepared": kp, "us_per_call": us,
                "gbps": call_bytes(wl) / (us * 1e3), "copies": ncopy,
                "variant": variant if variant.endswith("_gather") else "act_order_gather + " + variant}

    def gemm(self, wl, steps, warmup, sampler, calls, repacked: bool, shared_act: bool = False):
        """shared_act: one activation block for every call (a decode-time verify step reads the
        rows the previous op just wrote, so they sit in L2); otherwise each weight copy has its
        own activation copy and both come from HBM."""
        torch, mnb = self.torch, self.mnb
        per_copy = weight_bytes(wl) + (0 if shared_act else wl.M * wl.K * 2)
        ncopy = self.copies_for(per_copy)
        _, copies = self.upload_weights(wl, "B", ncopy)
        A0 = torch.from_numpy(syn.make_activation(wl)).to(self.dev)
        As = [A0] * ncopy if shared_act else [A0] + [A0.clone() for _ in range(ncopy - 1)]
        rps = [mnb.mnb_repack(c[0], wl.K, wl.N, wl.block_size) if repacked else None for c in copies]
        Y = torch.empty((wl.M, wl.N), dtype=torch.float16, device=self.dev)
        need = mnb.mnb_workspace_bytes(wl.M, wl.K, wl.N, wl.block_size)
        ws = torch.empty(max(need, 16), dtype=torch.uint8, device=self.dev) if need else None

        def rec():
            for i in range(calls):
                j = i % ncopy
                mnb.mnb_gemm(As[j], *copies[j], wl.K, wl.N, wl.block_size, repacked=rps[j],
                             workspace=ws, out=Y)

        ms, _ = self.time_graph(rec, calls, steps, warmup, sampler)
        us = ms * 1e3 / calls
        return {"workload": wl.name, "M": wl.M, "us_per_call": us,
                "gbps": call_bytes(wl) / (us * 1e3), "tflops": call_flops(wl) / (us * 1e6),
                "copies": ncopy, "activations": "shared (L2-resident)" if shared_act else "rotated with the weights",
                "variant": mnb.mnb_last_variant()}

    def gemm_f32(self, wl, steps, warmup, sampler, calls):
        """fp32 activations and output: the fp32 GEMV at M = 1, the split-activation
        kernels (split pass + GEMM, two launches) for M >= 2."""
        torch, mnb = self.torch, self.mnb
        per_copy = weight_bytes(wl) + wl.M * wl.K * 4
        ncopy = self.copies_for(per_copy)
        _, copies = self.upload_weights(wl, "B", ncopy)
        A0 = torch.from_numpy(syn.make_activation_f32(wl)).to(self.dev)
        As = [A0] + [A0.clone() for _ in range(ncopy - 1)]
        rps = [mnb.mnb_repack(c[0], wl.K, wl.N, wl.block_size) if wl.M > 8 else None for c in copies]
        Y = torch.empty((wl.M, wl.N), dtype=torch.float32, device=self.dev)
        need = mnb.mnb_workspace_bytes_f32(wl.M, wl.K, wl.N, wl.block_size)
        ws = torch.empty(max(need, 16), dtype=torch.uint8, device=self.dev)

        def rec():
            for i in range(calls):
                j = i % ncopy
                mnb.mnb_gemm_f32(As[j], *copies[j], wl.K, wl.N, wl.block_size, repacked=rps[j],
                                 workspace=ws, out=Y)

        launches = calls if wl.M == 1 else 2 * calls
        ms, _ = self.time_graph(rec, launches, steps, warmup, sampler)
        us = ms * 1e3 / calls
        nbytes = weight_bytes(wl) + 4 * wl.M * wl.K + 4 * wl.M * wl.N
        return {"workload": wl.name + "_f32act", "M": wl.M, "us_per_call": us, "gbps": nbytes / (us * 1e3),
                "tflops": call_flops(wl) / (us * 1e6), "copies": ncopy, "variant": mnb.mnb_last_variant()}

    def e2e_gemv(self, res, steps):
        """Host activations in, host result out, around the same graph of 1000 calls."""
        torch = self.torch
        A_host = res["A"].cpu().pin_memory()
        Y_host = torch.empty(res["Y"].shape, dtype=torch.float16).pin_memory()
        g = res["graph"]
        torch.cuda.synchronize()
        barrier()
        t0 = time.perf_counter()
        for _ in range(steps):
            res["A"].copy_(A_host, non_blocking=True)
            g.replay()
            Y_host.copy_(res["Y"], non_blocking=True)
            torch.cuda.current_stream().synchronize()
        dt = max_over_ranks(time.perf_counter() - t0)
        self.launches += steps * res["calls_per_replay"]
        us = dt * 1e6 / (steps * res["calls_per_replay"])
        wl = syn.WORKLOADS[res["workload"]]
        # One call as a caller makes it: A in, one mnb_gemv through the binding (no graph),
        # Y out, synchronised; host-to-host latency per call, median over the samples.
        mnb = self.mnb
        pk, sc, zp = res["buffers"][0]
        single = []
        for i in range(steps + 3):
            t1 = time.perf_counter()
            res["A"].copy_(A_host, non_blocking=True)
            mnb.mnb_gemv(res["A"], pk, sc, zp, wl.K, wl.N, wl.block_size, out=res["Y"])
            Y_host.copy_(res["Y"], non_blocking=True)
            torch.cuda.current_stream().synchronize()
            if i >= 3:
                single.append(time.perf_counter() - t1)
        self.launches += steps + 3
        us1 = float(np.median(single)) * 1e6
        return {"value": call_bytes(wl) / (us * 1e3), "unit": "GB/s", "us_per_call": us,
                "h2d_bytes_per_step": int(A_host.numel() * 2),
                "d2h_bytes_per_step": int(Y_host.numel() * 2),
                "note": "pinned host A -> device, one graph replay of the 1000 calls, device Y -> pinned host, "
                        "synchronised, per step",
                "single_call": {"us_host_to_host_median": us1, "samples": len(single),
                                "note": "one eager mnb_gemv per sample with its own 8 KB copy in and 8 KB copy "
                                        "out, synchronised: the per-call host latency (launch and copies "
                                        "included, nothing amortised)"}}


def log(msg: str):
    if int(os.environ.get("RANK", "0")) == 0:
        print(msg, file=sys.stderr, flush=True)


# ---------------------------------------------------------------------------------
# Distributed plumbing (replicas only: no data-path collective)
# ---------------------------------------------------------------------------------
_DIST = {"on": False}


def barrier():
    if _DIST["on"]:
        import torch.distributed as dist
        dist.barrier()


def max_over_ranks(x: float) -> float:
    if not _DIST["on"]:
        return x
    import torch
    import torch.distributed as dist
    t = torch.tensor([x], dtype=torch.float64, device=_DIST["device"])
    dist.all_reduce(t, op=dist.ReduceOp.MAX)
    return float(t.item())


# ---------------------------------------------------------------------------------
# CPU oracle timing (baseline leg and the reference arm)
# ---------------------------------------------------------------------------------
def oracle_sample(wl):
    """One call of the fp64 C++ oracle on the whole workload (every output column), split
    over the output columns on all CPUs this process may use."""
    from oracle import mnb_oracle as orc
    orc.lib()
    w = syn.make_weight(wl)
    A = syn.make_activation(wl)
    cores = orc.threads()

    def run():
        orc.matmul(A, w.packed, w.scales, w.zero_points, wl.K, wl.N, wl.block_size, nthreads=cores)

    return run, call_bytes(wl), cores


def cpu_baseline(budget_s: float = 12.0):
    wl = syn.WORKLOADS[HEADLINE]
    run, nbytes, cores = oracle_sample(wl)
    run()
    t0 = time.perf_counter()
    n = 0
    while True:
        run()
        n += 1
        if time.perf_counter() - t0 >= budget_s:
            break
    dt = time.perf_counter() - t0
    return {"value": n * nbytes / dt / 1e9, "unit": "GB/s", "cores": cores, "kind": "oracle",
            "host_cpus": os.cpu_count(),
            "sample": f"{HEADLINE}: all {wl.N} output columns per call, {n} calls in {dt:.1f} s "
                      f"(C++ fp64 oracle, output columns split over {cores} threads)",
            "us_per_call": dt / n * 1e6}


def run_reference(args):
    rank = int(os.environ.get("RANK", "0"))
    if rank != 0:
        return
    wl = syn.WORKLOADS[HEADLINE]
    run, nbytes, cores = oracle_sample(wl)
    for _ in range(args.warmup):
        run()
    t0 = time.perf_counter()
    for _ in range(args.steps):
        run()
    dt = time.perf_counter() - t0
    value = args.steps * nbytes / dt / 1e9
    line = {"impl": "reference", "metric": METRIC, "value": value, "unit": "GB/s", "n_gpus": args.gpus,
            "steps": args.steps, "warmup": args.warmup, "ms_per_step": dt * 1e3 / args.steps,
            "higher_is_better": True, "scaling": "weak", "vs_baseline": None, "dtype": "f64",
            "data": "synthetic (seeded SplitMix64)",
            "config": {"workload": HEADLINE, "M": 1, "K": wl.K, "N": wl.N, "block_size": wl.block_size,
                       "scales": wl.scales_dtype, "zero_points": wl.has_zp, "parallelism": "replicas"},
            "cpu_baseline": {"value": value, "unit": "GB/s", "cores": cores, "kind": "oracle",
                             "host_cpus": os.cpu_count(),
                             "sample": f"each step: one call of the C++ fp64 oracle on all {wl.N} output "
                                       f"columns, split over {cores} threads"},
            "e2e": {"value": value, "unit": "GB/s", "h2d_bytes_per_step": 0, "d2h_bytes_per_step": 0}}
    print(json.dumps(line))


def run_stream_control() -> str:
    """Compiles and runs the streaming-only control; returns its JSON line."""
    root = os.path.dirname(os.path.abspath(__file__))
    exe = os.path.join(root, "_build", "stream_control")
    os.makedirs(os.path.dirname(exe), exist_ok=True)
    src = os.path.join(root, "bench_stream_control.cu")
    subprocess.run(["nvcc", "-gencode", "arch=compute_103a,code=sm_103a", "-O3", "-std=c++17", "-I",
                    os.path.join(root, "gemm_mnb_gemv_gb300", "csrc"), src, "-o", exe], check=True)
    return subprocess.run([exe], check=True, capture_output=True, text=True).stdout.strip()


def run_single(db, name, steps, warmup):
    W = syn.WORKLOADS
    if name == "attn":
        return db.gemv(W[HEADLINE], steps, warmup, None)
    if name == "gate_up":
        return db.swiglu(W["mlp_gate_up_k4096_n14336"], steps, warmup, None)
    if name == "down":
        return db.gemv(W["mlp_down_k14336_n4096"], steps, warmup, None, calls=200)
    if name.startswith("verify_m"):
        rot = name.endswith("_rot")  # activations rotated with the weight copies
        base = name[:-4] if rot else name
        return db.gemm(W[f"{base}_k4096_n4096"], steps, warmup, None, calls=200, repacked=False,
                       shared_act=not rot)
    if name == "mlp_chain":
        return db.mlp_chain(steps, warmup, None)
    if name == "act_order_attn":
        return db.act_order(W[HEADLINE], steps, warmup, None)
    if name == "f32_attn":
        return db.gemm_f32(W[HEADLINE], steps, warmup, None, calls=200)
    if name == "f32_prefill":
        return db.gemm_f32(W["prefill_m2048_k4096_n14336"], steps, warmup, None, calls=5)
    if name == "prefill":
        return db.gemm(W["prefill_m2048_k4096_n14336"], steps, warmup, None, calls=9, repacked=True)
    raise SystemExit(f"unknown workload {name}")


# ---------------------------------------------------------------------------------
def secondary_lines(extras: dict) -> list:
    """One log line per secondary entry: timings, or the JSON of derived entries (ratios)."""
    out = []
    for k, v in extras.items():
        if "us_per_call" not in v:
            out.append(f"{k}: {json.dumps(v)}")
            continue
        out.append(f"{k}: {v['us_per_call']:.3f} us/call, {v.get('gbps', 0):.1f} GB/s, "
                   f"{v.get('tflops', 0):.1f} TFLOP/s ({v.get('variant', '?')})")
    return out


def annotate_secondary(extras: dict, hbm: float, tc: float, peak_src: str) -> dict:
    """Roofline of the prefill entry against the tensor peak, HBM fraction of the others
    (not of the labelled hot-L2 entry)."""
    pf = extras.get("prefill")
    if pf is not None:
        pf["roofline"] = {"bound": "tensor", "achieved": pf["tflops"], "peak": tc, "unit": "TFLOP/s",
                          "frac": pf["tflops"] / tc,
                          "peak_source": f"{peak_src} bf16_tflops (burst; fp16 rate equals bf16)"}
    for k, v in extras.items():
        if "gbps" in v and k not in ("prefill", "headline_hot_l2"):
            v["hbm_frac"] = v["gbps"] / hbm
    return extras


def main():
    ap = argparse.ArgumentParser()
    ap.add_argument("--gpus", type=int, default=1)
    ap.add_argument("--steps", type=int, default=300)
    ap.add_argument("--warmup", type=int, default=5)
    ap.add_argument("--impl", default="mnb", choices=["mnb", "reference"])
    ap.add_argument("--quick", action="store_true", help="headline only, short CPU baseline")
    ap.add_argument("--no-cpu-baseline", action="store_true")
    ap.add_argument("--clock-log", default=None,
                    help="keep the nvidia-smi clock samples of the timed regions in this CSV "
                         "(default: a temporary file; the JSON line carries their summary)")
    ap.add_argument("--workload", default=None,
                    help="time one workload only (attn, gate_up, down, verify_m2/4/8/16 [_rot: activations rotated "
                         "with the weights], prefill, mlp_chain, "
                         "act_order_attn, f32_attn, f32_prefill) "
                         "and print its record; for profiling")
    ap.add_argument("--stream-control", action="store_true",
                    help="build and run bench_stream_control.cu (the M = 1 GEMV's copy and launch structure with "
                         "no arithmetic) and print its record")
    args = ap.parse_args()
    if args.stream_control:
        print(run_stream_control())
        return
    if args.warmup < 3:
        ap.error("--warmup must be >= 3")
    if args.impl == "reference":
        run_reference(args)
        return

    import torch
    world = int(os.environ.get("WORLD_SIZE", "1"))
    rank = int(os.environ.get("RANK", "0"))
    local = int(os.environ.get("LOCAL_RANK", "0"))
    dev = torch.device(f"cuda:{local}")
    torch.cuda.set_device(dev)
    if world > 1:
        import torch.distributed as dist
        dist.init_process_group("nccl", device_id=dev)
        _DIST.update(on=True, device=dev)

    import __graft_entry__
    __graft_entry__.build()
    import gemm_mnb_gemv_gb300 as mnb

    peaks, peak_src = load_peaks()
    props = torch.cuda.get_device_properties(dev)
    l2 = getattr(props, "L2_cache_size", 126 * 1024 * 1024)
    clock_path = None
    if rank == 0:
        clock_path = args.clock_log or os.path.join(tempfile.gettempdir(), f"mnb_bench_clocks_{os.getpid()}.csv")
        if os.path.dirname(clock_path):
            os.makedirs(os.path.dirname(clock_path), exist_ok=True)
    sampler = ClockSampler(local, clock_path)
    db = DeviceBench(torch, mnb, dev, l2, rank)
    sampler.start()

    if args.workload:
        res = run_single(db, args.workload, args.steps, args.warmup)
        sampler.stop()
        if rank == 0:
            print(json.dumps({k: v for k, v in res.items() if k not in ("graph", "A", "Y", "w", "buffers")}))
        return

    wl = syn.WORKLOADS[HEADLINE]
    head = db.gemv(wl, args.steps, args.warmup, sampler)
    log(f"headline {head['us_per_call']:.3f} us/call {head['gbps']:.1f} GB/s ({head['variant']})")
    launches_headline = args.steps * CALLS_PER_STEP
    extras = {}
    if not args.quick:
        extras["gate_up_swiglu"] = db.swiglu(syn.WORKLOADS["mlp_gate_up_k4096_n14336"], 20, 3, sampler)
        d = db.gemv(syn.WORKLOADS["mlp_down_k14336_n4096"], 20, 3, sampler, calls=200)
        extras["down_gemv"] = {k: v for k, v in d.items() if k not in ("graph", "A", "Y", "w", "buffers")}
        del d
        for M in (2, 4, 8, 16):
            extras[f"verify_m{M}"] = db.gemm(syn.WORKLOADS[f"verify_m{M}_k4096_n4096"], 20, 3, sampler,
                                             calls=200, repacked=False, shared_act=True)
        # latency against M (same K, N and storage as the verify shapes except bs 32 at M = 1):
        # the pages' concern is a cliff from M = 1 to M = 2
        extras["verify_over_m1"] = {f"M{M}": extras[f"verify_m{M}"]["us_per_call"] / head["us_per_call"]
                                    for M in (2, 4, 8, 16)}
        # mid-size M on the tensor-core kernel (verify storage): few output tiles, K split
        extras["mid_m64"] = db.gemm(syn.custom("mid_m64_k4096_n4096", 64, 4096, 4096, 64), 20, 3, sampler,
                                    calls=100, repacked=True, shared_act=True)
        extras["prefill"] = db.gemm(syn.WORKLOADS["prefill_m2048_k4096_n14336"], 10, 3, sampler,
                                    calls=9, repacked=True)
        extras["mlp_chain"] = db.mlp_chain(10, 3, sampler)
        hot = db.gemv(wl, 20, 3, sampler, copies=1)
        extras["headline_hot_l2"] = {k: v for k, v in hot.items() if k not in ("graph", "A", "Y", "w", "buffers")}
        extras["headline_hot_l2"]["label"] = ("hot: one weight copy, resident in L2 across calls (not an HBM "
                                              "number; the headline rotates copies)")
        del hot
        extras["act_order_attn"] = db.act_order(wl, 20, 3, sampler)
        extras["f32_attn"] = db.gemm_f32(wl, 20, 3, sampler, calls=200)
        extras["f32_prefill"] = db.gemm_f32(syn.WORKLOADS["prefill_m2048_k4096_n14336"], 5, 3, sampler, calls=5)
    for msg in secondary_lines(extras):
        log(msg)
    clocks = sampler.stop()
    e2e = db.e2e_gemv(head, max(3, args.steps // 10))

    gbps_total = head["gbps"] * world
    hbm = float(peaks["hbm_gbs"])
    gemv_files = ["gemm_mnb_gemv_gb300/csrc/gemv_mma.cu", "gemm_mnb_gemv_gb300/csrc/mma_sync.cuh",
                  "gemm_mnb_gemv_gb300/csrc/mnb_device.cuh", "gemm_mnb_gemv_gb300/csrc/tcgen05.cuh"]
    roof = {"bound": "hbm", "achieved": head["gbps"], "peak": hbm, "unit": "GB/s",
            "frac": head["gbps"] / hbm, "traffic": profiled_traffic("gemv_attnproj", gemv_files),
            "algorithmic_bytes_per_launch": call_bytes(wl), "kernel": head["variant"],
            "peak_source": f"{peak_src} hbm_gbs (copy bandwidth)"}
    line = {"metric": METRIC, "value": gbps_total, "unit": "GB/s", "n_gpus": world, "steps": args.steps,
            "warmup": args.warmup, "ms_per_step": head["ms_per_replay"], "higher_is_better": True,
            "scaling": "weak", "vs_baseline": None, "dtype": "f16",
            "data": "synthetic (seeded SplitMix64 per tensor; fp16 A ~N(0,1) clipped to +-4)",
            "config": {"workload": HEADLINE, "M": 1, "K": wl.K, "N": wl.N, "block_size": wl.block_size,
                       "scales": wl.scales_dtype, "zero_points": wl.has_zp,
                       "calls_per_step": CALLS_PER_STEP, "launch": "CUDA graph, programmatic dependent launch",
                       "l2": f"inputs larger than L2: {head['copies']} weight copies rotated "
                             f"({head['copies'] * weight_bytes(wl) / 1e6:.0f} MB > 3 x {l2 / 1e6:.0f} MB L2); "
                             "one 8 KB activation vector shared by all calls",
                       "parallelism": f"replicas x{world}"},
            "us_per_call": head["us_per_call"], "us_per_call_median": head["us_per_call_median"],
            "roofline": roof, "clocks": clocks, "e2e": e2e,
            "gpu_launches": launches_headline}
    if extras:
        tc = float(peaks.get("bf16_tflops", FALLBACK_PEAKS["bf16_tflops"]))
        line["secondary"] = annotate_secondary(extras, hbm, tc, peak_src)
    if rank == 0 and not args.no_cpu_baseline:
        line["cpu_baseline"] = cpu_baseline(4.0 if args.quick else 12.0)
    if rank == 0:
        print(json.dumps(line))
    if _DIST["on"]:
        import torch.distributed as dist
        dist.destroy_process_group()


if __name__ == "__main__":
    main()
