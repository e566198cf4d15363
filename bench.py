#!/usr/bin/env python3
"""Benchmark of the W4A16 routed mixture-of-experts layer on GB300.

One step = one pass of the whole layer over one batch: token-to-expert
alignment with the activation gather, grouped gate_up GEMM with the gated
activation, grouped down GEMM, fixed-order combine (four launches of
libw4moe.so on one stream, each a programmatic dependent of the one before).  The
workload is one 256-token canvas at the pages' layer shape: M=256, d=2816,
m=704, E=128, top-8, uint4 weights with fp16 scale/zero (groups of 128 for
gate_up, 64 for down), bf16 activations; inputs are seeded synthetic tensors
(the pages' synthetic one-layer microbenchmark: "Inference: Making every
denoising pass fast" -- The final best W4 MoE kernel).

value = algorithmic bytes per step / device time per step (GB/s):
  bytes = packed weights + fp16 scales/zeros of the experts the batch touches
          + x read (M*d*2) + out write (M*d*2) + ids and weights (M*k*8).
The timed region is K back-to-back steps between one pair of CUDA events, with
no L2 flush: each step streams all packed weights (415 MB at layer256), more
than the 126 MB L2, so no step finds the previous one's weights cached.  --impl reference times the float64 CPU oracle on the host cores on a
bounded sample of the same workload, in the same unit.

Prints one JSON line (rank 0).  Multi-GPU runs (torchrun) are independent
replicas of the same layer, one per GPU, with no collective on the data path.

--workload sampler times the per-step sampler beside the layer instead: one
pass over [256, 262144] fp32 vocabulary logits giving the entropy, a
Gumbel-max sample and the argmax per row ("dg-w4-kernels" -- Sampler);
value = logits bytes / device time.  --workload rmsnorm times fused_rmsnorm
over [256, 2816] bf16 ("dg-w4-kernels" -- RMSNorm); value = (x + weight + y)
bytes / device time.  --workload linear times the dense W4A16 linear
("dg-w4-kernels" -- W4A16; "Inference: Making every denoising pass fast" --
Dense W4 everywhere: 256-row QKV and LM-head-tile tests against cuBLAS BF16),
value = TFLOP/s of the QKV shape, with torch's bf16 F.linear (cuBLAS) on the
same shapes timed alongside.
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

import numpy as np

ROOT = os.path.dirname(os.path.abspath(__file__))
sys.path.insert(0, ROOT)

METRIC = "W4A16 MoE layer µs & HBM GB/s (% GB300 roofline) at M=256,d2816,m704,E128,top8"
METRIC_SAMPLER = ("one-pass logits sampler (entropy + Gumbel-max sample + argmax) µs & HBM GB/s "
                  "at [256, 262144] fp32")
METRIC_RMSNORM = "fused RMSNorm µs & HBM GB/s at [256, 2816] bf16"
METRIC_LINEAR = ("dense W4A16 linear µs & TFLOP/s at 256 rows (QKV 2816->4096, LM-head tile "
                 "2816->16384) vs cuBLAS BF16")
FALLBACK_HBM_GBS = 6800.0


# ----------------------------------------------------------------------------
# helpers
# ----------------------------------------------------------------------------
def per_expert_bytes(d, m, gu_group=128, dn_group=64):
    gu = 2 * m * d // 2 + 2 * (2 * m * (d // gu_group) * 2)
    dn = d * m // 2 + 2 * (d * (m // dn_group) * 2)
    return gu, dn


def layer_alg_bytes(M, d, m, k, touched):
    gu, dn = per_expert_bytes(d, m)
    return touched * (gu + dn) + M * d * 2 + M * d * 2 + M * k * 8


def gate_up_alg_bytes(M, d, m, touched):
    gu, _ = per_expert_bytes(d, m)
    return touched * gu + M * d * 2


def measured_peaks():
    path = os.path.join(ROOT, "MEASURED_PEAKS.json")
    try:
        with open(path) as f:
            p = json.load(f)
        return float(p["hbm_gbs"]), "measured"
    except Exception:
        return FALLBACK_HBM_GBS, "fallback"


def bf16_peak():
    """Measured dense bf16 tensor throughput (TFLOP/s), burst."""
    try:
        with open(os.path.join(ROOT, "MEASURED_PEAKS.json")) as f:
            return float(json.load(f)["bf16_tflops"]), "measured"
    except Exception:
        return 1900.0, "fallback"


def kernel_source_hash():
    h = hashlib.sha256()
    for f in ("grouped_gemm.cu", "ptx.cuh"):
        with open(os.path.join(ROOT, "w4a16_moe_expert_sync_gb300", "csrc", f), "rb") as fh:
            h.update(fh.read())
    return h.hexdigest()[:16]


def recorded_traffic(kernel, workload):
    """DRAM bytes per launch from the committed ncu summary, if it was taken on
    the kernel source as it is now; else None."""
    path = os.path.join(ROOT, "profiles", "dram_traffic.json")
    try:
        with open(path) as f:
            rec = json.load(f)
        e = rec[kernel][workload]
        if e.get("source_sha") == kernel_source_hash():
            return float(e["dram_bytes_per_launch"])
    except Exception:
        pass
    return None


class ClockSampler:
    """nvidia-smi clocks and throttle reasons, sampled while the timed region runs."""
    FIELDS = ("index,clocks.sm,clocks.max.sm,power.draw,clocks_event_reasons.active,"
              "clocks_event_reasons.hw_slowdown,clocks_event_reasons.hw_thermal_slowdown,"
              "clocks_event_reasons.sw_thermal_slowdown,clocks_event_reasons.sw_power_cap")
    REASONS = ("hw_slowdown", "hw_thermal_slowdown", "sw_thermal_slowdown", "sw_power_cap")

    def __init__(self, gpu_id: str, interval_ms: int = 20):
        self.cmd = ["nvidia-smi", f"--query-gpu={self.FIELDS}", "--format=csv,noheader,nounits",
                    "-lms", str(interval_ms), "-i", gpu_id]
        self.proc = None

    def __enter__(self):
        try:
            self.proc = subprocess.Popen(self.cmd, stdout=subprocess.PIPE,
                                         stderr=subprocess.DEVNULL, text=True)
            time.sleep(0.3)      # let the first sample land before the timed region
        except Exception:
            self.proc = None
        return self

    def __exit__(self, *exc):
        self.lines = []
        if self.proc is not None:
            time.sleep(0.05)
            self.proc.terminate()
            try:
                out, _ = self.proc.communicate(timeout=5)
            except Exception:
                self.proc.kill()
                out = ""
            self.lines = [l for l in out.splitlines() if l.strip()]
        return False

    def summary(self):
        sm, mx, reasons, power = [], None, set(), []
        for line in getattr(self, "lines", []):
            parts = [p.strip() for p in line.split(",")]
            if len(parts) < 9:
                continue
            try:
                sm.append(float(parts[1]))
                mx = float(parts[2])
                power.append(float(parts[3]))
            except ValueError:
                continue
            for name, flag in zip(self.REASONS, parts[5:9]):
                if flag.lower().startswith("active"):
                    reasons.add(name)
        if not sm:
            return {"sm_mhz": None, "sm_max_mhz": None, "reasons": [], "samples": 0}
        return {"sm_mhz": statistics.median(sm), "sm_max_mhz": mx, "reasons": sorted(reasons),
                "samples": len(sm), "power_w_max": max(power) if power else None}


def gpu_smi_id(dev):
    import torch
    p = torch.cuda.get_device_properties(dev)
    try:
        return f"{p.pci_domain_id:08X}:{p.pci_bus_id:02X}:{p.pci_device_id:02X}.0"
    except Exception:
        return str(dev)


# ----------------------------------------------------------------------------
# distributed plumbing (replicas; barrier + max over ranks only)
# ----------------------------------------------------------------------------
def dist_setup(n_gpus):
    world = int(os.environ.get("WORLD_SIZE", "1"))
    rank = int(os.environ.get("RANK", "0"))
    local = int(os.environ.get("LOCAL_RANK", "0"))
    if world > 1:
        import torch.distributed as dist
        backend = "nccl"
        try:
            import torch
            if not torch.cuda.is_available():
                backend = "gloo"
        except Exception:
            backend = "gloo"
        dist.init_process_group(backend=backend)
    return world, rank, local


def barrier(world):
    if world > 1:
        import torch.distributed as dist
        dist.barrier()


def max_over_ranks(world, value, device=None):
    if world == 1:
        return value
    import torch
    import torch.distributed as dist
    t = torch.tensor([value], dtype=torch.float64, device=device)
    dist.all_reduce(t, op=dist.ReduceOp.MAX)
    return float(t.item())


# ----------------------------------------------------------------------------
# CPU oracle timing (cpu_baseline leg and the reference arm)
# ----------------------------------------------------------------------------
def oracle_sample_setup(cfg, experts=None):
    """Oracle-side inputs: its own routing and its own quantisation of the
    experts a sample needs (untimed preparation)."""
    import oracle
    from w4a16_moe_expert_sync_gb300 import workloads as wl
    x_bits = wl.activations(cfg)
    ids, w = oracle.route(wl.router_logits(cfg), cfg.k)
    if experts is None:
        experts = range(cfg.E)
    gu_q = np.zeros((cfg.E, 2 * cfg.m, cfg.d // 2), np.uint8)
    gu_s = np.zeros((cfg.E, 2 * cfg.m, cfg.d // cfg.gu_group), np.uint16)
    gu_z = np.zeros_like(gu_s)
    dn_q = np.zeros((cfg.E, cfg.d, cfg.m // 2), np.uint8)
    dn_s = np.zeros((cfg.E, cfg.d, cfg.m // cfg.dn_group), np.uint16)
    dn_z = np.zeros_like(dn_s)
    for e in sorted(set(int(v) for v in experts)):
        gu_q[e], gu_s[e], gu_z[e] = oracle.quantize_w4(wl.gate_up_weight(cfg, e), cfg.gu_group)
        dn_q[e], dn_s[e], dn_z[e] = oracle.quantize_w4(wl.down_weight(cfg, e), cfg.dn_group)
    return x_bits, ids, w, (gu_q, gu_s, gu_z), (dn_q, dn_s, dn_z)


def time_oracle_assignments(cfg, assign, setup, nthreads):
    """Oracle layer on a list of flat assignments a = t*k + j, each run as its
    own one-expert row (x_t, expert ids[a], weight w[a]).  Returns
    (seconds, algorithmic bytes of that sample)."""
    import oracle
    x_bits, ids, w, gu, dn = setup
    t = assign // cfg.k
    e = ids.ravel()[assign]
    wt = w.ravel()[assign]
    t0 = time.perf_counter()
    oracle.moe_layer(x_bits[t], gu, dn, e[:, None].astype(np.int32),
                     wt[:, None].astype(np.float32), nthreads=nthreads)
    dt = time.perf_counter() - t0
    touched = len(set(int(v) for v in e))
    gu_b, dn_b = per_expert_bytes(cfg.d, cfg.m)
    nbytes = touched * (gu_b + dn_b) + len(assign) * (cfg.d * 4 + 8)
    return dt, nbytes


def cpu_baseline(cfg, n_tokens):
    """The oracle on n_tokens evenly spaced tokens of the workload (all k
    experts each), on every host core; GB/s of that sample's algorithmic bytes."""
    import oracle
    from w4a16_moe_expert_sync_gb300 import workloads as wl
    nthreads = os.cpu_count() or 1
    tokens = np.linspace(0, cfg.M - 1, n_tokens).round().astype(int)
    ids, _ = oracle.route(wl.router_logits(cfg), cfg.k)
    x_bits, ids, w, gu, dn = oracle_sample_setup(cfg, ids[tokens].ravel())
    t0 = time.perf_counter()
    oracle.moe_layer(x_bits[tokens], gu, dn, ids[tokens], w[tokens], nthreads=nthreads)
    dt = time.perf_counter() - t0
    touched = len(set(int(v) for v in ids[tokens].ravel()))
    nbytes = layer_alg_bytes(len(tokens), cfg.d, cfg.m, cfg.k, touched)
    # the same oracle on one thread, two tokens (the per-token cost is the same
    # work, so seconds per layer scale by tokens)
    t1 = time.perf_counter()
    oracle.moe_layer(x_bits[tokens[:2]], gu, dn, ids[tokens[:2]], w[tokens[:2]], nthreads=1)
    dt1 = time.perf_counter() - t1
    return {"value": nbytes / dt / 1e9, "unit": "GB/s", "cores": nthreads, "kind": "oracle",
            "sample": f"{n_tokens} of {cfg.M} tokens of the {cfg.name} workload (all {cfg.k} "
                      f"experts each, {n_tokens * cfg.k} assignments, {touched} experts), "
                      f"float64 C oracle on {nthreads} threads, {dt:.2f} s wall",
            "s_per_layer": {"all_cores": dt / len(tokens) * cfg.M,
                            "one_thread": dt1 / 2 * cfg.M,
                            "note": f"extrapolated from the samples to all {cfg.M} tokens"}}


def run_reference(args, cfg, world, rank):
    """The reference arm: the float64 oracle, as it stands, on the host cores."""
    if rank != 0:
        return
    nthreads = os.cpu_count() or 1
    steps, warm = args.steps, args.warmup
    setup = oracle_sample_setup(cfg)
    A = cfg.M * cfg.k
    # one step = `per` assignments (one per core), rotating through the
    # canvas's M*k assignments
    per = max(1, min(nthreads, A))
    times, nbytes = [], []
    for i in range(warm + steps):
        assign = (np.arange(per) + i * per) % A
        dt, nb = time_oracle_assignments(cfg, assign, setup, nthreads)
        if i >= warm:
            times.append(dt)
            nbytes.append(nb)
    total_t, total_b = sum(times), sum(nbytes)
    value = total_b / total_t / 1e9
    sample = (f"{per} (token, expert) assignments per step of the {cfg.name} workload, "
              f"rotating over its {A} assignments; float64 C oracle on {nthreads} threads")
    line = {
        "impl": "reference", "metric": METRIC, "value": value, "unit": "GB/s",
        "n_gpus": world, "steps": steps, "warmup": warm,
        "ms_per_step": 1e3 * total_t / steps, "higher_is_better": True, "scaling": "weak",
        "vs_baseline": None, "dtype": "f64", "data": "synthetic",
        "config": config_dict(cfg, args),
        "cpu_baseline": {"value": value, "unit": "GB/s", "cores": nthreads, "kind": "oracle",
                         "sample": sample},
        "e2e": {"value": value, "unit": "GB/s", "h2d_bytes_per_step": 0,
                "d2h_bytes_per_step": 0},
    }
    print(json.dumps(line), flush=True)


def config_dict(cfg, args):
    return {"workload": f"{cfg.name}: W4A16 routed-MoE layer M={cfg.M} d={cfg.d} m={cfg.m} "
                        f"E={cfg.E} top-{cfg.k}, uint4 weights with fp16 scale/zero "
                        f"(g{cfg.gu_group} gate_up, g{cfg.dn_group} down), bf16 activations, "
                        f"seed {cfg.seed}",
            "M": cfg.M, "d": cfg.d, "m": cfg.m, "E": cfg.E, "k": cfg.k,
            "block_m": args.block_m, "routing": cfg.routing,
            "l2": "not flushed: inputs larger than L2 (each step streams all packed weights, "
                  "415 MB at layer256, through the 126 MB L2)",
            "parallelism": "replicas"}


# ----------------------------------------------------------------------------
# the GPU arm
# ----------------------------------------------------------------------------
def prepare_gpu(cfg, dev):
    import torch
    import w4a16_moe_expert_sync_gb300 as w4
    from w4a16_moe_expert_sync_gb300 import workloads as wl
    x = torch.from_numpy(wl.activations(cfg).view(np.int16)).to(dev).view(torch.bfloat16)
    logits = torch.from_numpy(wl.router_logits(cfg)).to(dev)
    gu = (torch.empty((cfg.E, 2 * cfg.m, cfg.d // 2), dtype=torch.uint8, device=dev),
          torch.empty((cfg.E, 2 * cfg.m, cfg.d // cfg.gu_group), dtype=torch.float16, device=dev),
          torch.empty((cfg.E, 2 * cfg.m, cfg.d // cfg.gu_group), dtype=torch.float16, device=dev))
    dn = (torch.empty((cfg.E, cfg.d, cfg.m // 2), dtype=torch.uint8, device=dev),
          torch.empty((cfg.E, cfg.d, cfg.m // cfg.dn_group), dtype=torch.float16, device=dev),
          torch.empty((cfg.E, cfg.d, cfg.m // cfg.dn_group), dtype=torch.float16, device=dev))
    for e in range(cfg.E):
        w4.w4_quantize(torch.from_numpy(wl.gate_up_weight(cfg, e)).to(dev), cfg.gu_group,
                       out=tuple(t[e:e + 1] for t in gu))
        w4.w4_quantize(torch.from_numpy(wl.down_weight(cfg, e)).to(dev), cfg.dn_group,
                       out=tuple(t[e:e + 1] for t in dn))
    ids, w = w4.w4_moe_route(logits, cfg.k)
    torch.cuda.synchronize()
    return x, ids, w, gu, dn


SWEEP_CONFIGS = ("sweep_M1", "sweep_M8", "sweep_M32", "sweep_M64", "sweep_M128", "sweep_M256",
                 "zipf256", "canvas2048")


def time_configs(args, gu, dn, dev, status):
    """The layer across the survey's other configurations (the M sweep, Zipf
    routing, the 2048-token canvas), compactly: each config's own activations
    and routing (its seed) with the packed weights already on the device
    (same shapes; the time does not depend on the weight values).  Per
    config: back-to-back w4_moe_layer calls between one pair of events, then a
    serialised pass for the two GEMMs."""
    import torch
    import w4a16_moe_expert_sync_gb300 as w4
    from w4a16_moe_expert_sync_gb300 import workloads as wl
    peak, _ = measured_peaks()
    tpeak = bf16_peak()[0]
    res = {}
    for name in SWEEP_CONFIGS:
        c = wl.CONFIGS[name]
        x = torch.from_numpy(wl.activations(c).view(np.int16)).to(dev).view(torch.bfloat16)
        ids, w = w4.w4_moe_route(torch.from_numpy(wl.router_logits(c)).to(dev), c.k)
        touched = int(torch.unique(ids).numel())
        ws = torch.empty(w4.w4_moe_layer_workspace_size(c.M, c.d, c.m, c.E, c.k, args.block_m),
                         dtype=torch.uint8, device=dev)
        out = torch.empty((c.M, c.d), dtype=torch.bfloat16, device=dev)
        steps = 50 if c.M <= 256 else 20

        def layer():
            w4.w4_moe_layer(x, ids, w, gu, dn, block_m=args.block_m, workspace=ws, out=out,
                            dev_status=status)

        for _ in range(3):
            layer()
        a, b = torch.cuda.Event(enable_timing=True), torch.cuda.Event(enable_timing=True)
        torch.cuda.synchronize()
        a.record()
        for _ in range(steps):
            layer()
        b.record()
        torch.cuda.synchronize()
        ms = a.elapsed_time(b) / steps
        al, xg = w4.w4_moe_align_gather(ids, x, c.E, args.block_m, dev_status=status)
        h = w4.w4_grouped_gemm_gate_up(xg, *gu, al, dev_status=status)
        y = w4.w4_grouped_gemm_down(h, *dn, al, dev_status=status)
        ev = [torch.cuda.Event(enable_timing=True) for _ in range(3)]
        gsum = [0.0, 0.0]
        for i in range(12):
            ev[0].record()
            w4.w4_grouped_gemm_gate_up(xg, *gu, al, h=h, dev_status=status)
            ev[1].record()
            w4.w4_grouped_gemm_down(h, *dn, al, y=y, dev_status=status)
            ev[2].record()
            torch.cuda.synchronize()
            if i >= 2:
                gsum[0] += ev[0].elapsed_time(ev[1]) / 10
                gsum[1] += ev[1].elapsed_time(ev[2]) / 10
        nbytes = layer_alg_bytes(c.M, c.d, c.m, c.k, touched)
        flops = c.M * c.k * 2.0 * 3 * c.m * c.d
        res[name] = {"M": c.M, "routing": c.routing, "touched_experts": touched,
                     "us_per_layer": ms * 1e3,
                     "frac_hbm": nbytes / (ms * 1e-3) / 1e9 / peak,
                     "frac_tensor": flops / (ms * 1e-3) / 1e12 / tpeak,
                     "gate_up_us": gsum[0] * 1e3, "down_us": gsum[1] * 1e3}
    if int(status.item()) != 0:
        raise RuntimeError(f"device status {int(status.item()):#x} in the config sweep")
    return res


def run_gpu(args, cfg, world, rank, local):
    import torch
    import w4a16_moe_expert_sync_gb300 as w4
    w4.load_library()
    dev = torch.device("cuda", local)
    torch.cuda.set_device(dev)
    x, ids, w, gu, dn = prepare_gpu(cfg, dev)
    touched = int(torch.unique(ids).numel())
    nbytes = layer_alg_bytes(cfg.M, cfg.d, cfg.m, cfg.k, touched)
    gu_bytes = gate_up_alg_bytes(cfg.M, cfg.d, cfg.m, touched)

    bm = args.block_m
    status = torch.zeros(1, dtype=torch.int32, device=dev)
    al, xg = w4.w4_moe_align_gather(ids, x, cfg.E, bm, dev_status=status)
    h = w4.w4_grouped_gemm_gate_up(xg, *gu, al, dev_status=status)
    y = torch.empty((cfg.M * cfg.k, cfg.d), dtype=torch.float32, device=dev)
    out = torch.empty((cfg.M, cfg.d), dtype=torch.bfloat16, device=dev)
    ws = torch.empty(w4.w4_moe_layer_workspace_size(cfg.M, cfg.d, cfg.m, cfg.E, cfg.k, bm),
                     dtype=torch.uint8, device=dev)

    # one step = one w4_moe_layer call: its four launches (align+gather,
    # gate_up, down, combine) go out back to back on one stream, each a
    # programmatic dependent of the one before
    def layer():
        w4.w4_moe_layer(x, ids, w, gu, dn, block_m=bm, workspace=ws, out=out, dev_status=status)

    for _ in range(args.warmup):
        layer()
    torch.cuda.synchronize()
    if int(status.item()) != 0:
        raise RuntimeError(f"device status {int(status.item()):#x} during warm-up")

    # timed region: K back-to-back layers between one pair of events.  No L2
    # flush: every step streams all packed weights (415 MB at layer256), more
    # than the 126 MB L2, so no step finds the previous one's weights cached.
    t_start, t_end = torch.cuda.Event(enable_timing=True), torch.cuda.Event(enable_timing=True)
    sampler = ClockSampler(gpu_smi_id(local)) if not args.skip_clocks else None
    barrier(world)
    torch.cuda.synchronize()
    if sampler:
        sampler.__enter__()
    t_wall = time.perf_counter()
    t_start.record()
    for _ in range(args.steps):
        layer()
    t_end.record()
    torch.cuda.synchronize()
    t_wall = time.perf_counter() - t_wall
    if sampler:
        sampler.__exit__(None, None, None)
    barrier(world)
    if int(status.item()) != 0:
        raise RuntimeError(f"device status {int(status.item()):#x} in the timed region")
    mean_ms = t_start.elapsed_time(t_end) / args.steps
    mean_ms_all = max_over_ranks(world, mean_ms, dev)
    value = world * nbytes / (mean_ms_all * 1e-3) / 1e9

    # per-kernel times: the same launches through the binding's entry
    # points of the same names, events between them (which serialises the
    # launches: no overlap of one kernel's start with the previous one's end)
    def step_split(ev):
        ev[0].record()
        w4.w4_moe_align_gather(ids, x, cfg.E, bm, dev_status=status, out=al, xg=xg)
        ev[1].record()
        w4.w4_grouped_gemm_gate_up(xg, *gu, al, h=h, dev_status=status)
        ev[2].record()
        w4.w4_grouped_gemm_down(h, *dn, al, y=y, dev_status=status)
        ev[3].record()
        w4.w4_moe_combine_fixed_order(y, ids, w, cfg.E, out=out)
        ev[4].record()

    n_split = max(3, min(args.steps, 300))
    evs = [[torch.cuda.Event(enable_timing=True) for _ in range(5)] for _ in range(n_split + 3)]
    for i in range(n_split + 3):
        step_split(evs[i])
    torch.cuda.synchronize()
    evs = evs[3:]
    per_kernel = {name: [e[i].elapsed_time(e[i + 1]) for e in evs]
                  for i, name in enumerate(("align_gather", "gate_up", "down", "combine"))}
    serial_ms = statistics.fmean(e[0].elapsed_time(e[4]) for e in evs)

    # ---------------------------------------------------------------- e2e
    e2e = None
    if not args.skip_e2e:
        # The step from host memory through the host-buffer entry point
        # (w4_moe_layer_host: x, ids and weights copied in, out copied back,
        # all on the call's stream).  Two streams with their own workspaces
        # and output buffers take the steps in turn, so one step's copies
        # overlap the other's kernels; the timed region runs from the first
        # copy in to the last copy out, K steps.
        x_h = x.cpu().pin_memory()
        ids_h = ids.cpu().pin_memory()
        w_h = w.cpu().pin_memory()
        need = w4.w4_moe_layer_host_workspace_size(cfg.M, cfg.d, cfg.m, cfg.E, cfg.k, bm)
        lanes = [(torch.cuda.Stream(device=dev),
                  torch.empty(need, dtype=torch.uint8, device=dev),
                  torch.empty((cfg.M, cfg.d), dtype=torch.bfloat16).pin_memory())
                 for _ in range(2)]

        def e2e_steps(n):
            cur = torch.cuda.current_stream()
            for st, _, _ in lanes:
                st.wait_stream(cur)
            for i in range(n):
                st, ws_i, out_i = lanes[i % 2]
                w4.w4_moe_layer_host(x_h, ids_h, w_h, gu, dn, out_i, ws_i, block_m=bm,
                                     dev_status=status, stream=st)
            for st, _, _ in lanes:
                cur.wait_stream(st)

        e2e_steps(max(args.warmup, 2))
        torch.cuda.synchronize()
        e_start, e_end = torch.cuda.Event(enable_timing=True), torch.cuda.Event(enable_timing=True)
        barrier(world)
        torch.cuda.synchronize()
        e_start.record()
        e2e_steps(args.steps)
        e_end.record()
        torch.cuda.synchronize()
        barrier(world)
        e2e_ms = max_over_ranks(world, e_start.elapsed_time(e_end) / args.steps, dev)
        h2d = x.numel() * 2 + ids.numel() * 4 + w.numel() * 4
        d2h = out.numel() * 2
        e2e = {"value": world * nbytes / (e2e_ms * 1e-3) / 1e9, "unit": "GB/s",
               "h2d_bytes_per_step": h2d, "d2h_bytes_per_step": d2h,
               "ms_per_step": e2e_ms,
               "api": "w4_moe_layer_host (one C-ABI call per step: x, ids and weights copied "
                      "from page-locked host memory, align+gather, gate_up, down, combine, out "
                      "copied back), two streams taking the steps in turn"}
        ref_out = out.cpu()
        for _, _, out_i in lanes:
            if not torch.equal(out_i.view(torch.int16), ref_out.view(torch.int16)):
                raise RuntimeError("e2e output copy mismatch")

    # ------------------------------------------------------------ roofline
    peak, peak_kind = measured_peaks()
    gu_ms = statistics.fmean(per_kernel["gate_up"])
    achieved = gu_bytes / (gu_ms * 1e-3) / 1e9
    roofline = {"bound": "hbm", "achieved": achieved, "peak": peak, "unit": "GB/s",
                "frac": achieved / peak, "traffic": recorded_traffic("gate_up", cfg.name),
                "kernel": "grouped_gemm_kernel<gate_up> (w4_grouped_gemm_gate_up)",
                "alg_bytes_per_launch": gu_bytes,
                "peak_source": f"{peak_kind} (MEASURED_PEAKS.json hbm_gbs: STREAM-style copy)"
                if peak_kind == "measured" else "fallback 6.8 TB/s"}

    line = {
        "metric": METRIC, "value": value, "unit": "GB/s", "n_gpus": world,
        "steps": args.steps, "warmup": args.warmup, "ms_per_step": mean_ms_all,
        "higher_is_better": True, "scaling": "weak", "vs_baseline": None,
        "dtype": "fp16", "data": "synthetic", "config": config_dict(cfg, args),
        "us_per_layer": mean_ms_all * 1e3,
        "us_per_layer_serialised": serial_ms * 1e3,
        "layer_frac_of_hbm_peak": value / world / peak,
        # the layer's dense-contraction work, A * 2 * (2 m d + d m) FLOP, against
        # the measured bf16 tensor peak (the 2048-token canvas is compute-bound)
        "layer_tflops": cfg.M * cfg.k * 2.0 * 3 * cfg.m * cfg.d / (mean_ms_all * 1e-3) / 1e12,
        "layer_frac_of_tensor_peak": (cfg.M * cfg.k * 2.0 * 3 * cfg.m * cfg.d /
                                      (mean_ms_all * 1e-3) / 1e12) / bf16_peak()[0],
        "alg_bytes_per_step": nbytes, "touched_experts": touched,
        "kernels_us": {k: statistics.fmean(v) * 1e3 for k, v in per_kernel.items()},
        "kernels_us_note": "serialised pass (events between the launches), "
                           f"{n_split} steps after the timed region",
        "roofline": roofline,
        "e2e": e2e,
        "gpu_launches": 4 * args.steps,
        "clocks": sampler.summary() if sampler else None,
        "timed_region_wall_s": t_wall,
        "precision": "uint4 weights dequantised to fp16 in registers (q*s + fp16(-z*s), one "
                     "fused rounding), fp16 x fp16 tcgen05 MMA with fp32 accumulation, bf16 "
                     "activations in and out",
    }
    if rank == 0 and world == 1 and not args.skip_configs and cfg.name == "layer256":
        line["configs"] = time_configs(args, gu, dn, dev, status)
        line["configs_note"] = ("the other configurations of the layer, each with its own "
                                "activations and routing and the layer256 packed weights: "
                                "back-to-back w4_moe_layer calls (50, or 20 at M=2048); "
                                "gate_up and down from a serialised pass; fractions of the "
                                "measured HBM and bf16 peaks")
    if rank == 0 and world == 1 and not args.skip_cpu_baseline:
        line["cpu_baseline"] = {k: v for k, v in cpu_baseline(cfg, args.cpu_tokens).items()
                                if k != "seconds"}
    if rank == 0:
        print(json.dumps(line), flush=True)


# ----------------------------------------------------------------------------
# beside the layer: the sampler and RMSNorm
# ----------------------------------------------------------------------------
def time_region(step, args, world, dev, local):
    """Warm-up, then K back-to-back steps between one pair of CUDA events on the
    current stream (barrier + synchronize on both sides), clocks sampled
    meanwhile.  Returns (max-over-ranks ms per step, clocks summary, wall s)."""
    import torch
    for i in range(args.warmup):
        step(i)
    torch.cuda.synchronize()
    t0, t1 = torch.cuda.Event(enable_timing=True), torch.cuda.Event(enable_timing=True)
    sampler = ClockSampler(gpu_smi_id(local)) if not args.skip_clocks else None
    barrier(world)
    torch.cuda.synchronize()
    if sampler:
        sampler.__enter__()
    wall = time.perf_counter()
    t0.record()
    for i in range(args.steps):
        step(args.warmup + i)
    t1.record()
    torch.cuda.synchronize()
    wall = time.perf_counter() - wall
    if sampler:
        sampler.__exit__(None, None, None)
    barrier(world)
    ms = max_over_ranks(world, t0.elapsed_time(t1) / args.steps, dev)
    return ms, (sampler.summary() if sampler else None), wall


def time_e2e(step, args, world, dev):
    import torch
    for i in range(args.warmup):
        step(i)
    torch.cuda.synchronize()
    pairs = [(torch.cuda.Event(enable_timing=True), torch.cuda.Event(enable_timing=True))
             for _ in range(args.steps)]
    barrier(world)
    torch.cuda.synchronize()
    for i in range(args.steps):
        pairs[i][0].record()
        step(args.warmup + i)
        pairs[i][1].record()
    torch.cuda.synchronize()
    barrier(world)
    return max_over_ranks(world, statistics.fmean(a.elapsed_time(b) for a, b in pairs), dev)


def hbm_roofline(nbytes, ms, kernel, note):
    peak, kind = measured_peaks()
    achieved = nbytes / (ms * 1e-3) / 1e9
    return {"bound": "hbm", "achieved": achieved, "peak": peak, "unit": "GB/s",
            "frac": achieved / peak, "traffic": None, "kernel": kernel,
            "alg_bytes_per_launch": nbytes, "note": note,
            "peak_source": f"{kind} (MEASURED_PEAKS.json hbm_gbs: STREAM-style copy)"
            if kind == "measured" else "fallback 6.8 TB/s"}


def sampler_cpu(cfg, logits, rows, nthreads):
    """The oracle's entropy and Gumbel-max pass on `rows` rows; GB/s of logits."""
    import oracle
    t0 = time.perf_counter()
    oracle.entropy(logits[:rows], nthreads=nthreads)
    oracle.gumbel_argmax(logits[:rows], 7, 0, nthreads=nthreads)
    dt = time.perf_counter() - t0
    return rows * cfg.V * 4 / dt / 1e9, dt


def run_sampler(args, world, rank, local):
    import torch
    import w4a16_moe_expert_sync_gb300 as w4
    from w4a16_moe_expert_sync_gb300 import workloads as wl
    cfg = wl.SAMPLER_CONFIGS["canvas"]
    logits_np = wl.vocab_logits(cfg)
    nbytes = cfg.M * cfg.V * 4
    config = {"workload": f"sampler {cfg.name}: vocabulary logits [{cfg.M}, {cfg.V}] fp32 "
                          f"(rows N(0, s^2), s log-uniform in [0.5, 4], half the rows with a "
                          f"peak of 5..25), seed {cfg.seed}; entropy, Gumbel-max sample (Philox "
                          f"noise, offset = step) and argmax per row in one pass",
              "M": cfg.M, "V": cfg.V,
              "l2": "not flushed: the 268 MB of logits exceed the 126 MB L2",
              "parallelism": "replicas"}
    nthreads = os.cpu_count() or 1
    if args.impl == "reference":
        if rank != 0:
            return
        rows = 8
        for _ in range(args.warmup):
            sampler_cpu(cfg, logits_np, rows, nthreads)
        vals, dts = zip(*[sampler_cpu(cfg, logits_np, rows, nthreads) for _ in range(args.steps)])
        value = rows * cfg.V * 4 * args.steps / sum(dts) / 1e9
        sample = (f"{rows} of {cfg.M} rows per step; float64 C oracle (entropy, Philox noise, "
                  f"Gumbel-max) on {nthreads} threads")
        print(json.dumps({
            "impl": "reference", "metric": METRIC_SAMPLER, "value": value, "unit": "GB/s",
            "n_gpus": world, "steps": args.steps, "warmup": args.warmup,
            "ms_per_step": 1e3 * sum(dts) / args.steps, "higher_is_better": True,
            "scaling": "weak", "vs_baseline": None, "dtype": "f64", "data": "synthetic",
            "config": config,
            "cpu_baseline": {"value": value, "unit": "GB/s", "cores": nthreads, "kind": "oracle",
                             "sample": sample},
            "e2e": {"value": value, "unit": "GB/s", "h2d_bytes_per_step": 0,
                    "d2h_bytes_per_step": 0}}), flush=True)
        return
    w4.load_library()
    dev = torch.device("cuda", local)
    torch.cuda.set_device(dev)
    lt = torch.from_numpy(logits_np).to(dev)
    ws = torch.empty(w4.w4_sample_logits_workspace_size(cfg.M, cfg.V), dtype=torch.uint8,
                     device=dev)
    ent = torch.empty(cfg.M, device=dev)
    smp = torch.empty(cfg.M, dtype=torch.int64, device=dev)
    amx = torch.empty(cfg.M, dtype=torch.int64, device=dev)

    def step(i):
        w4.w4_sample_logits(lt, 7, i, ent, smp, amx, workspace=ws)

    ms, clocks, wall = time_region(step, args, world, dev, local)
    value = world * nbytes / (ms * 1e-3) / 1e9
    # the two launches alone, serialised, for the roofline of the dominant one
    # (the per-row merge is ~2 us)
    parts = {}
    for name, kw in (("all", dict(entropy=ent, sample=smp, argmax=amx)),
                     ("entropy", dict(entropy=ent, sample=False, argmax=False)),
                     ("argmax", dict(entropy=False, sample=False, argmax=amx))):
        evs = [(torch.cuda.Event(enable_timing=True), torch.cuda.Event(enable_timing=True))
               for _ in range(20)]
        for a, b in evs:
            torch.cuda._sleep(200000)
            a.record()
            w4.w4_sample_logits(lt, 7, 0, workspace=ws, **kw)
            b.record()
        torch.cuda.synchronize()
        parts[name] = statistics.median(a.elapsed_time(b) for a, b in evs[3:]) * 1e3
    e2e = None
    if not args.skip_e2e:
        lh = lt.cpu().pin_memory()
        eh = torch.empty(cfg.M).pin_memory()
        sh = torch.empty(cfg.M, dtype=torch.int64).pin_memory()
        ah = torch.empty(cfg.M, dtype=torch.int64).pin_memory()
        ld = torch.empty_like(lt)

        def e2e_step(i):
            ld.copy_(lh, non_blocking=True)
            w4.w4_sample_logits(ld, 7, i, ent, smp, amx, workspace=ws)
            eh.copy_(ent, non_blocking=True)
            sh.copy_(smp, non_blocking=True)
            ah.copy_(amx, non_blocking=True)

        e_ms = time_e2e(e2e_step, args, world, dev)
        e2e = {"value": world * nbytes / (e_ms * 1e-3) / 1e9, "unit": "GB/s",
               "h2d_bytes_per_step": nbytes, "d2h_bytes_per_step": cfg.M * 20,
               "ms_per_step": e_ms,
               "api": "w4_sample_logits with the logits copied in from pinned host memory and "
                      "the three outputs copied back each step"}
    line = {
        "metric": METRIC_SAMPLER, "value": value, "unit": "GB/s", "n_gpus": world,
        "steps": args.steps, "warmup": args.warmup, "ms_per_step": ms,
        "higher_is_better": True, "scaling": "weak", "vs_baseline": None, "dtype": "f32",
        "data": "synthetic", "config": config, "us_per_step": ms * 1e3,
        "variants_us": parts,
        "roofline": hbm_roofline(nbytes, parts["all"] * 1e-3, "sampler_partial_kernel "
                                 "(w4_sample_logits, all three outputs)",
                                 "one pass over the logits is the floor; the kernel is bound "
                                 "by instruction issue (Philox and the Gumbel transform per "
                                 "logit), see the profile summary"),
        "e2e": e2e, "gpu_launches": 2 * args.steps, "clocks": clocks,
        "timed_region_wall_s": wall,
    }
    if rank == 0 and world == 1 and not args.skip_cpu_baseline:
        rows = 8
        v, dt = sampler_cpu(cfg, logits_np, rows, nthreads)
        line["cpu_baseline"] = {"value": v, "unit": "GB/s", "cores": nthreads, "kind": "oracle",
                                "sample": f"{rows} of {cfg.M} rows, float64 C oracle on "
                                          f"{nthreads} threads, {dt:.2f} s wall"}
    if rank == 0:
        print(json.dumps(line), flush=True)


def run_rmsnorm(args, world, rank, local):
    import torch
    import w4a16_moe_expert_sync_gb300 as w4
    from w4a16_moe_expert_sync_gb300 import workloads as wl
    cfg = wl.NORM_CONFIGS["layer256"]
    x_np, w_np = wl.norm_inputs(cfg)
    nbytes = 2 * cfg.M * cfg.d * 2 + cfg.d * 2
    config = {"workload": f"rmsnorm {cfg.name}: x [{cfg.M}, {cfg.d}] bf16 (rows N(0, s^2), s "
                          f"log-uniform in [0.1, 10]), weight 1 + 0.1 N(0, 1), eps 1e-6, "
                          f"seed {cfg.seed}",
              "M": cfg.M, "d": cfg.d,
              "l2": "not flushed: 2.9 MB per step stays in L2, the figure is launch- and "
                    "latency-bound, not HBM-bound",
              "parallelism": "replicas"}
    nthreads = os.cpu_count() or 1
    if args.impl == "reference" or (rank == 0 and world == 1 and not args.skip_cpu_baseline):
        import oracle
        t0 = time.perf_counter()
        n = 0
        while time.perf_counter() - t0 < 2.0:
            oracle.rmsnorm(x_np, w_np, 1e-6)
            n += 1
        dt = (time.perf_counter() - t0) / n
        cpu = {"value": nbytes / dt / 1e9, "unit": "GB/s", "cores": 1, "kind": "oracle",
               "sample": f"the whole [{cfg.M}, {cfg.d}] input, float64 C oracle, one thread, "
                         f"{n} runs"}
        if args.impl == "reference":
            if rank == 0:
                print(json.dumps({
                    "impl": "reference", "metric": METRIC_RMSNORM, "value": cpu["value"],
                    "unit": "GB/s", "n_gpus": world, "steps": n, "warmup": 0,
                    "ms_per_step": dt * 1e3, "higher_is_better": True, "scaling": "weak",
                    "vs_baseline": None, "dtype": "f64", "data": "synthetic", "config": config,
                    "cpu_baseline": cpu,
                    "e2e": {"value": cpu["value"], "unit": "GB/s", "h2d_bytes_per_step": 0,
                            "d2h_bytes_per_step": 0}}), flush=True)
            return
    w4.load_library()
    dev = torch.device("cuda", local)
    torch.cuda.set_device(dev)
    x = torch.from_numpy(x_np.view(np.int16)).to(dev).view(torch.bfloat16)
    wt = torch.from_numpy(w_np.view(np.int16)).to(dev).view(torch.bfloat16)
    y = torch.empty_like(x)

    # A launch costs more host time than the kernel takes on the device, so
    # back-to-back calls from Python would time the host.  The steps are
    # captured in a CUDA graph (the library is graph-safe) and the graph is
    # replayed: device time per step with the launches back to back.
    per_graph = min(args.steps, 1000)
    replays = max(1, (args.steps + per_graph - 1) // per_graph)
    side = torch.cuda.Stream()
    side.wait_stream(torch.cuda.current_stream())
    with torch.cuda.stream(side):
        for _ in range(3):
            w4.w4_rmsnorm(x, wt, 1e-6, out=y)
    torch.cuda.current_stream().wait_stream(side)
    graph = torch.cuda.CUDAGraph()
    with torch.cuda.graph(graph):
        for _ in range(per_graph):
            w4.w4_rmsnorm(x, wt, 1e-6, out=y)

    def step(i):
        graph.replay()

    n_steps = replays * per_graph
    g_args = argparse.Namespace(**{**vars(args), "steps": replays,
                                   "warmup": max(1, args.warmup // per_graph + 1)})
    ms_replay, clocks, wall = time_region(step, g_args, world, dev, local)
    ms = ms_replay / per_graph
    e2e = None
    if not args.skip_e2e:
        xh = x.cpu().pin_memory()
        yh = torch.empty_like(xh).pin_memory()
        xd = torch.empty_like(x)

        def e2e_step(i):
            xd.copy_(xh, non_blocking=True)
            w4.w4_rmsnorm(xd, wt, 1e-6, out=y)
            yh.copy_(y, non_blocking=True)

        e_ms = time_e2e(e2e_step, args, world, dev)
        e2e = {"value": world * nbytes / (e_ms * 1e-3) / 1e9, "unit": "GB/s",
               "h2d_bytes_per_step": cfg.M * cfg.d * 2, "d2h_bytes_per_step": cfg.M * cfg.d * 2,
               "ms_per_step": e_ms, "api": "w4_rmsnorm with x copied in and y copied out"}
    line = {
        "metric": METRIC_RMSNORM, "value": world * nbytes / (ms * 1e-3) / 1e9, "unit": "GB/s",
        "n_gpus": world, "steps": n_steps, "warmup": args.warmup, "ms_per_step": ms,
        "higher_is_better": True, "scaling": "weak", "vs_baseline": None, "dtype": "f32",
        "data": "synthetic", "config": config, "us_per_step": ms * 1e3,
        "timing": f"{replays} replays of a CUDA graph of {per_graph} w4_rmsnorm calls",
        "roofline": hbm_roofline(nbytes, ms, "rmsnorm_warp_kernel<12> (w4_rmsnorm)",
                                 "back-to-back launches; 2.9 MB is far below what it takes to "
                                 "reach HBM bandwidth, the time is the launch and one "
                                 "load-reduce-store latency chain"),
        "e2e": e2e, "gpu_launches": n_steps, "clocks": clocks, "timed_region_wall_s": wall,
    }
    if rank == 0 and world == 1 and not args.skip_cpu_baseline:
        line["cpu_baseline"] = cpu
    if rank == 0:
        print(json.dumps(line), flush=True)


def graph_time(fn, per_graph, replays, warm_replays=2):
    """Device time per call of fn, captured per_graph times in a CUDA graph and
    replayed: back-to-back launches without the host in the way."""
    import torch
    side = torch.cuda.Stream()
    side.wait_stream(torch.cuda.current_stream())
    with torch.cuda.stream(side):
        for _ in range(3):
            fn()
    torch.cuda.current_stream().wait_stream(side)
    graph = torch.cuda.CUDAGraph()
    with torch.cuda.graph(graph):
        for _ in range(per_graph):
            fn()
    for _ in range(warm_replays):
        graph.replay()
    torch.cuda.synchronize()
    a, b = torch.cuda.Event(enable_timing=True), torch.cuda.Event(enable_timing=True)
    a.record()
    for _ in range(replays):
        graph.replay()
    b.record()
    torch.cuda.synchronize()
    return a.elapsed_time(b) / (replays * per_graph), graph


def run_linear(args, world, rank, local):
    import torch
    import oracle
    import w4a16_moe_expert_sync_gb300 as w4
    from w4a16_moe_expert_sync_gb300 import workloads as wl
    shapes = [wl.LINEAR_CONFIGS["qkv256"], wl.LINEAR_CONFIGS["lmhead256"]]
    config = {"workload": "dense W4A16 linear at 256 rows: qkv256 (K=2816, N=4096) and lmhead256 "
                          "(K=2816, N=16384, a tile of the vocabulary head); x ~ N(0, 1) bf16, "
                          "W ~ N(0, 0.02^2) quantised to uint4 with fp16 scale/zero per 128",
              "shapes": [dataclasses_asdict(c) for c in shapes],
              "l2": "not flushed: the graph replays the same weights (5.8 MB and 23 MB packed); "
                    "the L2 holds the QKV weights between calls",
              "parallelism": "replicas"}
    nthreads = os.cpu_count() or 1
    cfg0 = shapes[0]
    if args.impl == "reference" or (rank == 0 and world == 1 and not args.skip_cpu_baseline):
        x_np, W_np = wl.linear_inputs(cfg0)
        q_np, s_np, z_np = oracle.quantize_w4(W_np, 128)
        rows = 16
        t0 = time.perf_counter()
        oracle.w4a16_linear(x_np[:rows], q_np, s_np, z_np, 128, nthreads=nthreads)
        dt = time.perf_counter() - t0
        flops = 2.0 * rows * cfg0.K * cfg0.N
        cpu = {"value": flops / dt / 1e12, "unit": "TFLOP/s", "cores": nthreads, "kind": "oracle",
               "sample": f"{rows} of {cfg0.M} rows of qkv256, float64 C oracle on {nthreads} "
                         f"threads, {dt:.2f} s wall"}
        if args.impl == "reference":
            if rank == 0:
                print(json.dumps({
                    "impl": "reference", "metric": METRIC_LINEAR, "value": cpu["value"],
                    "unit": "TFLOP/s", "n_gpus": world, "steps": 1, "warmup": 0,
                    "ms_per_step": dt * 1e3, "higher_is_better": True, "scaling": "weak",
                    "vs_baseline": None, "dtype": "f64", "data": "synthetic", "config": config,
                    "cpu_baseline": cpu,
                    "e2e": {"value": cpu["value"], "unit": "TFLOP/s", "h2d_bytes_per_step": 0,
                            "d2h_bytes_per_step": 0}}), flush=True)
            return
    w4.load_library()
    dev = torch.device("cuda", local)
    torch.cuda.set_device(dev)
    per_graph = 50
    replays = max(1, args.steps // per_graph)
    results, keep = {}, []
    for cfg in shapes:
        x_np, W_np = wl.linear_inputs(cfg)
        x = torch.from_numpy(x_np.view(np.int16)).to(dev).view(torch.bfloat16)
        W = torch.from_numpy(W_np).to(dev)
        q, s_, z = (t[0] for t in w4.w4_quantize(W, cfg.group))
        ws = torch.empty(w4.w4_w4a16_linear_workspace_size(cfg.M, cfg.K, cfg.N, cfg.group),
                         dtype=torch.uint8, device=dev)
        y = torch.empty((cfg.M, cfg.N), dtype=torch.bfloat16, device=dev)
        Wb = W.to(torch.bfloat16)
        ms_w4, g1 = graph_time(lambda: w4.w4_w4a16_linear(x, q, s_, z, cfg.group, workspace=ws,
                                                          out=y), per_graph, replays)
        ms_bf, g2 = graph_time(lambda: torch.nn.functional.linear(x, Wb), per_graph, replays)
        keep += [g1, g2]
        flops = 2.0 * cfg.M * cfg.K * cfg.N
        results[cfg.name] = {"us_w4a16": ms_w4 * 1e3, "us_cublas_bf16": ms_bf * 1e3,
                             "tflops_w4a16": flops / (ms_w4 * 1e-3) / 1e12,
                             "speed_vs_cublas_bf16": ms_bf / ms_w4,
                             "weight_bytes": cfg.N * cfg.K // 2 + 2 * 2 * cfg.N * (cfg.K // cfg.group)}
    # the timed region proper: replays of the QKV graph, clocks sampled
    cfg = shapes[0]
    x_np, W_np = wl.linear_inputs(cfg)
    x = torch.from_numpy(x_np.view(np.int16)).to(dev).view(torch.bfloat16)
    q, s_, z = (t[0] for t in w4.w4_quantize(torch.from_numpy(W_np).to(dev), cfg.group))
    ws = torch.empty(w4.w4_w4a16_linear_workspace_size(cfg.M, cfg.K, cfg.N, cfg.group), dtype=torch.uint8,
                     device=dev)
    y = torch.empty((cfg.M, cfg.N), dtype=torch.bfloat16, device=dev)
    _, graph = graph_time(lambda: w4.w4_w4a16_linear(x, q, s_, z, cfg.group, workspace=ws, out=y),
                          per_graph, 1)
    g_args = argparse.Namespace(**{**vars(args), "steps": replays, "warmup": 3})
    ms_replay, clocks, wall = time_region(lambda i: graph.replay(), g_args, world, dev, local)
    ms = ms_replay / per_graph
    flops = 2.0 * cfg.M * cfg.K * cfg.N
    value = world * flops / (ms * 1e-3) / 1e12
    peak_bf16 = None
    try:
        with open(os.path.join(ROOT, "MEASURED_PEAKS.json")) as f:
            peak_bf16 = float(json.load(f)["bf16_tflops"])
        peak_kind = "measured (MEASURED_PEAKS.json bf16_tflops: cuBLAS bf16 burst; fp16 runs at the same rate)"
    except Exception:
        peak_bf16, peak_kind = 1900.0, "fallback 1.9 PFLOP/s"
    e2e = None
    if not args.skip_e2e:
        xh = x.cpu().pin_memory()
        yh = torch.empty((cfg.M, cfg.N), dtype=torch.bfloat16).pin_memory()
        xd = torch.empty_like(x)

        def e2e_step(i):
            xd.copy_(xh, non_blocking=True)
            w4.w4_w4a16_linear(xd, q, s_, z, cfg.group, workspace=ws, out=y)
            yh.copy_(y, non_blocking=True)

        e_ms = time_e2e(e2e_step, args, world, dev)
        e2e = {"value": world * flops / (e_ms * 1e-3) / 1e12, "unit": "TFLOP/s",
               "h2d_bytes_per_step": cfg.M * cfg.K * 2, "d2h_bytes_per_step": cfg.M * cfg.N * 2,
               "ms_per_step": e_ms, "api": "w4_w4a16_linear with x copied in and y copied out"}
    line = {
        "metric": METRIC_LINEAR, "value": value, "unit": "TFLOP/s", "n_gpus": world,
        "steps": replays * per_graph, "warmup": args.warmup, "ms_per_step": ms,
        "higher_is_better": True, "scaling": "weak", "vs_baseline": None, "dtype": "fp16",
        "data": "synthetic", "config": config, "us_per_step": ms * 1e3, "shapes": results,
        "timing": f"{replays} replays of a CUDA graph of {per_graph} calls (qkv256)",
        "roofline": {"bound": "tensor", "achieved": value / world, "peak": peak_bf16,
                     "unit": "TFLOP/s", "frac": value / world / peak_bf16, "traffic": None,
                     "kernel": "dense_gemm_kernel (w4_w4a16_linear, qkv256)",
                     "alg_flops_per_launch": flops, "peak_source": peak_kind,
                     "note": "each 128-row weight panel is dequantised once per pass of up "
                             "to 256 token rows; at these sizes the call is bound by its "
                             "fixed per-call and per-CTA latency, not by the tensor pipe"},
        "e2e": e2e, "gpu_launches": 2 * replays * per_graph, "clocks": clocks,
        "timed_region_wall_s": wall,
    }
    if rank == 0 and world == 1 and not args.skip_cpu_baseline:
        line["cpu_baseline"] = cpu
    if rank == 0:
        print(json.dumps(line), flush=True)


def dataclasses_asdict(c):
    import dataclasses
    return dataclasses.asdict(c)


def main():
    ap = argparse.ArgumentParser(description=__doc__.split("\n")[0])
    ap.add_argument("--gpus", type=int, default=1)
    ap.add_argument("--steps", type=int, default=1000)
    ap.add_argument("--warmup", type=int, default=10)
    ap.add_argument("--impl", choices=["w4moe", "reference"], default="w4moe")
    ap.add_argument("--config", default="layer256")
    ap.add_argument("--block-m", type=int, default=16)
    ap.add_argument("--cpu-tokens", type=int, default=16)
    ap.add_argument("--skip-cpu-baseline", action="store_true")
    ap.add_argument("--skip-e2e", action="store_true")
    ap.add_argument("--skip-clocks", action="store_true")
    ap.add_argument("--skip-configs", action="store_true",
                    help="leave out the compact timing of the other layer configurations")
    ap.add_argument("--workload", choices=["layer", "sampler", "rmsnorm", "linear"],
                    default="layer")
    args = ap.parse_args()
    if args.warmup < 3:
        ap.error("--warmup must be at least 3")
    from w4a16_moe_expert_sync_gb300 import workloads as wl
    cfg = wl.CONFIGS[args.config]
    world, rank, local = dist_setup(args.gpus)
    if args.workload == "sampler":
        run_sampler(args, world, rank, local)
    elif args.workload == "rmsnorm":
        run_rmsnorm(args, world, rank, local)
    elif args.workload == "linear":
        run_linear(args, world, rank, local)
    elif args.impl == "reference":
        run_reference(args, cfg, world, rank)
    else:
        run_gpu(args, cfg, world, rank, local)
    if world > 1:
        import torch.distributed as dist
        dist.destroy_process_group()


if __name__ == "__main__":
    main()
