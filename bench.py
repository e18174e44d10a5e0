"""Benchmark of the FAVOR+ attention forward pass on GB300 (one JSON line).

A step is one forward pass (feature maps, state reduction, causal scan or
non-causal output, normalisation) over the whole workload, inputs resident
in HBM.  Default workload: causal, B=4, H=16, L=8192, d=dv=64, m=256,
block-orthogonal omega, bf16 inputs (synthetic, seeded).

  python bench.py [--gpus N] [--steps K] [--warmup W] [--impl ours|reference]
                  [--workload causal8k|nc4096|long64k|long64k_nc|sweep16k|sweep16k_m128|sweep16k_m512|
                              decode8k|decode_b256|causal8k_bwd|nc4096_bwd]

--impl reference times the float64 CPU oracle (the slow, obviously correct
statement of the method) on bounded samples of the same workload.
Multi-GPU (torchrun): every rank runs its own replica of the workload (the
path shards over heads with no exchange), value = all ranks' tokens / max time.
"""
from __future__ import annotations

import argparse
import json
import os
import statistics
import subprocess
import sys
import threading
import time

ROOT = os.path.dirname(os.path.abspath(__file__))
sys.path.insert(0, ROOT)

METRIC = "FAVOR+ fwd tokens/sec (B·H·L/s) at L=8192 causal m=256; % of roofline"
# the fp32 SIMT kernels (shapes the tensor-core layouts do not cover)
SIMT_KERNELS = ("chunk_rows", "simt_project", "simt_features", "simt_key_scale", "state_scan", "state_sum")


def metric_for(name, w, causal):
    """The headline workload keeps the published headline metric string; the
    others name their own shape."""
    if name == "causal8k" and w.name == "causal8k":
        return METRIC
    return (f"FAVOR+ fwd tokens/sec (B·H·L/s) on {name}: L={w.L} "
            f"{'causal' if causal else 'non-causal'} d={w.d} m={w.m}; % of roofline")
L2_BYTES = 129 * 1024 * 1024
FALLBACK_HBM_GBS = 6800.0
FALLBACK_BF16_TFLOPS = 1900.0

# DRAM traffic (read + write bytes per launch) of a kernel from one ncu capture
# (profiles/), valid while the kernel's source section is unchanged.
TRAFFIC = {
    ("tc_causal", "causal8k"): (309.65e6, "bf625141d5c0677b"),
    ("tc_causal", "long64k"): (309.21e6, "bf625141d5c0677b"),
    ("tc_causal_split", "sweep16k"): (308.31e6, "6187aa4fa5316de2"),
    # captured on the first 8 of 16 heads, scaled by heads
    ("tc_causal", "sweep16k_m128"): (270.6e6, "bf625141d5c0677b"),
    ("tc_causal_split", "sweep16k_m512"): (285.4e6, "6187aa4fa5316de2"),
    ("tc_state", "causal8k"): (68.93e6, "219f9714fc031c6e"),
    ("tc_state", "nc4096"): (104.77e6, "219f9714fc031c6e"),
    ("tc_state", "long64k_nc"): (138.46e6, "219f9714fc031c6e"),
    ("tc_output", "nc4096"): (102.45e6, "60759cfc8dee8c7e"),
    ("decode_step", "decode_b256"): (496.87e6, "74c42f3d2b49b28e"),
}
KERNEL_SECTIONS = {   # kernel: (source file, first line of its section, first line after it)
    "tc_causal": ("favor_tc.cu", "// tc_causal: the chunked causal scan, warp-specialised.",
                  "// tc_causal_split: the chunked causal scan of a head whose features are"),
    "tc_causal_split": ("favor_tc.cu", "// tc_causal_split: the chunked causal scan of a head whose features are",
                        "// tc_output: non-causal rows"),
    "tc_output": ("favor_tc.cu", "// tc_output: non-causal rows", "// host side"),
    "tc_state": ("favor_tc.cu", "// tc_state: per (feature group, piece, head) the state of a run of keys",
                 "// tc_combine:"),
    "decode_step": ("favor_decode.cu", "// decode_step: persistent CTAs", "bool overlaps("),
}


def kernel_source_hash(kernel):
    import hashlib
    if kernel not in KERNEL_SECTIONS:
        return None
    f, a, b = KERNEL_SECTIONS[kernel]
    path = os.path.join(ROOT, "favor_random_feature_gb300", "csrc", f)
    try:
        s = open(path).read()
        return hashlib.sha256(s[s.index(a):s.index(b)].encode()).hexdigest()[:16]
    except (OSError, ValueError):
        return None


def measured_traffic(kernel, workload_name):
    entry = TRAFFIC.get((kernel, workload_name))
    if entry and kernel_source_hash(kernel) == entry[1]:
        return entry[0]
    return None


def workload(name):
    from favor_inputs import CAUSAL8K, LONG64K, NC4096, SWEEP16K
    table = {
        "causal8k": (CAUSAL8K, True),
        "nc4096": (NC4096, False),
        "long64k": (LONG64K, True),
        "long64k_nc": (LONG64K, False),
        "sweep16k": (SWEEP16K, True),
        "sweep16k_m128": (SWEEP16K.with_(m=128), True),
        "sweep16k_m512": (SWEEP16K.with_(m=512), True),
    }
    return table[name]


def describe(w, causal):
    return {
        "workload": f"{w.name}: B={w.B} H={w.H} L={w.L} d={w.d} dv={w.dv} m={w.m} "
                    f"{'causal' if causal else 'non-causal'} positive-features "
                    f"omega={w.omega} seed={w.seed}",
        "B": w.B, "H": w.H, "L": w.L, "d": w.d, "dv": w.dv, "m": w.m, "causal": causal,
        "feature_map": "positive", "omega": w.omega,
        "inputs": "bf16 q,k,v; fp32 omega; fp32 out",
        "l2": "flushed between steps (256 MiB write, outside the timed events); "
              "step inputs+outputs exceed L2",
    }


def per_token(w):
    """Algorithmic work per token: flops, HBM bytes, exps (positive map)."""
    flops = 2 * w.m * (2 * w.d + 2 * w.dv)
    hbm = 2 * (2 * w.d + w.dv) + 4 * w.dv
    exps = 2 * w.m
    return flops, hbm, exps


def peaks():
    path = os.path.join(ROOT, "MEASURED_PEAKS.json")
    try:
        with open(path) as f:
            j = json.load(f)
        return float(j["hbm_gbs"]), float(j["bf16_tflops"]), "measured"
    except Exception:
        return FALLBACK_HBM_GBS, FALLBACK_BF16_TFLOPS, "fallback"


class ClockSampler:
    """nvidia-smi samples (host timestamped) while the benchmark runs."""

    FIELDS = ("index,clocks.sm,clocks.max.sm,power.draw,clocks_event_reasons.active,"
              "clocks_event_reasons.hw_slowdown,clocks_event_reasons.hw_thermal_slowdown,"
              "clocks_event_reasons.sw_thermal_slowdown,clocks_event_reasons.sw_power_cap")

    def __init__(self, gpu_index):
        self.samples = []
        self.proc = None
        try:
            self.proc = subprocess.Popen(
                ["nvidia-smi", f"--query-gpu={self.FIELDS}", "--format=csv,noheader,nounits",
                 "-i", str(gpu_index), "-lms", "100"],
                stdout=subprocess.PIPE, stderr=subprocess.DEVNULL, text=True)
        except Exception:
            return
        self.thread = threading.Thread(target=self._read, daemon=True)
        self.thread.start()

    def _read(self):
        for line in self.proc.stdout:
            parts = [p.strip() for p in line.split(",")]
            if len(parts) >= 9:
                self.samples.append((time.time(), parts))

    def stop(self):
        if self.proc:
            self.proc.terminate()
            try:
                self.proc.wait(timeout=5)
            except Exception:
                self.proc.kill()

    def summary(self, t0, t1):
        if not self.samples:
            return {"sm_mhz": None, "sm_max_mhz": None, "reasons": ["nvidia-smi unavailable"]}
        win = [s for t, s in self.samples if t0 - 0.25 <= t <= t1 + 0.25]
        if not win:
            win = [s for _, s in self.samples[-5:]]
        sm = [float(s[1]) for s in win if s[1].replace(".", "").isdigit()]
        mx = [float(s[2]) for s in win if s[2].replace(".", "").isdigit()]
        names = ["hw_slowdown", "hw_thermal_slowdown", "sw_thermal_slowdown", "sw_power_cap"]
        reasons = sorted({n for s in win for n, v in zip(names, s[5:9]) if v.lower() == "active"})
        return {"sm_mhz": statistics.median(sm) if sm else None,
                "sm_max_mhz": max(mx) if mx else None,
                "reasons": reasons, "samples": len(win)}


def cpu_baseline(inp, causal, heads_per_sample=None):
    """The float64 oracle, as it stands, on a bounded sample of the workload."""
    import oracle
    w = inp.w
    cores = oracle.threads_used()
    n = heads_per_sample or min(w.B * w.H, 2 * cores)
    # the first n heads as a batch of one: q/k/v [1][n][L][.], omega [n][m][d]
    sel = lambda a: a.reshape(w.B * w.H, w.L, a.shape[-1])[:n][None]
    q, k, v = sel(inp.q32), sel(inp.k32), sel(inp.v32)
    om = inp.omega[[h % w.H for h in range(n)]]
    t0 = time.perf_counter()
    oracle.forward(q, k, v, om, causal=causal)
    dt = time.perf_counter() - t0
    return {"value": n * w.L / dt, "unit": "tokens/s", "cores": cores, "kind": "oracle",
            "sample": f"{n} of {w.B * w.H} heads x L={w.L} (float64 C oracle, OpenMP over heads)",
            "seconds": dt}


def max_over_ranks(values, dist, device):
    """The per-rank timings reduced to their maximum over the ranks (the job
    takes as long as its slowest replica); unchanged on one process."""
    if not dist:
        return list(values)
    import torch
    t = torch.tensor(list(values), dtype=torch.float64, device=device)
    dist.all_reduce(t, op=dist.ReduceOp.MAX)
    return t.tolist()


def job_throughput(tokens_per_rank, world, ms):
    """Whole-job tokens/s: every rank's tokens over the slowest rank's time."""
    return world * tokens_per_rank / (ms / 1000.0)


def rank_inputs_seed(seed, rank):
    """Each replica draws its own inputs (rank 0 the workload's seed)."""
    return seed + 1000 * rank


def run_reference(args):
    rank = int(os.environ.get("RANK", "0"))
    if rank != 0:
        return 0
    import oracle
    from favor_inputs import make_inputs
    w, causal = workload(args.workload)
    if args.workload == "long64k_nc":
        causal = False
    inp = make_inputs(w)
    cores = oracle.threads_used()
    n = min(w.B * w.H, cores)
    for _ in range(args.warmup):
        cpu_baseline(inp, causal, heads_per_sample=n)
    times = []
    for _ in range(args.steps):
        r = cpu_baseline(inp, causal, heads_per_sample=n)
        times.append(r["seconds"])
    ms = 1000 * statistics.mean(times)
    value = n * w.L / (ms / 1000)
    line = {
        "impl": "reference", "metric": metric_for(args.workload, w, causal), "value": value,
        "unit": "tokens/s", "n_gpus": 0,
        "steps": args.steps, "warmup": args.warmup, "ms_per_step": ms, "higher_is_better": True,
        "scaling": "weak", "vs_baseline": None, "dtype": "f64", "data": "synthetic",
        "config": describe(w, causal),
        "cpu_baseline": {"value": value, "unit": "tokens/s", "cores": cores, "kind": "oracle",
                         "sample": f"{n} of {w.B * w.H} heads x L={w.L} per step"},
        "e2e": {"value": value, "unit": "tokens/s", "h2d_bytes_per_step": 0,
                "d2h_bytes_per_step": 0},
    }
    print(json.dumps(line))
    return 0


def run_ours(args):
    import numpy as np
    import torch

    rank = int(os.environ.get("RANK", "0"))
    world = int(os.environ.get("WORLD_SIZE", "1"))
    local = int(os.environ.get("LOCAL_RANK", "0"))
    if world != args.gpus:
        raise SystemExit(f"--gpus {args.gpus} but WORLD_SIZE={world}")
    torch.cuda.set_device(local)
    dist = None
    if world > 1:
        import torch.distributed as dist
        dist.init_process_group("nccl")

    from favor_random_feature_gb300 import build as fbuild
    fbuild.build()
    import favor_random_feature_gb300 as fv
    from favor_inputs import make_inputs

    w, causal = workload(args.workload)
    if args.workload == "long64k_nc":
        causal = False
    if args.heads:   # a smaller case of the same workload, for ncu captures
        w = w.with_(B=max(1, args.heads // w.H), H=min(args.heads, w.H))
    inp = make_inputs(w.with_(seed=rank_inputs_seed(w.seed, rank)))
    dev = lambda a: torch.from_numpy(np.ascontiguousarray(a).view(np.int16)).view(
        torch.bfloat16).cuda()
    q, k, v = dev(inp.q), dev(inp.k), dev(inp.v)
    om = torch.from_numpy(np.ascontiguousarray(inp.omega)).cuda()
    out = torch.empty((w.B, w.H, w.L, w.dv), dtype=torch.float32, device="cuda")
    flush = torch.empty(256 * 1024 * 1024 // 4, dtype=torch.int32, device="cuda")
    stream = torch.cuda.current_stream()
    call = lambda: fv.favor_attn_forward(q, k, v, om, out, w.B, w.H, w.L, w.d, w.dv, w.m,
                                         int(causal), 0, stream)

    def check(rc):
        if rc != fv.FAVOR_OK:
            raise fv.FavorError(rc, "favor_attn_forward")

    for _ in range(max(3, args.warmup)):
        check(call())
    torch.cuda.synchronize()
    st = fv.favor_get_device_status(stream)
    if st != fv.FAVOR_OK:
        raise fv.FavorError(st, "device status")

    sampler = ClockSampler(torch.cuda.current_device() if "CUDA_VISIBLE_DEVICES" not in os.environ
                           else os.environ["CUDA_VISIBLE_DEVICES"].split(",")[local])
    # soak so that the clock samples see the GPU under load
    t_soak = time.time()
    while time.time() - t_soak < 1.0:
        check(call())
        torch.cuda.synchronize()

    evs = [(torch.cuda.Event(enable_timing=True), torch.cuda.Event(enable_timing=True))
           for _ in range(args.steps)]
    if dist:
        dist.barrier()
    torch.cuda.synchronize()
    t0 = time.time()
    for i in range(args.steps):
        flush.zero_()
        evs[i][0].record(stream)
        check(call())
        evs[i][1].record(stream)
    torch.cuda.synchronize()
    t1 = time.time()
    st = fv.favor_get_device_status(stream)
    if st != fv.FAVOR_OK:
        raise fv.FavorError(st, "device status after the timed steps")
    if dist:
        dist.barrier()
    sampler.stop()
    step_ms = [a.elapsed_time(b) for a, b in evs]
    ms = statistics.mean(step_ms)
    # the dominant kernel's own time and the launch count, from separate steps:
    # the measurement hook records events around that kernel, which would keep
    # it from overlapping its prologue with the kernel before it in the timed
    # steps above
    stat_steps = max(3, min(args.steps, 10))
    fv.favor_stats_enable(True)
    for _ in range(stat_steps):
        flush.zero_()
        check(call())
    torch.cuda.synchronize()
    stats = fv.favor_stats_read()
    fv.favor_stats_enable(False)
    dom_ms = stats.dominant_ms / max(1, stats.dominant_launches)
    launches_per_step = stats.kernel_launches / stat_steps
    ms, dom_ms = max_over_ranks([ms, dom_ms], dist, "cuda")
    tokens = w.B * w.H * w.L
    value = job_throughput(tokens, world, ms)

    flops_tok, bytes_tok, exps_tok = per_token(w)
    hbm_gbs, tflops, src = peaks()
    kname = stats.dominant_kernel.decode() if stats.dominant_kernel else ""
    # algorithmic HBM bytes of the dominant kernel per token: the causal scan
    # reads q, k, v and writes out; the non-causal state kernel reads k and v
    # (the output kernel then reads q and writes out)
    if kname == "tc_state":
        kbytes_tok = 2 * (w.d + w.dv)
    elif kname == "tc_output":
        kbytes_tok = 2 * w.d + 4 * w.dv
    else:
        kbytes_tok = bytes_tok
    achieved = kbytes_tok * tokens / (dom_ms / 1000.0) / 1e9
    simt = kname in SIMT_KERNELS   # the fp32 SIMT forward (shapes outside the tensor-core layouts)
    # the step's three bounds: tensor (measured bf16 rate; the path's fp16 MMAs run at
    # the same rate), HBM (measured copy), MUFU (measured: the ex2 throughput probe)
    clocks = sampler.summary(t0, t1)
    mufu_rate = fv.favor_probe_ex2_rate(stream)
    bounds_ms = {"tensor": flops_tok * tokens / (tflops * 1e12) * 1e3,
                 "hbm": bytes_tok * tokens / (hbm_gbs * 1e9) * 1e3,
                 "mufu": exps_tok * tokens / mufu_rate * 1e3}
    roof_ms = max(bounds_ms.values())
    binding = max(bounds_ms, key=bounds_ms.get)
    step_quantity = {"tensor": (flops_tok * tokens / 1e12, tflops, "TFLOP/s"),
                     "hbm": (bytes_tok * tokens / 1e9, hbm_gbs, "GB/s"),
                     "mufu": (exps_tok * tokens / 1e12, mufu_rate / 1e12, "T ex2/s")}[binding]

    # end to end through the host-buffer entry point (pinned host memory)
    pin = lambda a: torch.from_numpy(np.ascontiguousarray(a)).pin_memory().numpy()
    hq, hk, hv = pin(inp.q), pin(inp.k), pin(inp.v)
    hom = pin(np.ascontiguousarray(inp.omega, dtype=np.float32))
    hout = torch.empty((w.B, w.H, w.L, w.dv), dtype=torch.float32).pin_memory().numpy()
    ecall = lambda: fv.favor_attn_forward_host(hq, hk, hv, hom, hout, w.B, w.H, w.L, w.d, w.dv,
                                               w.m, int(causal), 0, stream)
    for _ in range(2):
        check(ecall())
    e2e_steps = max(3, min(args.steps, 20))
    if dist:
        dist.barrier()
    te0 = time.perf_counter()
    for _ in range(e2e_steps):
        check(ecall())
    te = (time.perf_counter() - te0) / e2e_steps
    st = fv.favor_get_device_status(stream)
    if st != fv.FAVOR_OK:
        raise fv.FavorError(st, "device status after the end-to-end steps")
    (te,) = max_over_ranks([te], dist, "cuda")
    h2d = inp.q.nbytes + inp.k.nbytes + inp.v.nbytes + hom.nbytes
    d2h = hout.nbytes

    if simt:
        # the fp32 SIMT path: the roofline is the step's (the method's three
        # bounds); the dominant kernel's fp32-ALU fraction goes under simt_alu
        roofline = {
            "bound": binding, "achieved": step_quantity[0] / (ms / 1000.0), "peak": step_quantity[1],
            "unit": step_quantity[2], "frac": roof_ms / ms, "traffic": None,
            "kernel": f"whole step (fp32 SIMT path; dominant kernel {kname})", "kernel_ms": ms,
            "peak_source": src, "step_roofline_ms": roof_ms, "step_frac": roof_ms / ms,
            "step_bounds_ms": bounds_ms, "mufu_peak_source": "measured: favor_probe_ex2_rate",
            "mufu_ex2_per_s": mufu_rate,
            "simt_alu": simt_rows_roofline(w, causal, tokens, dom_ms, clocks) if kname == "chunk_rows" else None,
        }
    else:
        roofline = {
            "bound": "hbm", "achieved": achieved, "peak": hbm_gbs, "unit": "GB/s",
            "frac": achieved / hbm_gbs, "traffic": measured_traffic(kname, args.workload),
            "kernel": kname or None,
            "kernel_ms": dom_ms, "peak_source": src,
            "algorithmic_bytes_per_launch": kbytes_tok * tokens,
            "step_roofline_ms": roof_ms, "step_frac": roof_ms / ms,
            "step_bounds_ms": bounds_ms,
            "mufu_peak_source": "measured: favor_probe_ex2_rate", "mufu_ex2_per_s": mufu_rate,
        }
    line = {
        "metric": metric_for(args.workload, w, causal), "value": value, "unit": "tokens/s", "n_gpus": world,
        "steps": args.steps, "warmup": args.warmup, "ms_per_step": ms, "higher_is_better": True,
        "scaling": "weak", "vs_baseline": None, "dtype": "f32" if simt else "f16", "data": "synthetic",
        "config": dict(describe(w, causal),
                       workload=(f"PROFILING CASE (first {w.B * w.H} heads, not a benchmark value) "
                                 if args.heads else "") + describe(w, causal)["workload"]),
        "roofline": roofline,
        "e2e": {"value": world * tokens / te, "unit": "tokens/s", "h2d_bytes_per_step": h2d,
                "d2h_bytes_per_step": d2h},
        "gpu_launches": int(round(launches_per_step * args.steps)),
        "clocks": clocks,
    }
    if rank == 0 and world == 1 and not args.no_cpu_baseline:
        cb = cpu_baseline(inp, causal)
        cb.pop("seconds", None)
        line["cpu_baseline"] = cb
    if rank == 0:
        print(json.dumps(line))
    if dist:
        dist.destroy_process_group()
    return 0


# decode workloads: (shape of the forward workload, batch, prefix length).
# The state of a prefix is built once; each step decodes one token per head
# and updates the state in place.  The large batch takes a short prefix: the
# state's size, and so the step's work, does not depend on its length.
DECODE_METRIC = "FAVOR+ decode tokens/sec (one token per head per step, B*H/s); % of HBM roofline"
DECODE = {"decode8k": ("causal8k", 4, 8192), "decode_b256": ("causal8k", 256, 128)}


def decode_bytes_per_head(w):
    """Algorithmic HBM bytes of one decode step of one head: the state read and
    written (r (dv + 2) fp32 each way), q, k, v (bf16) and out (fp32)."""
    return 8 * w.m * (w.dv + 2) + 2 * (2 * w.d + w.dv) + 4 * w.dv


def decode_cpu_baseline(w, n_heads, steps):
    """The float64 oracle's decode step on n heads (state of a 16-key prefix)."""
    import numpy as np
    import oracle
    from favor_inputs import make_inputs
    inp = make_inputs(w.with_(B=1, H=n_heads), L=16 + steps)
    om = inp.omega
    S, z = oracle.state(inp.k32[:, :, :16], inp.v32[:, :, :16], om)
    t0 = time.perf_counter()
    for t in range(16, 16 + steps):
        _, S, z = oracle.decode_step(inp.q32[:, :, t], inp.k32[:, :, t], inp.v32[:, :, t], om, S, z)
    dt = time.perf_counter() - t0
    return {"value": n_heads * steps / dt, "unit": "tokens/s", "cores": 1, "kind": "oracle",
            "sample": f"{n_heads} heads x {steps} decode steps (float64 C oracle, one thread)",
            "seconds": dt}


# backward workloads: the forward workload's shape; a step is one backward
# call (gradients of q, k, v and omega for a seeded dloss/dout)
BWD_METRIC = "FAVOR+ backward tokens/sec (B*H*L/s); % of the fp32 ALU roofline"
BACKWARD = {"causal8k_bwd": "causal8k", "nc4096_bwd": "nc4096"}
BWD_ROWS = 64   # rows per chunk of the SIMT forward and backward kernels


def simt_rows_roofline(w, causal, tokens, dom_ms, clocks):
    """The fp32 SIMT forward's dominant kernel (chunk_rows) against the fp32 ALU
    peak: algorithmic FLOPs per token num = phi_q S (2 r (dv + 1)) and, causal,
    the masked chunk product A (2 r C / 2) and A_m [V | 1] (2 (C / 2)(dv + 1))."""
    import torch
    r, dv, C = w.r, w.dv, BWD_ROWS
    flops = 2 * r * (dv + 1) + ((r * C + C * (dv + 1)) if causal else 0)
    mhz = clocks.get("sm_max_mhz") or 2070.0
    peak = torch.cuda.get_device_properties(torch.cuda.current_device()).multi_processor_count * 128 * 2 * mhz * 1e6 / 1e12
    achieved = flops * tokens / (dom_ms / 1000.0) / 1e12
    return {"bound": "alu", "achieved": achieved, "peak": peak, "unit": "TFLOP/s", "frac": achieved / peak,
            "traffic": None, "peak_source": "derived: SMs x 128 fp32 lanes x 2 flops x max SM clock",
            "algorithmic_bytes_per_launch": None, "algorithmic_flops_per_token": flops}


def bwd_chunk_flops_per_token(w, causal):
    """Algorithmic FLOPs per token of the backward chunk kernel: the masked
    chunk product B (causal, lower triangle; the masked A comes from the row
    kernel), dphi_q and dphi_k from the carried states plus the chunk sums,
    and dv; the dv + 1 state columns without padding.  The kernel executes
    more (a full 64 x 64 B tile, columns padded to dv + 4)."""
    r, dv, C = w.r, w.dv, BWD_ROWS
    intra = C / 2 if causal else 0
    ab = (C / 2) * (dv + 1) * 2 if causal else 0
    dphi = 2 * r * (dv + 1 + intra) * 2
    dvv = dv * (r + intra) * 2
    return ab + dphi + dvv


def run_backward(args):
    import numpy as np
    import torch
    from favor_random_feature_gb300 import build as fbuild
    fbuild.build()
    import favor_random_feature_gb300 as fv
    from favor_inputs import make_inputs

    if int(os.environ.get("WORLD_SIZE", "1")) != 1 or args.gpus != 1:
        raise SystemExit("backward workloads run on one GPU (replicas only)")
    w, causal = workload(BACKWARD[args.workload])
    if args.heads:   # a smaller case of the same workload, for ncu captures
        w = w.with_(B=1, H=min(args.heads, w.H))
    torch.cuda.set_device(int(os.environ.get("LOCAL_RANK", "0")))
    inp = make_inputs(w)
    dev16 = lambda a: torch.from_numpy(np.ascontiguousarray(a).view(np.int16)).view(torch.bfloat16).cuda()
    q, k, v = dev16(inp.q), dev16(inp.k), dev16(inp.v)
    om = torch.from_numpy(np.ascontiguousarray(inp.omega)).cuda()
    g_host = np.random.default_rng(w.seed + 500).standard_normal((w.B, w.H, w.L, w.dv)).astype(np.float32)
    g = torch.from_numpy(g_host).cuda()
    dq = torch.empty((w.B, w.H, w.L, w.d), dtype=torch.float32, device="cuda")
    dk, dv = torch.empty_like(dq), torch.empty((w.B, w.H, w.L, w.dv), dtype=torch.float32, device="cuda")
    dw = torch.empty((w.H, w.m, w.d), dtype=torch.float32, device="cuda")
    flush = torch.empty(256 * 1024 * 1024 // 4, dtype=torch.int32, device="cuda")
    stream = torch.cuda.current_stream()

    def call(qq=q, kk=k, vv=v, gg=g):
        rc = fv.favor_attn_backward(qq, kk, vv, om, gg, dq, dk, dv, dw, w.B, w.H, w.L, w.d, w.dv, w.m,
                                    int(causal), 0, stream)
        if rc != fv.FAVOR_OK:
            raise fv.FavorError(rc, "favor_attn_backward")

    for _ in range(max(3, args.warmup)):
        call()
    torch.cuda.synchronize()
    sampler = ClockSampler(torch.cuda.current_device() if "CUDA_VISIBLE_DEVICES" not in os.environ
                           else os.environ["CUDA_VISIBLE_DEVICES"].split(",")[0])
    t_soak = time.time()
    while time.time() - t_soak < 1.0:
        call()
        torch.cuda.synchronize()
    evs = [(torch.cuda.Event(enable_timing=True), torch.cuda.Event(enable_timing=True)) for _ in range(args.steps)]
    torch.cuda.synchronize()
    t0 = time.time()
    for i in range(args.steps):
        flush.zero_()
        evs[i][0].record(stream)
        call()
        evs[i][1].record(stream)
    torch.cuda.synchronize()
    t1 = time.time()
    sampler.stop()
    st = fv.favor_get_device_status(stream)
    if st != fv.FAVOR_OK:
        raise fv.FavorError(st, "device status after the timed steps")
    ms = statistics.mean(a.elapsed_time(b) for a, b in evs)
    stat_steps = max(3, min(args.steps, 5))
    fv.favor_stats_enable(True)
    for _ in range(stat_steps):
        flush.zero_()
        call()
    torch.cuda.synchronize()
    stats = fv.favor_stats_read()
    fv.favor_stats_enable(False)
    dom_ms = stats.dominant_ms / max(1, stats.dominant_launches)
    tokens = w.B * w.H * w.L
    clocks = sampler.summary(t0, t1)
    props = torch.cuda.get_device_properties(torch.cuda.current_device())
    mhz = clocks.get("sm_max_mhz") or 2070.0
    peak = props.multi_processor_count * 128 * 2 * mhz * 1e6 / 1e12   # fp32 FMA lanes x 2 flops x clock
    achieved = bwd_chunk_flops_per_token(w, causal) * tokens / (dom_ms / 1000.0) / 1e12

    # end to end: q, k, v and dloss/dout from pinned host memory, the
    # gradients back to it, every step
    pin16 = lambda a: torch.from_numpy(np.ascontiguousarray(a).view(np.int16)).view(torch.bfloat16).pin_memory()
    hq, hk, hv = pin16(inp.q), pin16(inp.k), pin16(inp.v)
    hg = torch.from_numpy(g_host).pin_memory()
    hdq, hdk, hdv = (torch.empty(t.shape, dtype=torch.float32).pin_memory() for t in (dq, dk, dv))
    hdw = torch.empty(dw.shape, dtype=torch.float32).pin_memory()
    dq_in, dk_in, dv_in, dg_in = torch.empty_like(q), torch.empty_like(k), torch.empty_like(v), torch.empty_like(g)
    e2e_steps = max(3, min(args.steps, 10))
    torch.cuda.synchronize()
    te0 = time.perf_counter()
    for _ in range(e2e_steps):
        dq_in.copy_(hq, non_blocking=True)
        dk_in.copy_(hk, non_blocking=True)
        dv_in.copy_(hv, non_blocking=True)
        dg_in.copy_(hg, non_blocking=True)
        call(dq_in, dk_in, dv_in, dg_in)
        for h_, d_ in ((hdq, dq), (hdk, dk), (hdv, dv), (hdw, dw)):
            h_.copy_(d_, non_blocking=True)
        torch.cuda.current_stream().synchronize()
    te = (time.perf_counter() - te0) / e2e_steps
    h2d = (q.numel() + k.numel() + v.numel()) * 2 + g.numel() * 4
    d2h = (dq.numel() + dk.numel() + dv.numel() + dw.numel()) * 4
    line = {
        "metric": BWD_METRIC, "value": tokens / (ms / 1000.0), "unit": "tokens/s", "n_gpus": 1,
        "steps": args.steps, "warmup": args.warmup, "ms_per_step": ms, "higher_is_better": True,
        "scaling": "weak", "vs_baseline": None, "dtype": "f32", "data": "synthetic",
        "config": dict(describe(w, causal),
                       workload=(f"PROFILING CASE (first {w.H} heads, not a benchmark value) " if args.heads else "")
                       + f"{args.workload}: backward of " + describe(w, causal)["workload"],
                       inputs="bf16 q,k,v; fp32 omega, dloss/dout and gradients"),
        "roofline": {
            "bound": "alu", "achieved": achieved, "peak": peak, "unit": "TFLOP/s", "frac": achieved / peak,
            "traffic": None, "kernel": stats.dominant_kernel.decode() if stats.dominant_kernel else None,
            "kernel_ms": dom_ms, "peak_source": "derived: SMs x 128 fp32 lanes x 2 flops x max SM clock",
            "algorithmic_flops_per_token": bwd_chunk_flops_per_token(w, causal),
        },
        "e2e": {"value": tokens / te, "unit": "tokens/s", "h2d_bytes_per_step": h2d, "d2h_bytes_per_step": d2h},
        "gpu_launches": int(round(stats.kernel_launches / stat_steps * args.steps)),
        "clocks": clocks,
    }
    if not args.no_cpu_baseline:
        import oracle
        n = min(w.B * w.H, 2 * oracle.threads_used())
        Lc = 1024
        sel = lambda a: a.reshape(w.B * w.H, w.L, a.shape[-1])[:n, :Lc][None]
        t_c = time.perf_counter()
        oracle.backward(sel(inp.q32), sel(inp.k32), sel(inp.v32), inp.omega[[h % w.H for h in range(n)]],
                        sel(g_host).astype(np.float64), causal, 0)
        dt = time.perf_counter() - t_c
        line["cpu_baseline"] = {"value": n * Lc / dt, "unit": "tokens/s", "cores": oracle.threads_used(),
                                "kind": "oracle",
                                "sample": f"{n} heads x the first {Lc} tokens (float64 C oracle backward)"}
    print(json.dumps(line))
    return 0


def run_decode_reference(args):
    if int(os.environ.get("RANK", "0")) != 0:
        return 0
    base, B, L0 = DECODE[args.workload]
    w = workload(base)[0].with_(B=B)
    for _ in range(args.warmup):
        decode_cpu_baseline(w, 64, 50)
    times = [decode_cpu_baseline(w, 64, 50)["seconds"] for _ in range(args.steps)]
    ms = 1000 * statistics.mean(times) / 50
    value = 64 / (ms / 1000)
    print(json.dumps({
        "impl": "reference", "metric": DECODE_METRIC, "value": value, "unit": "tokens/s", "n_gpus": 0,
        "steps": args.steps, "warmup": args.warmup, "ms_per_step": ms, "higher_is_better": True,
        "scaling": "weak", "vs_baseline": None, "dtype": "f64", "data": "synthetic",
        "config": {"workload": f"{args.workload}: the oracle's decode step on 64 of {w.B * w.H} heads"},
        "cpu_baseline": {"value": value, "unit": "tokens/s", "cores": 1, "kind": "oracle",
                         "sample": "64 heads x 50 decode steps per step"},
        "e2e": {"value": value, "unit": "tokens/s", "h2d_bytes_per_step": 0, "d2h_bytes_per_step": 0},
    }))
    return 0


def run_backward_reference(args):
    if int(os.environ.get("RANK", "0")) != 0:
        return 0
    import numpy as np
    import oracle
    from favor_inputs import make_inputs
    w, causal = workload(BACKWARD[args.workload])
    n, Lc = min(w.B * w.H, oracle.threads_used()), 1024
    inp = make_inputs(w.with_(B=1, H=n, L=Lc))
    g = np.random.default_rng(1).standard_normal((1, n, Lc, w.dv))
    times = []
    for i in range(args.warmup + args.steps):
        t_c = time.perf_counter()
        oracle.backward(inp.q32, inp.k32, inp.v32, inp.omega, g, causal, 0)
        if i >= args.warmup:
            times.append(time.perf_counter() - t_c)
    ms = 1000 * statistics.mean(times)
    value = n * Lc / (ms / 1000)
    print(json.dumps({
        "impl": "reference", "metric": BWD_METRIC, "value": value, "unit": "tokens/s", "n_gpus": 0,
        "steps": args.steps, "warmup": args.warmup, "ms_per_step": ms, "higher_is_better": True,
        "scaling": "weak", "vs_baseline": None, "dtype": "f64", "data": "synthetic",
        "config": {"workload": f"{args.workload}: the oracle's backward on {n} heads x {Lc} tokens per step"},
        "cpu_baseline": {"value": value, "unit": "tokens/s", "cores": oracle.threads_used(), "kind": "oracle",
                         "sample": f"{n} heads x {Lc} tokens per step"},
        "e2e": {"value": value, "unit": "tokens/s", "h2d_bytes_per_step": 0, "d2h_bytes_per_step": 0},
    }))
    return 0


def run_decode(args):
    import numpy as np
    import torch
    from favor_random_feature_gb300 import build as fbuild
    fbuild.build()
    import favor_random_feature_gb300 as fv
    from favor_inputs import make_inputs

    if int(os.environ.get("WORLD_SIZE", "1")) != 1 or args.gpus != 1:
        raise SystemExit("decode workloads run on one GPU (replicas only)")
    base, B, L0 = DECODE[args.workload]
    w = workload(base)[0].with_(B=B)
    torch.cuda.set_device(int(os.environ.get("LOCAL_RANK", "0")))
    dev = lambda a: torch.from_numpy(np.ascontiguousarray(a).view(np.int16)).view(
        torch.bfloat16).cuda()
    prefix = make_inputs(w, L=L0)
    om = torch.from_numpy(np.ascontiguousarray(prefix.omega)).cuda()
    stream = torch.cuda.current_stream()
    per = fv.favor_state_floats(w.d, w.dv, w.m, 0)
    state = torch.empty((w.B, w.H, per), dtype=torch.float32, device="cuda")

    def check(rc, what):
        if rc != fv.FAVOR_OK:
            raise fv.FavorError(rc, what)

    check(fv.favor_attn_state(dev(prefix.k), dev(prefix.v), om, state, w.B, w.H, L0, w.d, w.dv, w.m, 0,
                              stream), "favor_attn_state")
    del prefix
    # a pool of new tokens, [T][B][H][.] on the device, used in turn
    T = 64
    tok = make_inputs(w.with_(seed=w.seed + 77), L=T)
    tq = dev(np.moveaxis(tok.q, 2, 0))
    tk = dev(np.moveaxis(tok.k, 2, 0))
    tv = dev(np.moveaxis(tok.v, 2, 0))
    out = torch.empty((w.B, w.H, w.dv), dtype=torch.float32, device="cuda")
    flush = torch.empty(256 * 1024 * 1024 // 4, dtype=torch.int32, device="cuda")
    step = [0]

    def call():
        t = step[0] % T
        step[0] += 1
        return fv.favor_attn_decode(tq[t], tk[t], tv[t], om, state, out, w.B, w.H, w.d, w.dv, w.m, 0,
                                    stream)

    for _ in range(max(3, args.warmup)):
        check(call(), "favor_attn_decode")
    torch.cuda.synchronize()
    sampler = ClockSampler(torch.cuda.current_device() if "CUDA_VISIBLE_DEVICES" not in os.environ
                           else os.environ["CUDA_VISIBLE_DEVICES"].split(",")[0])
    t_soak = time.time()
    while time.time() - t_soak < 1.0:
        flush.zero_()
        check(call(), "favor_attn_decode")
        torch.cuda.synchronize()
    evs = [(torch.cuda.Event(enable_timing=True), torch.cuda.Event(enable_timing=True))
           for _ in range(args.steps)]
    torch.cuda.synchronize()
    t0 = time.time()
    for i in range(args.steps):
        flush.zero_()
        evs[i][0].record(stream)
        check(call(), "favor_attn_decode")
        evs[i][1].record(stream)
    torch.cuda.synchronize()
    t1 = time.time()
    sampler.stop()
    st = fv.favor_get_device_status(stream)
    if st != fv.FAVOR_OK:
        raise fv.FavorError(st, "device status after the timed steps")
    ms = statistics.mean(a.elapsed_time(b) for a, b in evs)
    # the kernel's own time and the launch count, from separate steps
    stat_steps = max(3, min(args.steps, 10))
    fv.favor_stats_enable(True)
    for _ in range(stat_steps):
        flush.zero_()
        check(call(), "favor_attn_decode")
    torch.cuda.synchronize()
    stats = fv.favor_stats_read()
    fv.favor_stats_enable(False)
    dom_ms = stats.dominant_ms / max(1, stats.dominant_launches)
    launches_per_step = stats.kernel_launches / stat_steps
    heads = w.B * w.H
    kbytes = heads * decode_bytes_per_head(w)
    hbm_gbs, _, src = peaks()
    achieved = kbytes / (dom_ms / 1000.0) / 1e9

    # end to end: each step copies its token's q, k, v (packed in one pinned
    # host buffer: one copy) to the device, decodes, and reads out back
    nq, nv = w.B * w.H * w.d, w.B * w.H * w.dv
    flat = lambda a: np.ascontiguousarray(np.moveaxis(a, 2, 0)).reshape(T, -1)
    packed = np.concatenate([flat(tok.q), flat(tok.k), flat(tok.v)], axis=1)   # [T][2 nq + nv] bf16 bits
    hqkv = torch.from_numpy(np.ascontiguousarray(packed).view(np.int16)).view(torch.bfloat16).pin_memory()
    hout = torch.empty((w.B, w.H, w.dv), dtype=torch.float32).pin_memory()
    dqkv = torch.empty((2 * nq + nv,), dtype=torch.bfloat16, device="cuda")
    dq, dk, dvv = dqkv[:nq], dqkv[nq:2 * nq], dqkv[2 * nq:]
    e2e_steps = max(3, min(args.steps, 50))
    torch.cuda.synchronize()
    te0 = time.perf_counter()
    for i in range(e2e_steps):
        t = i % T
        dqkv.copy_(hqkv[t], non_blocking=True)
        check(fv.favor_attn_decode(dq, dk, dvv, om, state, out, w.B, w.H, w.d, w.dv, w.m, 0, stream),
              "favor_attn_decode")
        hout.copy_(out, non_blocking=True)
        torch.cuda.current_stream().synchronize()
    te = (time.perf_counter() - te0) / e2e_steps
    h2d = (2 * nq + nv) * 2
    line = {
        "metric": DECODE_METRIC, "value": heads / (ms / 1000.0), "unit": "tokens/s", "n_gpus": 1,
        "steps": args.steps, "warmup": args.warmup, "ms_per_step": ms, "higher_is_better": True,
        "scaling": "weak", "vs_baseline": None, "dtype": "f32", "data": "synthetic",
        "config": {
            "workload": f"{args.workload}: B={w.B} H={w.H} d={w.d} dv={w.dv} m={w.m} positive-features, "
                        f"state of a {L0}-token prefix, one new token per head per step",
            "B": w.B, "H": w.H, "d": w.d, "dv": w.dv, "m": w.m, "prefix": L0,
            "inputs": "bf16 q,k,v; fp32 omega, state and out",
            "l2": "flushed between steps (256 MiB write, outside the timed events)",
        },
        "roofline": {
            "bound": "hbm", "achieved": achieved, "peak": hbm_gbs, "unit": "GB/s",
            "frac": achieved / hbm_gbs, "traffic": measured_traffic("decode_step", args.workload),
            "kernel": stats.dominant_kernel.decode() if stats.dominant_kernel else None,
            "kernel_ms": dom_ms, "peak_source": src, "algorithmic_bytes_per_launch": kbytes,
        },
        "e2e": {"value": heads / te, "unit": "tokens/s", "h2d_bytes_per_step": h2d,
                "d2h_bytes_per_step": hout.numel() * 4},
        "gpu_launches": int(round(launches_per_step * args.steps)),
        "clocks": sampler.summary(t0, t1),
    }
    if not args.no_cpu_baseline:
        cb = decode_cpu_baseline(w, 64, 200)
        cb.pop("seconds", None)
        line["cpu_baseline"] = cb
    print(json.dumps(line))
    return 0


def main():
    ap = argparse.ArgumentParser()
    ap.add_argument("--gpus", type=int, default=1)
    ap.add_argument("--steps", type=int, default=50)
    ap.add_argument("--warmup", type=int, default=5)
    ap.add_argument("--impl", choices=["ours", "reference"], default="ours")
    ap.add_argument("--workload", default="causal8k",
                    choices=["causal8k", "nc4096", "long64k", "long64k_nc", "sweep16k", "sweep16k_m128", "sweep16k_m512",
                             "decode8k",
                             "decode_b256", "causal8k_bwd", "nc4096_bwd"])
    ap.add_argument("--no-cpu-baseline", action="store_true")
    ap.add_argument("--heads", type=int, default=0,
                    help="profiling case: the workload on its first N heads; "
                         "the line is marked and is not a benchmark value")
    args = ap.parse_args()
    if args.warmup < 3:
        args.warmup = 3
    if args.workload in BACKWARD:
        if args.impl == "reference":
            return run_backward_reference(args)
        return run_backward(args)
    if args.workload in DECODE:
        if args.impl == "reference":
            return run_decode_reference(args)
        return run_decode(args)
    if args.impl == "reference":
        return run_reference(args)
    return run_ours(args)


if __name__ == "__main__":
    sys.exit(main())
