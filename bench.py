#!/usr/bin/env python3
"""Benchmark of the Gated DeltaNet mixer hot path on GB300.

    python bench.py [--gpus N] [--steps K] [--warmup W] [--impl ours|reference]
                    [--workload batched|decode1|tree|prefill]

Prints ONE JSON line (rank 0).  The metric is GDN state updates per second
(head.tokens/s) with the achieved HBM bandwidth against the measured peak.

Workloads (27B head shape: 16 key heads, 48 value heads, d = 128):
  batched  (default) one step = conv + decode of one token for 64 sequences in
           each of 48 GDN layers (independent fp32 states, 9.66 GB).
  decode1  one step = conv + decode of one token, one layer, batch 1 (L2
           flushed between steps, as the other layers would evict the state).
  tree     one step = tree conv + verify of a 32-node draft tree + commit of a
           random root-to-leaf path, one layer.
  prefill  one step = chunked prefill of 8,192 tokens, one layer.

Multi-GPU: the path shards without any exchange (sequences, layers and heads
are independent), so N ranks run N independent replicas; value = all ranks'
head.tokens / the slowest rank's time ("scaling": "weak").
"""
from __future__ import annotations

import argparse
import ctypes
import hashlib
import json
import os
import statistics
import subprocess
import sys
import tempfile
import time

ROOT = os.path.dirname(os.path.abspath(__file__))
if ROOT not in sys.path:
    sys.path.insert(0, ROOT)

METRIC = "GDN state-updates/sec (head·tokens/s) and achieved HBM GB/s vs GB300 peak"
UNIT = "head·tokens/s"
FALLBACK_PEAKS = {"hbm_gbs": 6800.0, "bf16_tflops": 1900.0, "bf16_tflops_sustained": 1700.0}
NOMINAL_HBM_GBS = 8000.0

# 27B head shape
HK, HV, DK, DV = 16, 48, 128, 128
C_QKV = 2 * HK * DK + HV * DV


# ---------------------------------------------------------------------------
# host-side helpers (no GPU needed; covered by CPU tests)
# ---------------------------------------------------------------------------
def load_peaks() -> tuple[dict, str]:
    path = os.path.join(ROOT, "MEASURED_PEAKS.json")
    if os.path.exists(path):
        with open(path) as f:
            return json.load(f), "measured"
    return dict(FALLBACK_PEAKS), "fallback"


def dist_env() -> tuple[int, int, int]:
    return (int(os.environ.get("RANK", "0")), int(os.environ.get("WORLD_SIZE", "1")),
            int(os.environ.get("LOCAL_RANK", "0")))


def max_over_ranks(x: float, world: int, device=None) -> float:
    """Max of a per-rank float over all ranks (identity when world == 1)."""
    if world == 1:
        return float(x)
    import torch
    import torch.distributed as dist
    t = torch.tensor([float(x)], dtype=torch.float64, device=device)
    dist.all_reduce(t, op=dist.ReduceOp.MAX)
    return float(t.item())


def sum_over_ranks(x: float, world: int, device=None) -> float:
    if world == 1:
        return float(x)
    import torch
    import torch.distributed as dist
    t = torch.tensor([float(x)], dtype=torch.float64, device=device)
    dist.all_reduce(t, op=dist.ReduceOp.SUM)
    return float(t.item())


def barrier(world: int):
    if world > 1:
        import torch.distributed as dist
        dist.barrier()


def aggregate(units_per_rank: float, seconds_per_rank: float, world: int, device=None) -> dict:
    """Whole-job throughput: all ranks' units over the slowest rank's time."""
    t = max_over_ranks(seconds_per_rank, world, device)
    u = sum_over_ranks(units_per_rank, world, device)
    return {"seconds": t, "units": u, "value": u / t if t > 0 else 0.0}


def source_sha(files) -> str:
    h = hashlib.sha256()
    for f in files:
        with open(os.path.join(ROOT, f), "rb") as fh:
            h.update(fh.read())
    return h.hexdigest()[:16]


def ncu_traffic(kernel: str, sources) -> float | None:
    """DRAM bytes per launch from the committed ncu capture of `kernel`, or
    None when the kernel's sources changed since the counters were taken."""
    path = os.path.join(ROOT, "profiles", "traffic.json")
    if not os.path.exists(path):
        return None
    with open(path) as f:
        rec = json.load(f).get(kernel)
    if not rec or rec.get("source_sha") != source_sha(sources):
        return None
    return float(rec["bytes_per_launch"])


class ClockSampler:
    """nvidia-smi clocks / throttle reasons sampled during the timed region."""

    FIELDS = ("index,clocks.sm,clocks.max.sm,power.draw,clocks_event_reasons.active,"
              "clocks_event_reasons.hw_slowdown,clocks_event_reasons.hw_thermal_slowdown,"
              "clocks_event_reasons.sw_thermal_slowdown,clocks_event_reasons.sw_power_cap")

    def __init__(self, gpu_index: int):
        self.gpu_index = gpu_index
        self.proc = None
        self.file = None

    def start(self):
        try:
            self.file = tempfile.NamedTemporaryFile("w+", suffix=".csv", delete=False)
            self.proc = subprocess.Popen(
                ["nvidia-smi", f"--query-gpu={self.FIELDS}", "--format=csv,noheader,nounits",
                 "-lms", "50", "-i", str(self.gpu_index)],
                stdout=self.file, stderr=subprocess.DEVNULL)
        except (OSError, FileNotFoundError):
            self.proc = None

    def stop(self) -> dict:
        if self.proc is None:
            return {"sm_mhz": None, "sm_max_mhz": None, "reasons": [], "note": "nvidia-smi unavailable"}
        self.proc.terminate()
        try:
            self.proc.wait(timeout=5)
        except subprocess.TimeoutExpired:
            self.proc.kill()
        self.file.flush()
        self.file.seek(0)
        lines = [ln.strip() for ln in self.file.read().splitlines() if ln.strip()]
        self.file.close()
        os.unlink(self.file.name)
        return self.parse(lines)

    @staticmethod
    def parse(lines) -> dict:
        names = ["hw_slowdown", "hw_thermal_slowdown", "sw_thermal_slowdown", "sw_power_cap"]
        sm, smax, power, reasons = [], [], [], set()
        for ln in lines:
            parts = [p.strip() for p in ln.split(",")]
            if len(parts) < 9:
                continue
            try:
                sm.append(float(parts[1]))
                smax.append(float(parts[2]))
                power.append(float(parts[3]))
            except ValueError:
                continue
            for name, val in zip(names, parts[5:9]):
                if val.lower() == "active":
                    reasons.add(name)
        if not sm:
            return {"sm_mhz": None, "sm_max_mhz": None, "reasons": [], "samples": 0}
        return {"sm_mhz": statistics.median(sm), "sm_max_mhz": max(smax),
                "power_w_max": max(power), "reasons": sorted(reasons), "samples": len(sm)}


# ---------------------------------------------------------------------------
# workloads
# ---------------------------------------------------------------------------
DECODE_SOURCES = ["hybrid_linear_attention_conv_gb300/csrc/gdn_decode.cu",
                  "hybrid_linear_attention_conv_gb300/csrc/gdn_step.cuh",
                  "hybrid_linear_attention_conv_gb300/csrc/gdn_internal.h"]


def decode_bytes_per_launch(B: int, T: int = 1) -> int:
    """Algorithmic HBM bytes of one decode launch: the state read and written
    once, q/k/v read once (bf16), alpha/beta read (fp32), outputs written (fp32)."""
    state = B * HV * DV * DK * 4 * 2
    act = B * T * C_QKV * 2 + B * T * HV * 4 * 2 + B * T * HV * DV * 4
    return state + act


def conv_bytes_per_launch(B: int, T: int = 1) -> int:
    """x read, taps read, the 4-entry tail read and rewritten, y written (bf16)."""
    return B * T * C_QKV * 2 + C_QKV * 4 * 2 + 2 * B * 4 * C_QKV * 2 + B * T * C_QKV * 2


class Batched:
    """48 GDN layers x 64 sequences, one token per sequence per layer."""

    name = "batched"
    L, B = 48, 64

    def __init__(self, device, seed: int, n_sets: int, layers: int = 48):
        self.L = layers
        import torch
        from hybrid_linear_attention_conv_gb300 import gdn
        self.torch, self.gdn = torch, gdn
        self.lib = gdn.load()
        L, B = self.L, self.B
        g = torch.Generator(device=device)
        g.manual_seed(seed)
        bf = torch.bfloat16
        self.state = torch.randn((L, B, HV, DV, DK), generator=g, device=device, dtype=torch.float32)
        self.state.mul_(0.1)
        self.w = (0.5 * torch.randn((L, C_QKV, 4), generator=g, device=device)).to(bf)
        self.tail = torch.randn((L, B, 4, C_QKV), generator=g, device=device).to(bf)
        self.n_sets = n_sets
        self.x = torch.randn((n_sets, L, B, 1, C_QKV), generator=g, device=device).to(bf)
        self.alpha = 0.9 + 0.1 * torch.rand((n_sets, L, B, 1, HV), generator=g, device=device)
        self.beta = torch.sigmoid(torch.randn((n_sets, L, B, 1, HV), generator=g, device=device))
        self.y = torch.empty((B, 1, C_QKV), dtype=bf, device=device)
        self.out = torch.empty((L, B, 1, HV, DV), dtype=torch.float32, device=device)
        self.shape = gdn.gdn_shape(B, HK, HV, DK, DV)
        self.stream = torch.cuda.current_stream()
        sp = ctypes.c_void_p(self.stream.cuda_stream)
        P = ctypes.c_void_p
        self.args = []
        for s in range(n_sets):
            per = []
            for l in range(L):
                conv = (B, 1, C_QKV, None, P(self.x[s, l].data_ptr()), P(self.w[l].data_ptr()),
                        P(self.tail[l].data_ptr()), P(self.y.data_ptr()), 0, sp)
                dec = (ctypes.byref(self.shape), 1, P(self.y.data_ptr()), P(self.alpha[s, l].data_ptr()),
                       P(self.beta[s, l].data_ptr()), P(self.state[l].data_ptr()),
                       P(self.out[l].data_ptr()), 1.0, gdn.GDN_NORMALIZE_QK, sp)
                per.append((conv, dec))
            self.args.append(per)
        self.launches_per_step = 2 * L
        self.units_per_step = L * B * HV  # head.tokens
        self.dominant = "gdn_decode_kernel"
        self.dominant_bytes = decode_bytes_per_launch(B)
        self.step_bytes = L * (decode_bytes_per_launch(B) + conv_bytes_per_launch(B))

    def step(self, i: int, events=None):
        """Enqueue step i; events (list of 2L+1) are recorded around each kernel."""
        lib = self.lib
        conv_fn, dec_fn = lib.gdn_conv_step, lib.gdn_decode_step
        if events is not None:
            events[0].record(self.stream)
        for l, (conv, dec) in enumerate(self.args[i % self.n_sets]):
            rc = conv_fn(*conv)
            if events is not None:
                events[2 * l + 1].record(self.stream)
            rc |= dec_fn(*dec)
            if events is not None:
                events[2 * l + 2].record(self.stream)
            if rc != 0:
                raise RuntimeError(f"gdn call failed: {self.gdn.last_error()}")

    def dominant_ms(self, events) -> list:
        """Durations of the decode launches of one instrumented step."""
        return [events[2 * l + 1].elapsed_time(events[2 * l + 2]) for l in range(self.L)]

    # end-to-end: inputs from pinned host memory, outputs back to the host
    def e2e_setup(self):
        torch = self.torch
        self.h_x = torch.empty(self.x[0].shape, dtype=self.x.dtype, pin_memory=True)
        self.h_x.copy_(self.x[0])
        self.h_a = torch.empty(self.alpha[0].shape, dtype=torch.float32, pin_memory=True)
        self.h_a.copy_(self.alpha[0])
        self.h_b = torch.empty(self.beta[0].shape, dtype=torch.float32, pin_memory=True)
        self.h_b.copy_(self.beta[0])
        self.h_out = torch.empty(self.out.shape, dtype=torch.float32, pin_memory=True)
        self.e2e_h2d = (self.h_x.numel() * 2 + self.h_a.numel() * 4 + self.h_b.numel() * 4)
        self.e2e_d2h = self.h_out.numel() * 4

    def e2e_step(self, i: int):
        self.x[0].copy_(self.h_x, non_blocking=True)
        self.alpha[0].copy_(self.h_a, non_blocking=True)
        self.beta[0].copy_(self.h_b, non_blocking=True)
        for conv, dec in self.args[0]:
            if self.lib.gdn_conv_step(*conv) | self.lib.gdn_decode_step(*dec):
                raise RuntimeError(self.gdn.last_error())
        self.h_out.copy_(self.out, non_blocking=True)

    def config(self=None) -> dict:
        L = Batched.L if self is None else self.L
        B = Batched.B
        sb = L * B * HV * DV * DK * 4
        return {"workload": f"batched decode over {L} GDN layers: batch {B} sequences, 27B head "
                            "shape (16 key / 48 value heads x 128), independent fp32 states, one token "
                            "per sequence per layer (conv + delta step)",
                "layers": L, "batch": B, "Hk": HK, "Hv": HV, "dk": DK, "dv": DV,
                "state_bytes": sb,
                "l2": f"inputs larger than L2: {sb / 1e9:.2f} GB of state streamed per step",
                "launch": "eager, CUDA events between kernels"}


def cpu_oracle_sample(seconds: float = 10.0) -> dict:
    """The oracle as it stands: conv + decode of one sequence, one layer, one
    token (48 head.tokens) at the 27B shape, repeated for about `seconds`."""
    import numpy as np
    import oracle
    from hybrid_linear_attention_conv_gb300 import inputs as gen
    s = gen.QWEN_27B
    c = gen.conv_inputs(0, 1, 1, s.C)
    d = gen.decode_inputs(0, s, 1)
    state = d["state"].astype(np.float64)
    n = 0
    t0 = time.perf_counter()
    while True:
        y, _ = oracle.conv_linear(c["x"], c["w"], c["tail"])
        _, state = oracle.decode(oracle.f64_to_bf16(y), d["alpha"], d["beta"], state, s.Hk, s.Hv, s.dk, s.dv)
        n += 1
        el = time.perf_counter() - t0
        if el >= seconds:
            break
    return {"value": n * s.Hv / el, "unit": UNIT, "cores": 1, "kind": "oracle",
            "sample": f"{n} x (conv + decode of 1 sequence x 1 layer x 1 token, 48 value heads, 27B "
                      f"head shape), fp64 C oracle, single thread, {el:.1f} s"}


# ---------------------------------------------------------------------------
# arms
# ---------------------------------------------------------------------------
def run_ours(args) -> dict | None:
    import torch
    rank, world, local = dist_env()
    if world > 1:
        import torch.distributed as dist
        dist.init_process_group("nccl")
    torch.cuda.set_device(local)
    device = torch.device("cuda", local)

    import __graft_entry__
    __graft_entry__.build()

    peaks, peaks_kind = load_peaks()
    wl = Batched(device, seed=1234 + rank, n_sets=min(4, args.steps + args.warmup), layers=args.layers)
    torch.cuda.synchronize()

    for i in range(args.warmup):
        wl.step(i)
    torch.cuda.synchronize()

    # timed region: K steps, an event after every kernel
    evs = [[torch.cuda.Event(enable_timing=True) for _ in range(wl.launches_per_step + 1)]
           for _ in range(args.steps)]
    clocks = ClockSampler(local)
    clocks.start()
    time.sleep(0.2)
    barrier(world)
    torch.cuda.synchronize()
    for i in range(args.steps):
        wl.step(args.warmup + i, evs[i])
    torch.cuda.synchronize()
    barrier(world)
    clk = clocks.stop()
    step_ms = [evs[i][0].elapsed_time(evs[i][-1]) for i in range(args.steps)]
    total_s = evs[0][0].elapsed_time(evs[-1][-1]) / 1e3
    dom_ms = [d for i in range(args.steps) for d in wl.dominant_ms(evs[i])]
    agg = aggregate(wl.units_per_step * args.steps, total_s, world, device)

    # end-to-end through the API with host buffers
    wl.e2e_setup()
    for i in range(2):
        wl.e2e_step(i)
    torch.cuda.synchronize()
    barrier(world)
    t0 = time.perf_counter()
    e0 = torch.cuda.Event(enable_timing=True)
    e1 = torch.cuda.Event(enable_timing=True)
    e0.record()
    for i in range(args.steps):
        wl.e2e_step(i)
    e1.record()
    torch.cuda.synchronize()
    e2e_s = max(e0.elapsed_time(e1) / 1e3, time.perf_counter() - t0)
    e2e = aggregate(wl.units_per_step * args.steps, e2e_s, world, device)

    if rank != 0:
        return None

    dom_avg_s = statistics.mean(dom_ms) / 1e3
    achieved = wl.dominant_bytes / dom_avg_s / 1e9
    peak = float(peaks["hbm_gbs"])
    traffic = ncu_traffic(wl.dominant, DECODE_SOURCES)
    step_gbs = wl.step_bytes * args.steps / total_s / 1e9
    line = {
        "metric": METRIC,
        "value": agg["value"],
        "unit": UNIT,
        "n_gpus": world,
        "steps": args.steps,
        "warmup": args.warmup,
        "ms_per_step": statistics.mean(step_ms),
        "higher_is_better": True,
        "scaling": "weak",
        "vs_baseline": None,
        "dtype": "f32",
        "data": "synthetic (seeded device RNG; 27B head shape, random-init states)",
        "config": wl.config(),
        "hbm_gbs_step": step_gbs,
        "hbm_frac_step": step_gbs / peak,
        "hbm_frac_step_nominal_8tbs": step_gbs / NOMINAL_HBM_GBS,
        "roofline": {"bound": "hbm", "kernel": wl.dominant, "achieved": achieved, "peak": peak,
                     "unit": "GB/s", "frac": achieved / peak, "peak_kind": peaks_kind,
                     "frac_nominal_8tbs": achieved / NOMINAL_HBM_GBS,
                     "bytes_per_launch": wl.dominant_bytes, "avg_launch_us": dom_avg_s * 1e6,
                     "traffic": traffic},
        "clocks": clk,
        "e2e": {"value": e2e["value"], "unit": UNIT, "h2d_bytes_per_step": wl.e2e_h2d,
                "d2h_bytes_per_step": wl.e2e_d2h, "ms_per_step": e2e_s * 1e3 / args.steps},
        "gpu_launches": wl.launches_per_step * args.steps,
    }
    if world == 1 and not args.no_cpu_baseline:
        line["cpu_baseline"] = cpu_oracle_sample(args.cpu_seconds)
    return line


def run_reference(args) -> dict | None:
    rank, world, _ = dist_env()
    if rank != 0:
        return None
    import numpy as np
    import oracle
    from hybrid_linear_attention_conv_gb300 import inputs as gen
    oracle.build()
    s = gen.QWEN_27B
    c = gen.conv_inputs(0, 1, 1, s.C)
    d = gen.decode_inputs(0, s, 1)
    state = d["state"].astype(np.float64)

    def one():
        nonlocal state
        y, _ = oracle.conv_linear(c["x"], c["w"], c["tail"])
        _, state = oracle.decode(oracle.f64_to_bf16(y), d["alpha"], d["beta"], state, s.Hk, s.Hv, s.dk, s.dv)

    for _ in range(args.warmup):
        one()
    t0 = time.perf_counter()
    for _ in range(args.steps):
        one()
    el = time.perf_counter() - t0
    value = args.steps * s.Hv / el
    sample = (f"each step: conv + decode of 1 sequence x 1 layer x 1 token (48 head.tokens) of the "
              f"batched workload, fp64 C oracle, single thread")
    return {
        "impl": "reference",
        "metric": METRIC, "value": value, "unit": UNIT, "n_gpus": world, "steps": args.steps,
        "warmup": args.warmup, "ms_per_step": el * 1e3 / args.steps, "higher_is_better": True,
        "scaling": "weak", "vs_baseline": None, "dtype": "f64", "data": "synthetic",
        "config": Batched.config(),
        "cpu_baseline": {"value": value, "unit": UNIT, "cores": 1, "kind": "oracle", "sample": sample},
        "e2e": {"value": value, "unit": UNIT, "h2d_bytes_per_step": 0, "d2h_bytes_per_step": 0},
    }


def main(argv=None):
    ap = argparse.ArgumentParser(description=__doc__, formatter_class=argparse.RawDescriptionHelpFormatter)
    ap.add_argument("--gpus", type=int, default=1)
    ap.add_argument("--steps", type=int, default=100)
    ap.add_argument("--warmup", type=int, default=5)
    ap.add_argument("--impl", choices=["ours", "reference"], default="ours")
    ap.add_argument("--workload", choices=["batched"], default="batched")
    ap.add_argument("--layers", type=int, default=48,
                    help="GDN layers in the batched workload (48 = the 27B model; fewer only for "
                         "profiling small cases)")
    ap.add_argument("--cpu-seconds", type=float, default=10.0)
    ap.add_argument("--no-cpu-baseline", action="store_true")
    args = ap.parse_args(argv)
    args.warmup = max(3, args.warmup)  # at least three untimed warm-up steps
    line = run_reference(args) if args.impl == "reference" else run_ours(args)
    if line is not None:
        print(json.dumps(line), flush=True)
    if dist_env()[1] > 1 and args.impl == "ours":
        import torch.distributed as dist
        dist.destroy_process_group()


if __name__ == "__main__":
    main()
