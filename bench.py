#!/usr/bin/env python3
"""Benchmark of the Gated DeltaNet mixer hot path on GB300.

    python bench.py [--gpus N] [--steps K] [--warmup W] [--impl ours|reference]
                    [--workload batched|decode1|tree|treebatch|prefill|...]

Prints ONE JSON line (rank 0).  The metric is GDN state updates per second
(head.tokens/s) with the achieved HBM bandwidth against the measured peak.
With no --workload, the line is the batched decode (the headline) and, under
the key "workloads", the other single-GPU configs measured in the same run:
decode1, tree and prefill, each with its own roofline, e2e and CPU baseline.

Workloads (27B head shape: 16 key heads, 48 value heads, d = 128):
  batched  (default) one step = conv + decode of one token for 64 sequences in
           each of 48 GDN layers (independent fp32 states, 9.66 GB).
  decode1  one step = conv + decode of one token, one layer, batch 1; L2 is
           flushed between steps (the other layers evict the state in a real
           decode) and the flush is outside the timed intervals.
  tree     one step = tree conv + verify of a 32-node draft tree + commit of a
           random root-to-leaf path, one layer (L2 flushed between steps).
  prefill  one step = chunked prefill of 8,192 tokens, one layer.

Timing: CUDA events on the launching stream after every kernel of a step, so
the same timed region gives the step time and each kernel's launch duration.

Multi-GPU: the path shards without any exchange (sequences, layers and heads
are independent), so N ranks run N independent replicas; value = all ranks'
head.tokens / the slowest rank's time ("scaling": "weak").
"""
from __future__ import annotations

import argparse
import ctypes
import hashlib
import json
import math
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
FALLBACK_PEAKS = {"hbm_gbs": 6800.0, "bf16_tflops": 1900.0, "bf16_tflops_sustained": 1700.0,
                  "sm_max_mhz": 2070.0}
NOMINAL_HBM_GBS = 8000.0
SMS = 152               # GB300 streaming multiprocessors
FP32_LANES_PER_SM = 128  # fp32 FMA lanes per SM

# 27B head shape
HK, HV, DK, DV = 16, 48, 128, 128
C_QKV = 2 * HK * DK + HV * DV
CHUNK = 64


# ---------------------------------------------------------------------------
# host-side helpers (no GPU needed; covered by CPU tests)
# ---------------------------------------------------------------------------
def load_peaks() -> tuple[dict, str]:
    path = os.path.join(ROOT, "MEASURED_PEAKS.json")
    if os.path.exists(path):
        with open(path) as f:
            return json.load(f), "measured"
    return dict(FALLBACK_PEAKS), "fallback"


def fp32_alu_peak_tflops(sm_mhz: float) -> float:
    """FP32 CUDA-core peak: SMs x fp32 lanes x 2 flops (FMA) x clock."""
    return SMS * FP32_LANES_PER_SM * 2 * sm_mhz * 1e6 / 1e12


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
# algorithmic work per launch (what the roofline divides by)
# ---------------------------------------------------------------------------
def decode_bytes_per_launch(B: int, T: int = 1) -> int:
    """HBM bytes of one decode launch: the state read and written once, q/k/v
    read once (bf16), alpha/beta read (fp32), outputs written (fp32)."""
    state = B * HV * DV * DK * 4 * 2
    act = B * T * C_QKV * 2 + B * T * HV * 4 * 2 + B * T * HV * DV * 4
    return state + act


def conv_bytes_per_launch(B: int, T: int = 1) -> int:
    """x read, taps read, the 4-entry tail read and rewritten, y written (bf16)."""
    return B * T * C_QKV * 2 + C_QKV * 4 * 2 + 2 * B * 4 * C_QKV * 2 + B * T * C_QKV * 2


def fused_bytes_per_launch(B: int, T: int = 1) -> int:
    """HBM bytes of one fused conv + decode launch: the state read and written
    once, x read (bf16), the last three tail inputs read and the four-input
    tail written (bf16), the taps, alpha/beta (fp32) and the outputs (fp32)."""
    state = B * HV * DV * DK * 4 * 2
    conv = B * T * C_QKV * 2 + B * 3 * C_QKV * 2 + B * 4 * C_QKV * 2 + C_QKV * 4 * 2
    gates_out = B * T * HV * 4 * 2 + B * T * HV * DV * 4
    return state + conv + gates_out


def kda_fused_bytes_per_launch(B: int, T: int = 1) -> int:
    """As fused_bytes_per_launch with a decay per key channel: alpha is dk
    fp32 values per head and token instead of one."""
    return fused_bytes_per_launch(B, T) + B * T * HV * (DK - 1) * 4


def step_flops_per_head_token() -> int:
    """fp32 flops of one state update of one head: s.k and s.q (2 x 2d per
    row), alpha s + u k (2d per row), the row scalars u and o (5 per row)."""
    return DV * (6 * DK + 5)


def prefill_flops(T: int) -> int:
    """Algorithmic flops of the chunk form over T tokens (chunk 64): per value
    head and chunk, S k and S q (2 x 2.64.d.d), T X and P U (2 x 2.64.64.d),
    the state update (2.d.d.64) and the triangular solve (64^3/3); per key head
    and chunk, K K^T and Q K^T (2 x 2.64.64.d)."""
    n = (T + CHUNK - 1) // CHUNK
    per_v = 2 * 2 * CHUNK * DV * DK + 2 * 2 * CHUNK * CHUNK * DV + 2 * DV * DK * CHUNK + CHUNK ** 3 // 3
    per_k = 2 * 2 * CHUNK * CHUNK * DK
    return n * (HV * per_v + HK * per_k)


def prefill_bytes(T: int) -> int:
    """q, k, v read once (bf16), alpha/beta read, outputs written (fp32), the
    state read and written once."""
    return T * C_QKV * 2 + T * HV * 8 + T * HV * DV * 4 + 2 * HV * DV * DK * 4


DECODE_SOURCES = ["hybrid_linear_attention_conv_gb300/csrc/gdn_decode.cu",
                  "hybrid_linear_attention_conv_gb300/csrc/gdn_step.cuh",
                  "hybrid_linear_attention_conv_gb300/csrc/gdn_internal.h"]
FUSED_SOURCES = DECODE_SOURCES + ["hybrid_linear_attention_conv_gb300/csrc/gdn_conv.cuh"]
PREFILL_SOURCES = ["hybrid_linear_attention_conv_gb300/csrc/gdn_prefill.cu",
                   "hybrid_linear_attention_conv_gb300/csrc/gdn_tc.cuh",
                   "hybrid_linear_attention_conv_gb300/csrc/gdn_internal.h"]


# ---------------------------------------------------------------------------
# workloads
# ---------------------------------------------------------------------------
class Recorder:
    """CUDA events recorded on the launching stream after every kernel."""

    def __init__(self, torch, stream, marks_per_step: int, steps: int):
        self.stream = stream
        self.events = [[torch.cuda.Event(enable_timing=True) for _ in range(marks_per_step + 1)]
                       for _ in range(steps)]
        self.names = [[None] * (marks_per_step + 1) for _ in range(steps)]
        self.i = -1
        self.k = 0

    def begin(self, i: int):
        """Start the next timed step (`i` is the workload's own step number)."""
        self.i, self.k = self.i + 1, 0
        self.events[self.i][0].record(self.stream)

    def mark(self, name: str):
        self.k += 1
        self.names[self.i][self.k] = name
        self.events[self.i][self.k].record(self.stream)

    def step_ms(self) -> list:
        return [ev[0].elapsed_time(ev[-1]) for ev in self.events]

    def kernel_ms(self, name: str) -> list:
        out = []
        for ev, nm in zip(self.events, self.names):
            for k in range(1, len(ev)):
                if nm[k] == name:
                    out.append(ev[k - 1].elapsed_time(ev[k]))
        return out


class _Marks:
    """Events e[1], e[2], ... recorded on `stream` at each mark of one step
    (the caller records e[0] before the step)."""

    def __init__(self, events, stream):
        self.events, self.stream, self.k = events, stream, 0

    def mark(self, name: str):
        self.k += 1
        self.events[self.k].record(self.stream)


def _call(fn, args, gdn):
    rc = fn(*args)
    if rc != 0:
        raise RuntimeError(f"{fn.__name__} failed: {gdn.last_error()}")


class Workload:
    """Common plumbing: device inputs, the stream, optional L2 flush."""

    flush = False
    launches_per_step = 0
    units_per_step = 0

    @property
    def marks_per_step(self) -> int:
        """CUDA events recorded per step after the first (one per marked call)."""
        return self.launches_per_step

    def __init__(self, device, seed: int):
        import torch
        from hybrid_linear_attention_conv_gb300 import gdn
        self.torch, self.gdn, self.lib = torch, gdn, gdn.load()
        self.device = device
        self.gen = torch.Generator(device=device)
        self.gen.manual_seed(seed)
        self.stream = torch.cuda.current_stream()
        self.sp = ctypes.c_void_p(self.stream.cuda_stream)
        self.flush_buf = None
        if self.flush:
            # 256 MB > the 129 MB L2: writing it evicts the previous step's lines
            self.flush_buf = torch.empty(64 * 1024 * 1024, dtype=torch.float32, device=device)

    def randn(self, shape, scale=1.0, dtype=None):
        t = self.torch.randn(shape, generator=self.gen, device=self.device)
        if scale != 1.0:
            t.mul_(scale)
        return t.to(dtype) if dtype is not None else t

    def gates(self, shape):
        torch = self.torch
        a = 0.9 + 0.1 * torch.rand(shape, generator=self.gen, device=self.device)
        b = torch.sigmoid(torch.randn(shape, generator=self.gen, device=self.device))
        return a, b

    def pre_step(self):
        if self.flush_buf is not None:
            self.flush_buf.zero_()

    def e2e_copy(self, dst, src):
        dst.copy_(src, non_blocking=True)

    def e2e_pack(self, hosts):
        """The small per-step inputs `hosts` (CPU tensors) packed back to back,
        each at a 16-byte boundary, into one pinned host buffer and one device
        buffer, so that a step moves them with one copy instead of one per
        tensor (for a few KB the copy's fixed cost dominates).  Returns the
        device views, shaped and typed like `hosts`."""
        torch = self.torch
        offs, n = [], 0
        for h in hosts:
            offs.append(n)
            n += (h.numel() * h.element_size() + 15) // 16 * 16
        self.e2e_hbuf = torch.zeros(n, dtype=torch.uint8, pin_memory=True)
        self.e2e_dbuf = torch.empty(n, dtype=torch.uint8, device=self.device)
        views = []
        for h, o in zip(hosts, offs):
            nb = h.numel() * h.element_size()
            self.e2e_hbuf[o:o + nb].copy_(h.contiguous().reshape(-1).view(torch.uint8))
            views.append(self.e2e_dbuf[o:o + nb].view(h.dtype).view(h.shape))
        return views

    def e2e_streams(self):
        """Copy streams of the overlapped end-to-end step: host->device and
        device->host copies run on their own streams, ordered against the
        compute stream by events, so that piece p's inputs arrive while piece
        p - 1 computes and its outputs leave while piece p + 1 computes."""
        torch = self.torch
        self.s_in = torch.cuda.Stream(device=self.device)
        self.s_out = torch.cuda.Stream(device=self.device)

    def e2e_pipeline(self, pieces, inputs, outputs, compute):
        """One end-to-end step in pieces: for piece k, copy inputs(k) in on
        s_in, run compute(k) on the current stream, copy outputs(k) out on
        s_out.  The step ends on the current stream once the last copy out
        has landed, so events on it bracket every copy."""
        torch = self.torch
        cs = torch.cuda.current_stream()
        start = torch.cuda.Event()
        start.record(cs)
        self.s_in.wait_event(start)
        self.s_out.wait_event(start)
        for k in range(pieces):
            with torch.cuda.stream(self.s_in):
                for dst, src in inputs(k):
                    dst.copy_(src, non_blocking=True)
                ev_in = torch.cuda.Event()
                ev_in.record(self.s_in)
            cs.wait_event(ev_in)
            compute(k)
            ev_c = torch.cuda.Event()
            ev_c.record(cs)
            with torch.cuda.stream(self.s_out):
                self.s_out.wait_event(ev_c)
                for dst, src in outputs(k):
                    dst.copy_(src, non_blocking=True)
        done = torch.cuda.Event()
        done.record(self.s_out)
        cs.wait_event(done)


class Batched(Workload):
    """48 GDN layers x 64 sequences, one token per sequence per layer."""

    name = "batched"
    kda = False
    L, B = 48, 64

    def __init__(self, device, seed: int, steps: int, layers: int = 48):
        super().__init__(device, seed)
        self.L = layers
        torch, gdn = self.torch, self.gdn
        L, B = self.L, self.B
        bf = torch.bfloat16
        self.state = self.randn((L, B, HV, DV, DK), 0.1)
        self.w = self.randn((L, C_QKV, 4), 0.5, bf)
        self.tail = self.randn((L, B, 4, C_QKV), 1.0, bf)
        self.n_sets = min(4, steps)
        self.x = self.randn((self.n_sets, L, B, 1, C_QKV), 1.0, bf)
        self.alpha, self.beta = self.gates((self.n_sets, L, B, 1, HV))
        if self.kda:
            self.alpha = 0.9 + 0.1 * torch.rand((self.n_sets, L, B, 1, HV, DK), generator=self.gen,
                                                device=device)
        self.fn = self.lib.gdn_kda_conv_decode_step if self.kda else self.lib.gdn_conv_decode_step
        self.out = torch.empty((L, B, 1, HV, DV), dtype=torch.float32, device=device)
        self.shape = gdn.gdn_shape(B, HK, HV, DK, DV)
        self._extra_inputs()
        self.args = [[self._args(s, l, self.sp) for l in range(L)] for s in range(self.n_sets)]
        self.launches_per_step = L
        self.units_per_step = L * B * HV
        self.dominant = "gdn_conv_decode_kernel[kda]" if self.kda else "gdn_conv_decode_kernel"
        self.dominant_sources = FUSED_SOURCES
        self.bound = "hbm"
        per_launch = kda_fused_bytes_per_launch(B) if self.kda else fused_bytes_per_launch(B)
        self.dominant_work = per_launch
        self.step_bytes = L * per_launch

    def _extra_inputs(self):
        """Inputs beyond the fused step's (the layer step's projections and parameters)."""

    def _args(self, s: int, l: int, sp):
        """C-ABI arguments of layer l's launch with input set s on stream sp."""
        P = ctypes.c_void_p
        tl = P(self.tail[l].data_ptr())
        return (ctypes.byref(self.shape), 1, P(self.x[s, l].data_ptr()), P(self.w[l].data_ptr()), tl, tl,
                P(self.alpha[s, l].data_ptr()), P(self.beta[s, l].data_ptr()), P(self.state[l].data_ptr()),
                P(self.out[l].data_ptr()), 1.0, self.gdn.GDN_NORMALIZE_QK, sp)

    def _launch_all(self, s: int, sp):
        for l in range(self.L):
            _call(self.fn, self._args(s, l, sp), self.gdn)

    def capture(self):
        """One CUDA graph per input set holding the step's L launches (the
        pages' engine captures its decode launches the same way)."""
        torch = self.torch
        self.graphs = []
        for s in range(self.n_sets):
            g = torch.cuda.CUDAGraph()
            with torch.cuda.graph(g):
                self._launch_all(s, ctypes.c_void_p(torch.cuda.current_stream().cuda_stream))
            self.graphs.append(g)
        torch.cuda.synchronize()

    @property
    def marks_per_step(self) -> int:
        return 1 if getattr(self, "graphs", None) else self.launches_per_step

    def step(self, i: int, rec: Recorder | None = None):
        lib, gdn = self.lib, self.gdn
        if rec:
            rec.begin(i)
        if getattr(self, "graphs", None):
            self.graphs[i % self.n_sets].replay()
            if rec:
                rec.mark("step")
            return
        for args in self.args[i % self.n_sets]:
            _call(self.fn, args, gdn)
            if rec:
                rec.mark(self.dominant)

    def dominant_ms(self, rec: Recorder) -> list:
        """Per-launch durations: measured per kernel in eager mode; in graph
        mode the step time spread over its L launches (an upper bound, since it
        includes any gap between launches)."""
        if getattr(self, "graphs", None):
            return [ms / self.L for ms in rec.step_ms()]
        return rec.kernel_ms(self.dominant)

    E2E_PIECES = 8  # layer groups of the overlapped end-to-end step

    def e2e_pairs(self):
        """(device, pinned host) pairs of a step's inputs, and (host, device)
        of its result; every tensor has the layer as its first dimension."""
        torch = self.torch
        self.h_x = self.x[0].cpu().pin_memory()
        self.h_a = self.alpha[0].cpu().pin_memory()
        self.h_b = self.beta[0].cpu().pin_memory()
        self.h_out = torch.empty(self.out.shape, dtype=torch.float32, pin_memory=True)
        return [(self.x[0], self.h_x), (self.alpha[0], self.h_a), (self.beta[0], self.h_b)], \
               [(self.h_out, self.out)]

    def e2e_setup(self):
        torch = self.torch
        self.e2e_in, self.e2e_out = self.e2e_pairs()
        self.e2e_h2d = sum(src.numel() * src.element_size() for _, src in self.e2e_in)
        self.e2e_d2h = sum(dst.numel() * dst.element_size() for dst, _ in self.e2e_out)
        self.e2e_streams()
        n = self.E2E_PIECES
        per = (self.L + n - 1) // n
        self.e2e_groups = [(l0, min(l0 + per, self.L)) for l0 in range(0, self.L, per)]
        # one CUDA graph per layer group (eager launches under --eager)
        self.e2e_graphs = []
        if getattr(self, "graphs", None):
            for l0, l1 in self.e2e_groups:
                g = torch.cuda.CUDAGraph()
                with torch.cuda.graph(g):
                    sp = ctypes.c_void_p(torch.cuda.current_stream().cuda_stream)
                    for l in range(l0, l1):
                        _call(self.fn, self._args(0, l, sp), self.gdn)
                self.e2e_graphs.append(g)
            torch.cuda.synchronize()

    def e2e_step(self, i: int):
        groups = self.e2e_groups

        def compute(k):
            if self.e2e_graphs:
                self.e2e_graphs[k].replay()
            else:
                l0, l1 = groups[k]
                for l in range(l0, l1):
                    _call(self.fn, self.args[0][l], self.gdn)

        self.e2e_pipeline(len(groups),
                          lambda k: [(d[groups[k][0]:groups[k][1]], h[groups[k][0]:groups[k][1]])
                                     for d, h in self.e2e_in],
                          lambda k: [(h[groups[k][0]:groups[k][1]], d[groups[k][0]:groups[k][1]])
                                     for h, d in self.e2e_out],
                          compute)

    def config(self=None) -> dict:
        L = Batched.L if self is None else self.L
        B = Batched.B
        sb = L * B * HV * DV * DK * 4
        return {"workload": f"batched decode over {L} GDN layers: batch {B} sequences, 27B head "
                            "shape (16 key / 48 value heads x 128), independent fp32 states, one token "
                            "per sequence per layer (fused conv + delta step, one launch per layer)",
                "layers": L, "batch": B, "Hk": HK, "Hv": HV, "dk": DK, "dv": DV, "state_bytes": sb,
                "l2": f"inputs larger than L2: {sb / 1e9:.2f} GB of state streamed per step",
                "launch": ("eager, CUDA events after every kernel" if self is not None and not
                           getattr(self, "graphs", None) else
                           f"one CUDA graph per step ({L} launches), CUDA events around each replay")}


def layer_bytes_per_launch(B: int, T: int = 1) -> int:
    """HBM bytes of one layer decode launch: the fused step's bytes without the
    fp32 gates and outputs, plus the a/b projections (bf16), the per-head
    parameters, z (bf16), the norm weight and y (bf16)."""
    state = B * HV * DV * DK * 4 * 2
    conv = B * T * C_QKV * 2 + B * 3 * C_QKV * 2 + B * 4 * C_QKV * 2 + C_QKV * 4 * 2
    around = B * T * HV * 2 * 2 + HV * 4 * 2 + B * T * HV * DV * 2 + DV * 4 + B * T * HV * DV * 2
    return state + conv + around


class LayerBatched(Batched):
    """The batched decode through the layer step: gates from projections in
    front, gated RMS norm after, y in bf16 (one launch per layer)."""

    name = "layer"

    def _extra_inputs(self):
        torch = self.torch
        L, B, bf = self.L, self.B, torch.bfloat16
        self.fn = self.lib.gdn_layer_decode_step
        self.a = self.randn((self.n_sets, L, B, 1, HV), 1.0, bf)
        self.b = self.randn((self.n_sets, L, B, 1, HV), 1.0, bf)
        self.A_log = torch.log(1.0 + 15.0 * torch.rand((L, HV), generator=self.gen, device=self.device))
        dt = torch.exp(math.log(1e-3) + (math.log(1e-1) - math.log(1e-3)) *
                       torch.rand((L, HV), generator=self.gen, device=self.device))
        self.dt_bias = dt + torch.log(-torch.expm1(-dt))
        self.z = self.randn((self.n_sets, L, B, 1, HV, DV), 1.0, bf)
        self.norm_w = 1.0 + 0.1 * torch.randn((L, DV), generator=self.gen, device=self.device)
        self.y = torch.empty((L, B, 1, HV, DV), dtype=bf, device=self.device)

    def __init__(self, device, seed: int, steps: int, layers: int = 48):
        super().__init__(device, seed, steps, layers)
        self.dominant = "gdn_conv_decode_kernel[layer]"
        self.dominant_work = layer_bytes_per_launch(self.B)
        self.step_bytes = self.L * self.dominant_work

    def _args(self, s: int, l: int, sp):
        P = ctypes.c_void_p
        tl = P(self.tail[l].data_ptr())
        return (ctypes.byref(self.shape), 1, P(self.x[s, l].data_ptr()), P(self.w[l].data_ptr()), tl, tl,
                P(self.a[s, l].data_ptr()), P(self.b[s, l].data_ptr()), P(self.A_log[l].data_ptr()),
                P(self.dt_bias[l].data_ptr()), P(self.z[s, l].data_ptr()), P(self.norm_w[l].data_ptr()), 1e-6,
                P(self.state[l].data_ptr()), None, P(self.y[l].data_ptr()), 1.0, self.gdn.GDN_NORMALIZE_QK, sp)

    def e2e_pairs(self):
        torch = self.torch
        self.h_x = self.x[0].cpu().pin_memory()
        self.h_a = self.a[0].cpu().pin_memory()
        self.h_b = self.b[0].cpu().pin_memory()
        self.h_z = self.z[0].cpu().pin_memory()
        self.h_y = torch.empty(self.y.shape, dtype=torch.bfloat16, pin_memory=True)
        return [(self.x[0], self.h_x), (self.a[0], self.h_a), (self.b[0], self.h_b), (self.z[0], self.h_z)], \
               [(self.h_y, self.y)]

    def config(self=None) -> dict:
        L = Batched.L if self is None else self.L
        cfg = Batched.config(self)
        cfg["workload"] = (f"batched layer decode over {L} GDN layers: batch {Batched.B} sequences, 27B head "
                           "shape; per layer one launch of conv + SiLU, gates from the a/b projections "
                           "(A_log, dt_bias), L2-norm, the delta step and the gated RMS norm with z; y in bf16")
        return cfg


class KdaBatched(Batched):
    """The batched decode with the KDA step: a decay per key channel."""

    name = "kdabatch"
    kda = True

    def config(self=None) -> dict:
        L = Batched.L if self is None else self.L
        cfg = Batched.config(self)
        cfg["workload"] = (f"batched KDA decode over {L} layers: batch {Batched.B} sequences, 27B head shape "
                           "(16 key / 48 value heads x 128), a decay per key channel (alpha [B, Hv, 128] "
                           "fp32), fused conv + KDA step, one launch per layer")
        return cfg


class Decode1(Workload):
    """One layer, batch 1: conv + decode of one token per step."""

    name = "decode1"
    flush = True

    def __init__(self, device, seed: int, steps: int):
        super().__init__(device, seed)
        torch, gdn = self.torch, self.gdn
        bf = torch.bfloat16
        self.n = steps
        self.state = self.randn((1, HV, DV, DK), 0.1)
        self.w = self.randn((C_QKV, 4), 0.5, bf)
        self.tails = [self.randn((1, 4, C_QKV), 1.0, bf), torch.empty((1, 4, C_QKV), dtype=bf, device=device)]
        self.x = self.randn((self.n, 1, 1, C_QKV), 1.0, bf)
        self.alpha, self.beta = self.gates((self.n, 1, 1, HV))
        self.out = torch.empty((self.n, 1, 1, HV, DV), dtype=torch.float32, device=device)
        self.shape = gdn.gdn_shape(1, HK, HV, DK, DV)
        self.launches_per_step = 1
        self.units_per_step = HV
        self.dominant = "gdn_conv_decode_kernel"
        self.traffic_key = "gdn_conv_decode_kernel[b1]"
        self.dominant_sources = FUSED_SOURCES
        self.bound = "hbm"
        self.dominant_work = fused_bytes_per_launch(1)
        self.step_bytes = fused_bytes_per_launch(1)
        self.k = 0  # ping-pong position of the conv tail

    def _args(self, s, x=None, alpha=None, beta=None):
        P = ctypes.c_void_p
        tin, tout = self.tails[self.k % 2], self.tails[(self.k + 1) % 2]
        self.k += 1
        x = self.x[s] if x is None else x
        alpha = self.alpha[s] if alpha is None else alpha
        beta = self.beta[s] if beta is None else beta
        return (ctypes.byref(self.shape), 1, P(x.data_ptr()), P(self.w.data_ptr()), P(tin.data_ptr()),
                P(tout.data_ptr()), P(alpha.data_ptr()), P(beta.data_ptr()),
                P(self.state.data_ptr()), P(self.out[s].data_ptr()), 1.0, self.gdn.GDN_NORMALIZE_QK, self.sp)

    def step(self, i: int, rec: Recorder | None = None):
        args = self._args(i % self.n)
        if rec:
            rec.begin(i)
        _call(self.lib.gdn_conv_decode_step, args, self.gdn)
        if rec:
            rec.mark("gdn_conv_decode_kernel")

    def e2e_setup(self):
        self.e2e_views = self.e2e_pack([self.x[0].cpu(), self.alpha[0].cpu(), self.beta[0].cpu()])
        self.h_out = self.torch.empty(self.out[0].shape, dtype=self.torch.float32, pin_memory=True)
        self.e2e_h2d = self.e2e_hbuf.numel()
        self.e2e_d2h = self.h_out.numel() * 4

    def e2e_step(self, i: int):
        self.e2e_copy(self.e2e_dbuf, self.e2e_hbuf)  # x, alpha, beta in one copy
        vx, va, vb = self.e2e_views
        _call(self.lib.gdn_conv_decode_step, self._args(0, vx, va, vb), self.gdn)
        self.e2e_copy(self.h_out, self.out[0])

    B2B_STEPS = 100

    def extra_measures(self) -> dict:
        """The same steps back to back, as a decode loop runs one layer token
        after token: one CUDA graph of 100 consecutive steps (each launch a
        programmatic dependent of the previous one), replayed with events
        around the replay and L2 flushed before each replay.  No flush between
        the steps inside a replay, so the 3.15 MB state stays in L2 after the
        first: an optimistic bound beside the flushed per-step figure."""
        torch, n = self.torch, min(self.B2B_STEPS, self.n)
        g = torch.cuda.CUDAGraph()
        with torch.cuda.graph(g):
            st = ctypes.c_void_p(torch.cuda.current_stream().cuda_stream)
            for i in range(n):
                args = list(self._args(i))
                args[-1] = st
                _call(self.lib.gdn_conv_decode_step, tuple(args), self.gdn)
        for _ in range(3):
            g.replay()
        torch.cuda.synchronize()
        e0, e1 = torch.cuda.Event(enable_timing=True), torch.cuda.Event(enable_timing=True)
        times = []
        for _ in range(10):
            self.pre_step()  # L2 flushed before each replay (each timed iteration)
            e0.record()
            g.replay()
            e1.record()
            e1.synchronize()
            times.append(e0.elapsed_time(e1) * 1e3 / n)
        us = statistics.median(times)
        return {"back_to_back": {"us_per_step": us, "value": HV / (us * 1e-6), "unit": UNIT, "steps_per_graph": n,
                                 "replays": len(times),
                                 "how": "one CUDA graph of consecutive steps (programmatic dependent launches), L2 "
                                        "flushed before each replay, none between the steps inside it (the state "
                                        "stays L2-resident after the first), median over replays"}}

    @staticmethod
    def config() -> dict:
        return {"workload": "27B-shape single-token decode, one layer: batch 1, 16 key / 48 value heads "
                            "x 128, fp32 state 3.15 MB, bf16 inputs, 4-tap bf16 conv tail over 10,240 "
                            "channels (fused conv + delta step per token; conv tail ping-ponged "
                            "between two buffers)",
                "layers": 1, "batch": 1, "Hk": HK, "Hv": HV, "dk": DK, "dv": DV,
                "l2": "L2 flushed (256 MB write) before every step, outside the timed intervals",
                "launch": "eager, CUDA events around the step's kernels"}


class Tree(Workload):
    """One speculative round on one layer: the tree conv fused into the verify
    and the commit (two launches; the conv tail alternates between two
    buffers).  The three-launch round (conv, verify, commit) is timed beside it."""

    name = "tree"
    flush = True
    N = 32

    def __init__(self, device, seed: int, steps: int):
        super().__init__(device, seed)
        import numpy as np
        from hybrid_linear_attention_conv_gb300 import inputs as gen
        torch, gdn = self.torch, self.gdn
        bf = torch.bfloat16
        N = self.N
        self.parents = np.ascontiguousarray(gen.random_tree(seed, N, 8), np.int32)
        self.path = np.ascontiguousarray(gdn.tree_root_path(self.parents, gen.random_leaf(seed, self.parents)),
                                         np.int32)
        self.n_sets = min(8, steps)
        self.state = self.randn((HV, DV, DK), 0.1)
        self.w = self.randn((C_QKV, 4), 0.5, bf)
        self.tail = self.randn((1, 4, C_QKV), 1.0, bf)
        self.tails = [self.tail, self.tail.clone()]  # the fused commit writes the other buffer
        self.x = self.randn((self.n_sets, 1, N, C_QKV), 1.0, bf)
        self.alpha, self.beta = self.gates((self.n_sets, N, HV))
        self.y = torch.empty((1, N, C_QKV), dtype=bf, device=device)
        self.out = torch.empty((N, HV, DV), dtype=torch.float32, device=device)
        self.shape = gdn.gdn_shape(1, HK, HV, DK, DV)
        self.launches_per_step = 2  # conv + verify, conv + commit (replay + conv-tail update)
        self.tree_marks = 2
        self.units_per_step = (N + len(self.path)) * HV
        self.dominant = "gdn_tree_kernel"
        self.dominant_sources = FUSED_SOURCES  # the fused verify runs the conv arithmetic too
        self.bound = "alu"
        self.dominant_work = N * HV * step_flops_per_head_token()
        self.step_bytes = (2 * conv_bytes_per_launch(1, N) + HV * DV * DK * 4 +
                           N * (C_QKV * 2 + HV * 8 + HV * DV * 4) + 2 * HV * DV * DK * 4)

    @property
    def marks_per_step(self) -> int:
        return self.tree_marks

    def _run(self, s, rec=None, inputs=None, i=0, between=None):
        """The fused round: step i reads tail buffer i % 2 and writes the other.
        `between` runs after the verify is enqueued and before the commit."""
        P = ctypes.c_void_p
        lib, gdn = self.lib, self.gdn
        pp = self.parents.ctypes.data_as(P)
        x, alpha, beta = (self.x[s], self.alpha[s], self.beta[s]) if inputs is None else inputs
        t_in, t_out = self.tails[i % 2], self.tails[(i + 1) % 2]
        _call(lib.gdn_conv_tree_verify, (ctypes.byref(self.shape), self.N, pp, P(x.data_ptr()),
                                         P(self.w.data_ptr()), P(t_in.data_ptr()), P(alpha.data_ptr()),
                                         P(beta.data_ptr()), P(self.state.data_ptr()), P(self.out.data_ptr()), 1.0,
                                         gdn.GDN_NORMALIZE_QK, self.sp), gdn)
        if rec:
            rec.mark("gdn_tree_kernel")
        if between is not None:
            between()
        _call(lib.gdn_conv_commit_path, (ctypes.byref(self.shape), self.N, pp, self.path.ctypes.data_as(P),
                                         len(self.path), P(x.data_ptr()), P(self.w.data_ptr()),
                                         P(t_in.data_ptr()), P(t_out.data_ptr()), P(alpha.data_ptr()),
                                         P(beta.data_ptr()), P(self.state.data_ptr()), gdn.GDN_NORMALIZE_QK,
                                         self.sp), gdn)
        if rec:
            rec.mark("commit")  # conv + replay + tail update (one launch)

    def _run_unfused(self, s, rec=None):
        """The three-launch round: tree conv into y, verify, commit (tail in place)."""
        P = ctypes.c_void_p
        lib, gdn = self.lib, self.gdn
        pp = self.parents.ctypes.data_as(P)
        x, alpha, beta = self.x[s], self.alpha[s], self.beta[s]
        _call(lib.gdn_conv_step, (1, self.N, C_QKV, pp, P(x.data_ptr()), P(self.w.data_ptr()),
                                  P(self.tail.data_ptr()), P(self.y.data_ptr()), 0, self.sp), gdn)
        if rec:
            rec.mark("gdn_conv_kernel")
        _call(lib.gdn_tree_verify, (ctypes.byref(self.shape), self.N, pp, P(self.y.data_ptr()),
                                    P(alpha.data_ptr()), P(beta.data_ptr()),
                                    P(self.state.data_ptr()), P(self.out.data_ptr()), 1.0,
                                    gdn.GDN_NORMALIZE_QK, self.sp), gdn)
        if rec:
            rec.mark("gdn_tree_kernel")
        _call(lib.gdn_commit_path, (ctypes.byref(self.shape), self.N, pp, self.path.ctypes.data_as(P),
                                    len(self.path), P(self.y.data_ptr()), P(alpha.data_ptr()),
                                    P(beta.data_ptr()), P(x.data_ptr()),
                                    P(self.state.data_ptr()), P(self.tail.data_ptr()),
                                    gdn.GDN_NORMALIZE_QK, self.sp), gdn)
        if rec:
            rec.mark("commit")  # replay + tail update (one launch)

    def step(self, i: int, rec: Recorder | None = None):
        if rec:
            rec.begin(i)
        self._run(i % self.n_sets, rec, i=i)

    def extra_measures(self) -> dict:
        """The same rounds as three launches (gdn_conv_step into y, then the
        unfused verify and commit), L2 flushed before each, median of 50."""
        torch = self.torch
        # enqueued back to back like the timed steps (no host sync between
        # rounds), so the host's launch overhead hides behind the flushes
        n = 53
        ev = [[torch.cuda.Event(enable_timing=True) for _ in range(4)] for _ in range(n)]
        for i in range(n):
            self.pre_step()
            ev[i][0].record(self.stream)
            self._run_unfused(i % self.n_sets, _Marks(ev[i], self.stream))
        torch.cuda.synchronize()
        times = [e[0].elapsed_time(e[3]) * 1e3 for e in ev[3:]]
        parts = [[e[k].elapsed_time(e[k + 1]) * 1e3 for k in range(3)] for e in ev[3:]]
        us = statistics.median(times)
        med = [statistics.median(p[k] for p in parts) for k in range(3)]
        return {"unfused_round": {"us_per_step": us, "value": self.units_per_step / (us * 1e-6), "unit": UNIT,
                                  "conv_us": med[0], "verify_us": med[1], "commit_us": med[2], "launches": 3,
                                  "how": "gdn_conv_step (tree mode) + gdn_tree_verify + gdn_commit_path, L2 flushed "
                                         "before each round, rounds enqueued back to back, events between "
                                         "the launches, median of 50"}}

    def e2e_setup(self):
        self.e2e_views = self.e2e_pack([self.x[0].cpu(), self.alpha[0].cpu(), self.beta[0].cpu()])
        self.h_out = self.torch.empty(self.out.shape, dtype=self.torch.float32, pin_memory=True)
        self.e2e_h2d = self.e2e_hbuf.numel()
        self.e2e_d2h = self.h_out.numel() * 4
        self.e2e_streams()

    def e2e_step(self, i: int):
        """Inputs in (one packed copy), the verify, then the verify's outputs
        back to the host on their own stream while the commit runs; the step
        ends once both are done."""
        torch = self.torch
        cs = torch.cuda.current_stream()
        self.e2e_copy(self.e2e_dbuf, self.e2e_hbuf)  # x, alpha, beta in one copy

        def out_back():
            ev = torch.cuda.Event()
            ev.record(cs)
            with torch.cuda.stream(self.s_out):
                self.s_out.wait_event(ev)
                self.h_out.copy_(self.out, non_blocking=True)

        self._run(0, inputs=self.e2e_views, i=i, between=out_back)
        done = torch.cuda.Event()
        done.record(self.s_out)
        cs.wait_event(done)

    def config(self=None) -> dict:
        L = None if self is None else len(self.path)
        return {"workload": "tree verify + commit, 27B head shape, one layer: random 32-node draft tree "
                            "(depth <= 8, branching 1-4), state branched per node from its parent, random "
                            "root-to-leaf path committed (tree conv + verify + commit per step)",
                "nodes": Tree.N, "path_len": L, "Hk": HK, "Hv": HV, "dk": DK, "dv": DV,
                "units": "head.tokens = (verified nodes + committed tokens) x 48 value heads",
                "l2": "L2 flushed (256 MB write) before every step, outside the timed intervals",
                "launch": "eager, CUDA events around the step's kernels"}


class TreeBatch(Workload):
    """Joint verify of 8 sequences' draft trees (32 nodes each, own shapes) in one launch."""

    name = "treebatch"
    flush = True
    B, N = 8, 32

    def __init__(self, device, seed: int, steps: int):
        super().__init__(device, seed)
        import numpy as np
        from hybrid_linear_attention_conv_gb300 import inputs as gen
        torch, gdn = self.torch, self.gdn
        B, N = self.B, self.N
        self.parents = np.ascontiguousarray(np.stack([gen.random_tree(seed + b, N, 8) for b in range(B)]), np.int32)
        self.counts = np.full(B, N, np.int32)
        self.n_sets = min(8, steps)
        self.state = self.randn((B, HV, DV, DK), 0.1)
        self.qkv = self.randn((self.n_sets, B, N, C_QKV), 1.0, torch.bfloat16)
        self.alpha, self.beta = self.gates((self.n_sets, B, N, HV))
        self.out = torch.empty((B, N, HV, DV), dtype=torch.float32, device=device)
        self.shape = gdn.gdn_shape(B, HK, HV, DK, DV)
        self.launches_per_step = 1
        self.units_per_step = B * N * HV
        self.dominant = "gdn_tree_kernel"
        self.traffic_key = "gdn_tree_kernel[batch8]"  # the 8-tree launch, not the 1-tree one
        self.dominant_sources = DECODE_SOURCES
        self.bound = "alu"
        self.dominant_work = B * N * HV * step_flops_per_head_token()
        self.step_bytes = B * (HV * DV * DK * 4 + N * (C_QKV * 2 + HV * 8 + HV * DV * 4))

    def _args(self, s, inputs=None):
        P = ctypes.c_void_p
        qkv, alpha, beta = (self.qkv[s], self.alpha[s], self.beta[s]) if inputs is None else inputs
        return (ctypes.byref(self.shape), self.N, self.counts.ctypes.data_as(P), self.parents.ctypes.data_as(P),
                P(qkv.data_ptr()), P(alpha.data_ptr()), P(beta.data_ptr()),
                P(self.state.data_ptr()), P(self.out.data_ptr()), 1.0, self.gdn.GDN_NORMALIZE_QK, self.sp)

    def step(self, i: int, rec: Recorder | None = None):
        args = self._args(i % self.n_sets)
        if rec:
            rec.begin(i)
        _call(self.lib.gdn_tree_verify_batched, args, self.gdn)
        if rec:
            rec.mark("gdn_tree_kernel")

    def extra_measures(self) -> dict:
        """The same joint verify from pre-conv inputs: gdn_conv_tree_verify_batched
        (each tree's conv inside the verify, the q/k conv of a key head shared by
        its CTAs as one cluster).  L2 flushed before each, calls enqueued back to
        back, median of 50."""
        torch, P = self.torch, ctypes.c_void_p
        B, N = self.B, self.N
        x = self.randn((B, N, C_QKV), 1.0, torch.bfloat16)
        w = self.randn((C_QKV, 4), 0.5, torch.bfloat16)
        tails = self.randn((B, 4, C_QKV), 1.0, torch.bfloat16)
        n = 53
        ev = [[torch.cuda.Event(enable_timing=True) for _ in range(2)] for _ in range(n)]
        for i in range(n):
            self.pre_step()
            ev[i][0].record(self.stream)
            _call(self.lib.gdn_conv_tree_verify_batched,
                  (ctypes.byref(self.shape), N, self.counts.ctypes.data_as(P), self.parents.ctypes.data_as(P),
                   P(x.data_ptr()), P(w.data_ptr()), P(tails.data_ptr()), P(self.alpha[0].data_ptr()),
                   P(self.beta[0].data_ptr()), P(self.state.data_ptr()), P(self.out.data_ptr()), 1.0,
                   self.gdn.GDN_NORMALIZE_QK, self.sp), self.gdn)
            ev[i][1].record(self.stream)
        torch.cuda.synchronize()
        us = statistics.median(e[0].elapsed_time(e[1]) * 1e3 for e in ev[3:])
        return {"conv_fused": {"us_per_step": us, "value": self.units_per_step / (us * 1e-6), "unit": UNIT,
                               "how": "gdn_conv_tree_verify_batched on pre-conv inputs (8 trees x 32 nodes), L2 "
                                      "flushed before each call, median of 50"}}

    def e2e_setup(self):
        self.e2e_views = self.e2e_pack([self.qkv[0].cpu(), self.alpha[0].cpu(), self.beta[0].cpu()])
        self.h_out = self.torch.empty(self.out.shape, dtype=self.torch.float32, pin_memory=True)
        self.e2e_h2d = self.e2e_hbuf.numel()
        self.e2e_d2h = self.h_out.numel() * 4

    def e2e_step(self, i: int):
        self.e2e_copy(self.e2e_dbuf, self.e2e_hbuf)  # q/k/v, alpha, beta in one copy
        _call(self.lib.gdn_tree_verify_batched, self._args(0, self.e2e_views), self.gdn)
        self.e2e_copy(self.h_out, self.out)

    @staticmethod
    def config() -> dict:
        return {"workload": "joint tree verify of 8 sequences, 27B head shape, one layer: a random 32-node "
                            "draft tree per sequence (depth <= 8, branching 1-4, own shape), each sequence's "
                            "own state, all trees in one launch",
                "sequences": TreeBatch.B, "nodes": TreeBatch.N, "Hk": HK, "Hv": HV, "dk": DK, "dv": DV,
                "l2": "L2 flushed (256 MB write) before every step, outside the timed intervals",
                "launch": "eager, CUDA events around the launch"}


SNAPSHOT_SOURCES = ["hybrid_linear_attention_conv_gb300/csrc/gdn_snapshot.cu",
                    "hybrid_linear_attention_conv_gb300/csrc/gdn_internal.h"]


def snapshot_payload_bytes(layers: int = 48) -> int:
    """One sequence's sections over all layers: fp32 state + bf16 conv tail."""
    return layers * (HV * DV * DK * 4 + 4 * C_QKV * 2)


class Snapshot(Workload):
    """Snapshot one sequence's recurrent sections (48 layers) and restore them."""

    name = "snapshot"
    flush = True
    L, B = 48, 64
    metric = "state snapshot save + restore throughput (one sequence, every layer, bit-exact)"
    unit = "GB/s"
    dtype = "u8"  # raw bytes: fp32 and bf16 bit patterns copied as they are

    def __init__(self, device, seed: int, steps: int, layers: int = 48, seqs: int = 64):
        super().__init__(device, seed)
        torch, gdn = self.torch, self.gdn
        self.L, self.B = layers, seqs
        L, B = self.L, self.B
        self.state = self.randn((L, B, HV, DV, DK), 0.1)
        self.tail = self.randn((L, B, 4, C_QKV), 1.0, torch.bfloat16)
        self.shape = gdn.gdn_shape(B, HK, HV, DK, DV)
        self.nbytes = gdn.snapshot_bytes(L, HK, HV, DK, DV)
        self.payload = snapshot_payload_bytes(L)
        self.blob = torch.empty(self.nbytes, dtype=torch.uint8, device=device)
        self.ws = torch.zeros(256, dtype=torch.uint8, device=device)
        self.launches_per_step = 3       # gather; verify, scatter
        # algorithmic bytes: save reads and writes the payload, restore reads and writes it
        self.units_per_step = 4 * self.payload / 1e9
        self.dominant = "save"                          # the save call: workspace reset + gather kernel
        self.traffic_key = "gdn_snapshot_gather_kernel"
        self.dominant_sources = SNAPSHOT_SOURCES
        self.bound = "hbm"
        self.dominant_work = 2 * self.payload + 64
        self.step_bytes = 4 * self.payload

    @property
    def marks_per_step(self) -> int:
        return 2

    def _save(self, seq, blob):
        P = ctypes.c_void_p
        _call(self.lib.gdn_snapshot_save,
              (ctypes.byref(self.shape), self.L, seq, P(self.state.data_ptr()), self.state.stride(0),
               P(self.tail.data_ptr()), self.tail.stride(0), P(blob.data_ptr()), blob.numel(),
               P(self.ws.data_ptr()), 256, self.sp), self.gdn)

    def _restore(self, seq, blob):
        P = ctypes.c_void_p
        _call(self.lib.gdn_snapshot_restore,
              (ctypes.byref(self.shape), self.L, seq, P(blob.data_ptr()), blob.numel(), P(self.state.data_ptr()),
               self.state.stride(0), P(self.tail.data_ptr()), self.tail.stride(0), P(self.ws.data_ptr()), 256,
               self.sp), self.gdn)

    def step(self, i: int, rec: Recorder | None = None):
        seq = i % self.B
        if rec:
            rec.begin(i)
        self._save(seq, self.blob)
        if rec:
            rec.mark("save")
        self._restore(seq, self.blob)
        if rec:
            rec.mark("restore")

    def check_status(self):
        status = int(self.ws[:4].view(self.torch.int32).item())
        if status != 0:
            raise RuntimeError(f"snapshot restore refused the blob (status {status})")

    def e2e_setup(self):
        # the blob lives in pinned host memory: the kernels write and read it there
        self.h_blob = self.torch.empty(self.nbytes, dtype=self.torch.uint8, pin_memory=True)
        self.e2e_h2d = self.nbytes
        self.e2e_d2h = self.nbytes

    def e2e_step(self, i: int):
        seq = i % self.B
        self._save(seq, self.h_blob)
        self._restore(seq, self.h_blob)

    def config(self=None) -> dict:
        L = Snapshot.L if self is None else self.L
        B = Snapshot.B if self is None else self.B
        return {"workload": f"snapshot of one sequence's recurrent sections over {L} layers (fp32 state "
                            f"48 x 128 x 128 + bf16 conv tail 4 x 10,240 per layer) out of {B} sequences held "
                            "in HBM, into a device blob, then a verified restore of it",
                "layers": L, "sequences": B, "blob_bytes": snapshot_payload_bytes(L) + 64,
                "units": "algorithmic GB: payload read + written by save, read + written by restore",
                "l2": "L2 flushed (256 MB write) before every step, outside the timed intervals",
                "launch": "eager; CUDA events after the save call (workspace reset, gather) and after the "
                          "restore call (reset, verify, scatter); the roofline times the save call",
                "e2e": "the blob in pinned host memory instead, written and read by the kernels over the "
                       "host link"}


class Prefill(Workload):
    """Chunked prefill of 8,192 tokens, one layer."""

    name = "prefill"
    T = 8192

    def __init__(self, device, seed: int, steps: int):
        super().__init__(device, seed)
        torch, gdn = self.torch, self.gdn
        T = self.T
        self.state = self.randn((HV, DV, DK), 0.1)
        self.qkv = self.randn((T, C_QKV), 1.0, torch.bfloat16)
        self.alpha, self.beta = self.gates((T, HV))
        self.out = torch.empty((T, HV, DV), dtype=torch.float32, device=device)
        nbytes = gdn.prefill_workspace_bytes(T, HK, HV, DK, DV)
        self.ws = torch.zeros(max(nbytes, 256), dtype=torch.uint8, device=device)
        self.shape = gdn.gdn_shape(1, HK, HV, DK, DV)
        self.launches_per_step = 1       # one cooperative launch: pre-pass workers and chains
        self.units_per_step = T * HV
        self.dominant = "gdn_chunk_prefill"  # the whole call
        self.traffic_key = "gdn_prefill_fused_kernel"
        self.dominant_sources = PREFILL_SOURCES
        self.bound = "tensor"
        self.dominant_work = prefill_flops(T)
        self.step_bytes = prefill_bytes(T)

    @property
    def marks_per_step(self) -> int:
        return 1  # one event after the call

    def _args(self):
        P = ctypes.c_void_p
        return (ctypes.byref(self.shape), self.T, CHUNK, P(self.qkv.data_ptr()), P(self.alpha.data_ptr()),
                P(self.beta.data_ptr()), P(self.state.data_ptr()), P(self.out.data_ptr()),
                P(self.ws.data_ptr()), self.ws.numel(), 1.0, self.gdn.GDN_NORMALIZE_QK, self.sp)

    def step(self, i: int, rec: Recorder | None = None):
        if rec:
            rec.begin(i)
        _call(self.lib.gdn_chunk_prefill, self._args(), self.gdn)
        if rec:
            rec.mark("gdn_chunk_prefill")

    def check_status(self):
        st = int(self.ws[:4].view(self.torch.int32).item())
        if st != 0:
            raise RuntimeError("prefill reported a tensor-core wait timeout")

    def extra_measures(self) -> dict:
        """The prompt's conv ahead of the prefill (gdn_conv_step, linear mode,
        8,192 tokens x 10,240 channels): what producing the prefill's qkv input
        from the pre-conv projections costs.  Its 168 MB in and 168 MB out are
        larger than L2; calls enqueued back to back, median of 10."""
        torch, P = self.torch, ctypes.c_void_p
        T, n = self.T, 13
        x = self.randn((1, T, C_QKV), 1.0, torch.bfloat16)
        w = self.randn((C_QKV, 4), 0.5, torch.bfloat16)
        tail = self.randn((1, 4, C_QKV), 1.0, torch.bfloat16)
        y = torch.empty_like(x)
        ev = [[torch.cuda.Event(enable_timing=True) for _ in range(2)] for _ in range(n)]
        for i in range(n):
            ev[i][0].record(self.stream)
            _call(self.lib.gdn_conv_step, (1, T, C_QKV, None, P(x.data_ptr()), P(w.data_ptr()), P(tail.data_ptr()),
                                           P(y.data_ptr()), 0, self.sp), self.gdn)
            ev[i][1].record(self.stream)
        torch.cuda.synchronize()
        us = statistics.median(e[0].elapsed_time(e[1]) * 1e3 for e in ev[3:])
        nbytes = 2 * T * C_QKV * 2  # x read + y written (bf16); taps and tail are negligible
        return {"conv": {"us": us, "gbs": nbytes / (us * 1e-6) / 1e9, "bytes": nbytes, "tokens": T,
                         "channels": C_QKV,
                         "how": "gdn_conv_step over the prompt (linear mode), bf16 in and out, median of 10, "
                                "calls enqueued back to back"}}

    E2E_PIECE = 2048  # tokens per piece of the overlapped end-to-end step (a multiple of the chunk)

    def e2e_setup(self):
        self.h_qkv = self.qkv.cpu().pin_memory()
        self.h_a = self.alpha.cpu().pin_memory()
        self.h_b = self.beta.cpu().pin_memory()
        self.h_out = self.torch.empty(self.out.shape, dtype=self.torch.float32, pin_memory=True)
        self.e2e_h2d = self.h_qkv.numel() * 2 + self.h_a.numel() * 4 + self.h_b.numel() * 4
        self.e2e_d2h = self.h_out.numel() * 4
        self.e2e_streams()

    def e2e_step(self, i: int):
        """The 8,192 tokens as four consecutive calls of 2,048 (the state
        carries over; the chunk boundaries are the same, so the results are
        the same), each piece's copies overlapping its neighbours' compute."""
        P, n = ctypes.c_void_p, self.E2E_PIECE
        pieces = (self.T + n - 1) // n
        sl = lambda k: slice(k * n, min((k + 1) * n, self.T))

        def compute(k):
            t = sl(k)
            args = (ctypes.byref(self.shape), t.stop - t.start, CHUNK, P(self.qkv[t].data_ptr()),
                    P(self.alpha[t].data_ptr()), P(self.beta[t].data_ptr()), P(self.state.data_ptr()),
                    P(self.out[t].data_ptr()), P(self.ws.data_ptr()), self.ws.numel(), 1.0,
                    self.gdn.GDN_NORMALIZE_QK, ctypes.c_void_p(self.torch.cuda.current_stream().cuda_stream))
            _call(self.lib.gdn_chunk_prefill, args, self.gdn)

        self.e2e_pipeline(pieces,
                          lambda k: [(self.qkv[sl(k)], self.h_qkv[sl(k)]), (self.alpha[sl(k)], self.h_a[sl(k)]),
                                     (self.beta[sl(k)], self.h_b[sl(k)])],
                          lambda k: [(self.h_out[sl(k)], self.out[sl(k)])],
                          compute)

    @staticmethod
    def config() -> dict:
        return {"workload": "chunked prefill: 1 sequence, 8,192 tokens, 27B head shape, chunk 64, bf16 "
                            "q/k/v, fp32 alpha/beta/state, WY/UT chunk form on tcgen05 tensor cores",
                "tokens": Prefill.T, "chunk": CHUNK, "Hk": HK, "Hv": HV, "dk": DK, "dv": DV,
                "l2": "inputs larger than L2: 168 MB of q/k/v read and 201 MB of outputs per step",
                "launch": "eager, CUDA events around the call (status and flag resets, one cooperative launch: pre-pass workers and chains)"}


WORKLOADS = {"batched": Batched, "kdabatch": KdaBatched, "layer": LayerBatched, "decode1": Decode1, "tree": Tree, "treebatch": TreeBatch,
             "prefill": Prefill, "snapshot": Snapshot}
DEFAULT_STEPS = {"batched": 100, "kdabatch": 100, "layer": 100, "decode1": 1000, "tree": 200, "treebatch": 200, "prefill": 20,
                 "snapshot": 50}


# ---------------------------------------------------------------------------
# the oracle on the host cores (CPU baseline and the reference arm)
# ---------------------------------------------------------------------------
class OracleSample:
    """A bounded sample of a workload run by the fp64 C oracle as it stands."""

    def __init__(self, workload: str):
        import numpy as np
        import oracle
        from hybrid_linear_attention_conv_gb300 import inputs as gen
        oracle.build()
        self.np, self.oracle, self.gen = np, oracle, gen
        self.workload = workload
        s = self.s = gen.QWEN_27B
        if workload in ("batched", "decode1", "kdabatch"):
            self.c = gen.conv_inputs(0, 1, 1, s.C)
            self.d = gen.kda_inputs(0, s, 1) if workload == "kdabatch" else gen.decode_inputs(0, s, 1)
            self.state = self.d["state"].astype(np.float64)
            self.units = s.Hv
            step = "KDA decode" if workload == "kdabatch" else "decode"
            self.desc = f"conv + {step} of 1 sequence x 1 layer x 1 token (48 head.tokens)"
        elif workload in ("tree", "treebatch"):
            self.parents = gen.random_tree(0, 32, 8)
            self.c = gen.conv_inputs(0, 1, 32, s.C)
            self.d = gen.decode_inputs(0, s, 32, tag="tree")
            self.path = oracle.root_path(self.parents, gen.random_leaf(0, self.parents))
            if workload == "tree":
                self.units = (32 + len(self.path)) * s.Hv
                self.desc = (f"tree conv + verify (32 nodes, root-path replay) + commit ({len(self.path)} "
                             f"tokens) of one layer")
            else:
                self.units = 32 * s.Hv
                self.desc = "tree conv + verify of one sequence's 32-node tree (root-path replay), one layer"
        elif workload == "layer":
            self.d = gen.layer_inputs(0, s, 1)
            self.state = self.d["state"].astype(np.float64)
            self.units = s.Hv
            self.desc = "the layer decode step (conv, gates, delta step, gated norm) of 1 sequence x 1 layer x 1 token"
        elif workload == "snapshot":
            self.Ls = 4
            n_st = self.Ls * s.Hv * s.dv * s.dk
            self.snap_state = gen.normal(0, "snapshot.state", n_st).astype(np.float32).reshape(
                self.Ls, 1, s.Hv, s.dv, s.dk)
            self.snap_tail = gen.normal_bf16(0, "snapshot.tail", self.Ls * 4 * s.C).reshape(self.Ls, 1, 4, s.C)
            self.units = 4 * snapshot_payload_bytes(self.Ls) / 1e9
            self.desc = f"snapshot save + verified restore of one sequence over {self.Ls} of the 48 layers"
        else:
            self.Ts = 128
            self.d = gen.decode_inputs(0, s, self.Ts, tag="prefill")
            self.units = self.Ts * s.Hv
            self.desc = f"sequential prefill of {self.Ts} of the 8,192 tokens, all 48 value heads"

    def run_once(self) -> float:
        o, s, d = self.oracle, self.s, getattr(self, "d", None)
        if self.workload in ("batched", "decode1", "kdabatch"):
            y, _ = o.conv_linear(self.c["x"], self.c["w"], self.c["tail"])
            step = o.kda_decode if self.workload == "kdabatch" else o.decode
            _, self.state = step(o.f64_to_bf16(y), d["alpha"], d["beta"], self.state, s.Hk, s.Hv, s.dk, s.dv)
        elif self.workload == "tree":
            y = o.f64_to_bf16(o.conv_tree(self.parents, self.c["x"][0], self.c["w"], self.c["tail"][0]))
            o.tree_verify(self.parents, y, d["alpha"][0], d["beta"][0], d["state"][0], s.Hk, s.Hv, s.dk, s.dv)
            if self.workload == "treebatch":
                return self.units
            o.commit(self.parents, self.path, y, d["alpha"][0], d["beta"][0], d["state"][0], s.Hk, s.Hv,
                     s.dk, s.dv, x_tree=self.c["x"][0], tail=self.c["tail"][0])
        elif self.workload == "layer":
            _, _, self.state, _ = o.layer_decode(d["x"], d["w"], d["tail"], d["a"], d["b"], d["A_log"], d["dt_bias"],
                                                 d["z"], d["norm_w"], self.state, s.Hk, s.Hv, s.dk, s.dv)
        elif self.workload == "snapshot":
            blob = o.snapshot_save(self.snap_state, self.snap_tail, 0, s.Hk, s.Hv, s.dk, s.dv)
            rc, _, _ = o.snapshot_restore(blob, self.snap_state, self.snap_tail, 0, s.Hk, s.Hv, s.dk, s.dv)
            assert rc == 0
        else:
            o.prefill(d["qkv"], d["alpha"], d["beta"], d["state"], s.Hk, s.Hv, s.dk, s.dv)
        return self.units


def host_info() -> dict:
    """The host's core count and CPU model (the CPU baseline's machine)."""
    model = ""
    try:  # lscpu names Arm cores (e.g. Neoverse-V2) where /proc/cpuinfo has only part numbers
        out = subprocess.run(["lscpu"], capture_output=True, text=True, timeout=10).stdout
        for line in out.splitlines():
            if line.startswith("Model name"):
                model = line.split(":", 1)[1].strip()
                break
    except (OSError, subprocess.SubprocessError):
        pass
    if not model:
        try:
            with open("/proc/cpuinfo") as f:
                txt = f.read()
            for key in ("model name", "Model Name", "CPU part"):
                for line in txt.splitlines():
                    if line.startswith(key):
                        model = line.split(":", 1)[1].strip()
                        break
                if model:
                    break
        except OSError:
            pass
    import platform
    return {"nproc": os.cpu_count() or 1, "cpu_model": model or "unknown", "machine": platform.machine()}


def cpu_oracle_sample(workload: str, seconds: float, threads: int = 1) -> dict:
    """The oracle as it stands on a bounded sample of the workload for about
    `seconds`: one thread, or `threads` threads each running its own copy of
    the sample (independent sequences: the C oracle runs with the GIL
    released, so the threads take separate cores)."""
    from concurrent.futures import ThreadPoolExecutor
    samples = [OracleSample(workload) for _ in range(threads)]
    t0 = time.perf_counter()

    def loop(smp):
        n, units = 0, 0.0
        while True:
            units += smp.run_once()
            n += 1
            if time.perf_counter() - t0 >= seconds:
                return n, units

    if threads == 1:
        results = [loop(samples[0])]
    else:
        with ThreadPoolExecutor(max_workers=threads) as ex:
            results = list(ex.map(loop, samples))
    el = time.perf_counter() - t0
    n = sum(r[0] for r in results)
    units = sum(r[1] for r in results)
    how = "single thread" if threads == 1 else f"{threads} threads (one independent sample each)"
    return {"value": units / el, "unit": getattr(WORKLOADS[workload], "unit", UNIT), "cores": threads,
            "kind": "oracle",
            "sample": f"{n} x ({samples[0].desc}), 27B head shape, fp64 C oracle, {how}, {el:.1f} s"}


def cpu_baselines(workload: str, seconds: float) -> dict:
    """The single-thread oracle (the cpu_baseline) with, beside it, the same
    sample on every host core and the host's description."""
    one = cpu_oracle_sample(workload, seconds, 1)
    info = host_info()
    if info["nproc"] > 1:
        one["all_cores"] = cpu_oracle_sample(workload, seconds, info["nproc"])
    one["host"] = info
    return one


# ---------------------------------------------------------------------------
# arms
# ---------------------------------------------------------------------------
def measure(args, name: str, steps: int, warmup: int, device, peaks: dict, peaks_kind: str, cpu: bool) -> dict:
    """One workload's timed steps, roofline, end-to-end run and CPU baseline:
    the fields of a bench line (rank 0 gets the aggregate over ranks)."""
    import torch
    rank, world, local = dist_env()
    cls = WORKLOADS[name]
    if issubclass(cls, Batched):
        wl = cls(device, 1234 + rank, steps + warmup, layers=args.layers)
    elif cls is Snapshot:
        wl = cls(device, 1234 + rank, steps + warmup, layers=args.layers, seqs=args.seqs)
    else:
        wl = cls(device, 1234 + rank, steps + warmup)
    torch.cuda.synchronize()

    for i in range(warmup):
        wl.pre_step()
        wl.step(i)
    torch.cuda.synchronize()
    if hasattr(wl, "capture") and not args.eager:
        wl.capture()
        wl.step(0)  # one replay before the timed region
        torch.cuda.synchronize()

    rec = Recorder(torch, wl.stream, wl.marks_per_step, steps)
    clocks = ClockSampler(local)
    clocks.start()
    time.sleep(0.2)
    barrier(world)
    torch.cuda.synchronize()
    for i in range(steps):
        wl.pre_step()
        wl.step(warmup + i, rec)
    torch.cuda.synchronize()
    barrier(world)
    clk = clocks.stop()
    if hasattr(wl, "check_status"):
        wl.check_status()
    step_ms = rec.step_ms()
    total_s = sum(step_ms) / 1e3
    dom_ms = wl.dominant_ms(rec) if hasattr(wl, "dominant_ms") else rec.kernel_ms(wl.dominant)
    agg = aggregate(wl.units_per_step * steps, total_s, world, device)

    # end-to-end through the API with host buffers
    wl.e2e_setup()
    for i in range(2):
        wl.pre_step()
        wl.e2e_step(i)
    torch.cuda.synchronize()
    barrier(world)
    # each step: host->device copies of the step's inputs (pinned), the C-ABI
    # calls, the device->host copy of the outputs; timed by events on the stream
    e2e_total = 0.0
    e0 = torch.cuda.Event(enable_timing=True)
    e1 = torch.cuda.Event(enable_timing=True)
    for i in range(steps):
        wl.pre_step()
        e0.record()
        wl.e2e_step(i)
        e1.record()
        e1.synchronize()
        e2e_total += e0.elapsed_time(e1) / 1e3
    e2e = aggregate(wl.units_per_step * steps, e2e_total, world, device)
    if hasattr(wl, "check_status"):
        wl.check_status()

    dom_avg_s = statistics.mean(dom_ms) / 1e3
    if wl.bound == "hbm":
        achieved = wl.dominant_work / dom_avg_s / 1e9
        peak, unit = float(peaks["hbm_gbs"]), "GB/s"
        peak_kind = peaks_kind
    elif wl.bound == "tensor":
        achieved = wl.dominant_work / dom_avg_s / 1e12
        peak, unit = float(peaks["bf16_tflops"]), "TFLOP/s"
        peak_kind = f"{peaks_kind} bf16 dense (burst), algorithmic flops only"
    else:
        achieved = wl.dominant_work / dom_avg_s / 1e12
        mhz = float(peaks.get("sm_max_mhz", 2070.0))
        peak, unit = fp32_alu_peak_tflops(mhz), "TFLOP/s"
        peak_kind = f"derived fp32 FMA peak: {SMS} SMs x {FP32_LANES_PER_SM} lanes x 2 x {mhz:.0f} MHz"
    traffic = ncu_traffic(getattr(wl, "traffic_key", wl.dominant), wl.dominant_sources)
    step_gbs = wl.step_bytes * steps / total_s / 1e9
    roof = {"bound": wl.bound, "kernel": wl.dominant, "achieved": achieved, "peak": peak, "unit": unit,
            "frac": achieved / peak, "peak_kind": peak_kind, "avg_launch_us": dom_avg_s * 1e6,
            "work_per_launch": wl.dominant_work,
            "work_unit": "bytes" if wl.bound == "hbm" else "flops", "traffic": traffic}
    if wl.bound == "hbm":
        roof["frac_nominal_8tbs"] = achieved / NOMINAL_HBM_GBS
    metric, unit_v = getattr(wl, "metric", METRIC), getattr(wl, "unit", UNIT)
    line = {
        "metric": metric,
        "value": agg["value"],
        "unit": unit_v,
        "n_gpus": world,
        "steps": steps,
        "warmup": warmup,
        "ms_per_step": statistics.mean(step_ms),
        "higher_is_better": True,
        "scaling": "weak",
        "vs_baseline": None,
        "dtype": getattr(wl, "dtype", "f32"),
        "data": "synthetic (seeded device RNG; 27B head shape, random-init states)",
        "config": wl.config(),
        "hbm_gbs_step": step_gbs,
        "hbm_frac_step": step_gbs / float(peaks["hbm_gbs"]),
        "roofline": roof,
        "clocks": clk,
        "e2e": {"value": e2e["value"], "unit": unit_v, "h2d_bytes_per_step": wl.e2e_h2d,
                "d2h_bytes_per_step": wl.e2e_d2h, "ms_per_step": e2e_total * 1e3 / steps},
        "gpu_launches": wl.launches_per_step * steps,
    }
    if hasattr(wl, "extra_measures") and not args.no_extras:
        line.update(wl.extra_measures())
    del wl, rec
    torch.cuda.synchronize()
    torch.cuda.empty_cache()
    if cpu and rank == 0 and world == 1 and not args.no_cpu_baseline:
        line["cpu_baseline"] = cpu_baselines(name, args.cpu_seconds)
    return line


# the other single-GPU configs measured beside the headline in a default run
EXTRA_WORKLOADS = ("decode1", "tree", "prefill")


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
    name = args.workload or "batched"
    steps = args.steps if args.steps is not None else DEFAULT_STEPS[name]
    line = measure(args, name, steps, args.warmup, device, peaks, peaks_kind, cpu=True)
    if args.workload is None and world == 1 and not args.no_extras:
        # the other configs, each at its own step count (decode1 1,000 steps
        # as its config states; all of them finish in well under a second of
        # GPU time)
        line["workloads"] = {w: measure(args, w, DEFAULT_STEPS[w], args.warmup, device, peaks, peaks_kind,
                                        cpu=True)
                             for w in EXTRA_WORKLOADS}
    if rank != 0:
        return None
    return line


def run_reference(args) -> dict | None:
    rank, world, _ = dist_env()
    if rank != 0:
        return None
    name = args.workload or "batched"
    steps = args.steps if args.steps is not None else DEFAULT_STEPS[name]
    smp = OracleSample(name)
    for _ in range(args.warmup):
        smp.run_once()
    units = 0
    t0 = time.perf_counter()
    for _ in range(steps):
        units += smp.run_once()
    el = time.perf_counter() - t0
    value = units / el
    sample = f"each step: {smp.desc}, 27B head shape, fp64 C oracle, single thread"
    cls = WORKLOADS[name]
    cfg = cls.config()
    metric, unit = getattr(cls, "metric", METRIC), getattr(cls, "unit", UNIT)
    return {
        "impl": "reference",
        "metric": metric, "value": value, "unit": unit, "n_gpus": world, "steps": steps,
        "warmup": args.warmup, "ms_per_step": el * 1e3 / steps, "higher_is_better": True,
        "scaling": "weak", "vs_baseline": None, "dtype": getattr(cls, "dtype", "f64"), "data": "synthetic",
        "config": cfg,
        "cpu_baseline": {"value": value, "unit": unit, "cores": 1, "kind": "oracle", "sample": sample,
                         "host": host_info()},
        "e2e": {"value": value, "unit": unit, "h2d_bytes_per_step": 0, "d2h_bytes_per_step": 0},
    }


def main(argv=None):
    ap = argparse.ArgumentParser(description=__doc__, formatter_class=argparse.RawDescriptionHelpFormatter)
    ap.add_argument("--gpus", type=int, default=1)
    ap.add_argument("--steps", type=int, default=None)
    ap.add_argument("--warmup", type=int, default=5)
    ap.add_argument("--impl", choices=["ours", "reference"], default="ours")
    ap.add_argument("--workload", choices=sorted(WORKLOADS), default=None,
                    help="one workload alone (default: the batched decode, with decode1, tree and prefill "
                         "measured beside it under \"workloads\")")
    ap.add_argument("--no-extras", action="store_true",
                    help="measure the named workload (default: the batched decode) only, without the other "
                         "configs or the extra measurements beside it (for profiling runs)")
    ap.add_argument("--layers", type=int, default=48,
                    help="GDN layers in the batched workload (48 = the 27B model; fewer only for "
                         "profiling small cases)")
    ap.add_argument("--seqs", type=int, default=64,
                    help="sequences held in HBM by the snapshot workload (fewer only for profiling small cases)")
    ap.add_argument("--eager", action="store_true",
                    help="launch the batched step eagerly with an event after every kernel instead of "
                         "replaying it as a CUDA graph")
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
