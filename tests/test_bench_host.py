"""Host-side logic of bench.py that needs no GPU: the multi-rank aggregation
(world size 2 over gloo on CPU), the clock parser, the algorithmic work per
launch the roofline divides by, and the reference (oracle) arm's JSON line."""
import json
import os
import socket
import subprocess
import sys

import pytest
import torch.multiprocessing as mp

ROOT = os.path.dirname(os.path.dirname(os.path.abspath(__file__)))
sys.path.insert(0, ROOT)
import bench  # noqa: E402


def _free_port() -> int:
    with socket.socket() as s:
        s.bind(("127.0.0.1", 0))
        return s.getsockname()[1]


def _rank_main(rank, world, port, q):
    import torch.distributed as dist
    os.environ.update(MASTER_ADDR="127.0.0.1", MASTER_PORT=str(port), RANK=str(rank),
                      WORLD_SIZE=str(world), LOCAL_RANK=str(rank))
    dist.init_process_group("gloo", rank=rank, world_size=world)
    # rank r did 100*(r+1) units in (r+1) seconds
    agg = bench.aggregate(100.0 * (rank + 1), 1.0 + rank, world)
    bench.barrier(world)
    q.put((rank, agg))
    dist.destroy_process_group()


def test_aggregate_two_ranks_gloo():
    ctx = mp.get_context("spawn")
    q = ctx.Queue()
    port = _free_port()
    procs = [ctx.Process(target=_rank_main, args=(r, 2, port, q)) for r in range(2)]
    for p in procs:
        p.start()
    res = dict(q.get(timeout=120) for _ in range(2))
    for p in procs:
        p.join(timeout=60)
        assert p.exitcode == 0
    for r in range(2):
        assert res[r]["seconds"] == 2.0           # the slowest rank's time
        assert res[r]["units"] == 300.0           # every rank's units
        assert res[r]["value"] == pytest.approx(150.0)


def test_aggregate_single_rank():
    assert bench.aggregate(10.0, 2.0, 1) == {"seconds": 2.0, "units": 10.0, "value": 5.0}


def test_clock_parser():
    lines = [
        "0, 1980, 2070, 700.5, 0x0000000000000004, Not Active, Not Active, Not Active, Active",
        "0, 2070, 2070, 650.0, 0x0000000000000000, Not Active, Not Active, Not Active, Not Active",
        "0, 2010, 2070, 690.0, 0x0000000000000000, Not Active, Not Active, Not Active, Not Active",
        "garbage",
    ]
    c = bench.ClockSampler.parse(lines)
    assert c["sm_mhz"] == 2010 and c["sm_max_mhz"] == 2070 and c["samples"] == 3
    assert c["reasons"] == ["sw_power_cap"]
    assert bench.ClockSampler.parse([])["sm_mhz"] is None


def test_work_formulas():
    # decode: 132,019 bytes per head.token at B = 64 (state 131,072 + activations)
    assert bench.decode_bytes_per_launch(64) == 405_561_344
    assert round(bench.decode_bytes_per_launch(64) / (64 * 48)) == 132_019
    # one fp32 state update: 6 d^2 + 5 d flops
    assert bench.step_flops_per_head_token() == 6 * 128 * 128 + 5 * 128
    # prefill over 8,192 tokens, chunk 64
    assert bench.prefill_flops(8192) == 128 * (48 * (4 * 64 * 128 * 128 + 4 * 64 * 64 * 128 +
                                                     2 * 128 * 128 * 64 + 64 ** 3 // 3)
                                               + 16 * 4 * 64 * 64 * 128)
    assert bench.prefill_flops(65) == 2 * bench.prefill_flops(64)
    assert bench.fp32_alu_peak_tflops(2070.0) == pytest.approx(152 * 128 * 2 * 2.07e9 / 1e12)
    # KDA: alpha carries 128 fp32 decays per head.token instead of one
    assert bench.kda_fused_bytes_per_launch(64) - bench.fused_bytes_per_launch(64) == 64 * 48 * 127 * 4
    # the layer step: the fused bytes with bf16 gate projections and y instead of fp32 gates and outputs,
    # plus z, the per-head parameters and the norm weight
    assert bench.layer_bytes_per_launch(64) == (bench.fused_bytes_per_launch(64) - 64 * 48 * (8 + 128 * 4)
                                                + 64 * 48 * 4 + 48 * 8 + 2 * 64 * 48 * 128 * 2 + 128 * 4)
    # snapshot payload of one sequence: 48 layers x (fp32 state + bf16 tail)
    assert bench.snapshot_payload_bytes(48) == 48 * (48 * 128 * 128 * 4 + 4 * 10240 * 2) == 154_927_104


def test_peaks_present_or_fallback():
    peaks, kind = bench.load_peaks()
    assert kind in ("measured", "fallback")
    assert peaks["hbm_gbs"] > 1000 and peaks["bf16_tflops"] > 100


@pytest.mark.parametrize("workload", ["batched", "tree", "kdabatch", "snapshot", "layer"])
def test_reference_arm_line(workload):
    out = subprocess.run([sys.executable, os.path.join(ROOT, "bench.py"), "--impl", "reference",
                          "--workload", workload, "--steps", "2", "--warmup", "3"],
                         capture_output=True, text=True, timeout=300, check=True).stdout
    lines = [ln for ln in out.splitlines() if ln.strip()]
    assert len(lines) == 1
    d = json.loads(lines[0])
    assert d["impl"] == "reference" and d["value"] > 0 and d["warmup"] == 3
    assert d["cpu_baseline"]["kind"] == "oracle" and d["cpu_baseline"]["cores"] == 1
    assert d["e2e"]["h2d_bytes_per_step"] == 0 and d["e2e"]["value"] == d["value"]


def test_reference_arm_nonzero_rank_is_silent():
    env = dict(os.environ, RANK="1", WORLD_SIZE="2", LOCAL_RANK="1")
    out = subprocess.run([sys.executable, os.path.join(ROOT, "bench.py"), "--impl", "reference",
                          "--steps", "1"], capture_output=True, text=True, timeout=120, env=env, check=True)
    assert out.stdout.strip() == ""


def test_reference_arm_default_is_the_headline():
    """With no --workload the reference arm times the headline (batched) config."""
    out = subprocess.run([sys.executable, os.path.join(ROOT, "bench.py"), "--impl", "reference", "--steps", "2",
                          "--warmup", "3"], capture_output=True, text=True, timeout=300, check=True).stdout
    d = json.loads(out.strip().splitlines()[-1])
    assert d["config"]["workload"].startswith("batched decode")
    assert d["cpu_baseline"]["host"]["nproc"] >= 1


def test_cpu_baselines_single_and_all_cores():
    """The CPU baseline: one thread, and the same sample on every core, with the
    host's core count and CPU model."""
    b = bench.cpu_baselines("decode1", 0.2)
    assert b["cores"] == 1 and b["value"] > 0 and b["kind"] == "oracle"
    assert b["host"]["nproc"] == (os.cpu_count() or 1) and b["host"]["cpu_model"]
    if b["host"]["nproc"] > 1:
        allc = b["all_cores"]
        assert allc["cores"] == b["host"]["nproc"] and allc["value"] > 0
