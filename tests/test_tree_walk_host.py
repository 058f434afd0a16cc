"""The tree verify's walk schedules, checked on the host (no GPU).

tests/tree_walk_check.cu includes the host API's translation unit, builds
the single depth-first walk and the two- and three-walker splits for
thousands of random trees, and replays each schedule as the kernel walks it
(parent state taken from the right register set or slot, slots in range,
every node stored exactly once, the longest split walk at most 3/4 of the
tree).  It links against the library's other objects, which the build
leaves in the package's _build folder."""
import os
import shutil
import subprocess

import pytest

ROOT = os.path.dirname(os.path.dirname(os.path.abspath(__file__)))


def test_walk_schedules_replay(tmp_path):
    nvcc = shutil.which("nvcc") or "/usr/local/cuda/bin/nvcc"
    if not os.path.exists(nvcc):
        pytest.skip("nvcc not available")
    from hybrid_linear_attention_conv_gb300 import build
    build.build()
    objs = [os.path.join(build.BUILD, f + ".o") for f in ("gdn_decode", "gdn_conv", "gdn_prefill", "gdn_snapshot")]
    exe = str(tmp_path / "tree_walk_check")
    cmd = [nvcc, "-std=c++17", "-O1", *build.ARCH, "-I", build.INCLUDE, "-I", build.CSRC,
           os.path.join(ROOT, "tests", "tree_walk_check.cu"), *objs, "-o", exe]
    r = subprocess.run(cmd, capture_output=True, text=True)
    assert r.returncode == 0, r.stderr[-3000:]
    r = subprocess.run([exe], capture_output=True, text=True, timeout=300)
    assert r.returncode == 0 and "schedules OK" in r.stdout, (r.stdout[-2000:], r.stderr[-2000:])
