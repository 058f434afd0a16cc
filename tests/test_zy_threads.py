"""First calls from several host threads at once.

The library sets each device up on first use: shared-memory opt-ins for the
tree, fused-decode and prefill kernels, the cooperative-launch capacity, the
SM count.  That set-up is guarded (std::call_once, a mutex, atomics).  This
test makes those first calls from six host threads at the same moment, each on
its own stream, in a fresh process (so that nothing is set up yet), and checks
every result against the same call made again afterwards, bit for bit."""
import os
import subprocess
import sys

import pytest

pytestmark = pytest.mark.gpu

ROOT = os.path.dirname(os.path.dirname(os.path.abspath(__file__)))

SCRIPT = r'''
import sys, threading
sys.path.insert(0, ROOT)
sys.path.insert(0, ROOT + "/tests")
import numpy as np, torch
from hybrid_linear_attention_conv_gb300 import gdn, inputs as gen
from gdn_testutil import bf16, f32
gdn.load()
torch.cuda.init()
s = gen.QWEN_27B
N = 32
parents = gen.random_tree(300, N, 8)
d = gen.decode_inputs(301, s, N, tag="thr")
k = gen.kda_inputs(302, s, N, tag="thr")
c = gen.conv_inputs(303, 1, N, s.C, tag="thr")
db = gen.decode_inputs(304, s.with_batch(64), 1, tag="thrb")
cb = gen.conv_inputs(305, 64, 1, s.C, tag="thrb")
dp = gen.decode_inputs(306, s, 300, tag="thrp")
trees = [gen.random_tree(310 + b, 32, 8) for b in range(4)]
pb = np.stack(trees).astype(np.int32)
dj = gen.decode_inputs(307, s.with_batch(4), 32, tag="thrj")

def tree():
    return gdn.tree_verify(parents, bf16(d["qkv"][0]), f32(d["alpha"][0]), f32(d["beta"][0]), f32(d["state"][0]),
                           s.Hk, s.Hv, s.dk, s.dv)
def conv_tree():
    return gdn.conv_tree_verify(parents, bf16(c["x"][0]), bf16(c["w"]), bf16(c["tail"][0]), f32(d["alpha"][0]),
                                f32(d["beta"][0]), f32(d["state"][0]), s.Hk, s.Hv, s.dk, s.dv)
def kda_tree():
    return gdn.kda_tree_verify(parents, bf16(k["qkv"][0]), f32(k["alpha"][0]), f32(k["beta"][0]), f32(k["state"][0]),
                               s.Hk, s.Hv, s.dk, s.dv)
def joint():
    return gdn.tree_verify_batched(np.full(4, 32, np.int32), pb, bf16(dj["qkv"]), f32(dj["alpha"]), f32(dj["beta"]),
                                   f32(dj["state"]), s.Hk, s.Hv, s.dk, s.dv)
def fused_b64():
    st = f32(db["state"])
    out = gdn.conv_decode_step(bf16(cb["x"]), bf16(cb["w"]), bf16(cb["tail"]), f32(db["alpha"]), f32(db["beta"]), st,
                               s.Hk, s.Hv, s.dk, s.dv)
    return torch.cat([out.flatten(), st.flatten()])
def prefill():
    st = f32(dp["state"][0])
    out = gdn.chunk_prefill(bf16(dp["qkv"][0]), f32(dp["alpha"][0]), f32(dp["beta"][0]), st, s.Hk, s.Hv, s.dk, s.dv)
    return torch.cat([out.flatten(), st.flatten()])

fns = [tree, conv_tree, kda_tree, joint, fused_b64, prefill]
results = [None] * len(fns)
errors = []
gate = threading.Barrier(len(fns))
def work(i):
    try:
        stream = torch.cuda.Stream()
        with torch.cuda.stream(stream):
            gate.wait()
            r = fns[i]()
        stream.synchronize()
        results[i] = r
    except Exception as e:
        errors.append(repr(e))
threads = [threading.Thread(target=work, args=(i,)) for i in range(len(fns))]
for t in threads: t.start()
for t in threads: t.join(120)
torch.cuda.synchronize()
assert not errors, errors
for i, fn in enumerate(fns):
    again = fn()
    torch.cuda.synchronize()
    assert torch.equal(results[i], again), fn.__name__
print("THREADS OK")
'''


def test_first_calls_from_several_threads():
    code = "ROOT = " + repr(ROOT) + "\n" + SCRIPT
    r = subprocess.run([sys.executable, "-c", code], capture_output=True, text=True, timeout=600, cwd=ROOT)
    assert r.returncode == 0 and "THREADS OK" in r.stdout, (r.stdout[-2000:], r.stderr[-4000:])
