"""Pins for the fp64 oracle: each check ties it to something other than itself
(hand-worked examples, the textbook matrix form, library routines, invariants
of the recurrence, exhaustive enumeration, brute force on tiny inputs)."""
import itertools
import math

import numpy as np
import pytest

import oracle
from hybrid_linear_attention_conv_gb300 import inputs as gen
from conftest import read_golden


def _bf16(vals):
    return gen.f32_to_bf16_bits(np.asarray(vals, np.float32))


# ---------------------------------------------------------------------------
# bf16 storage conversion
# ---------------------------------------------------------------------------
def test_bf16_widen_exhaustive():
    """All 65,536 bf16 patterns widen exactly (numpy's own fp32 view as the check)."""
    h = np.arange(65536, dtype=np.uint32).astype(np.uint16)
    got = oracle.bf16_to_f64(h)
    with np.errstate(invalid="ignore"):
        want = (h.astype(np.uint32) << 16).view(np.float32).astype(np.float64)
    nan = np.isnan(want)
    assert np.array_equal(np.isnan(got), nan)
    assert np.array_equal(got[~nan], want[~nan])


def test_bf16_round_exhaustive_roundtrip_and_ties():
    """Every finite bf16 value rounds to itself; every midpoint between two
    neighbours rounds to the one with an even last bit; a hair above or below a
    midpoint rounds to the nearer neighbour."""
    h = np.arange(65536, dtype=np.uint32).astype(np.uint16)
    with np.errstate(invalid="ignore"):
        f = (h.astype(np.uint32) << 16).view(np.float32).astype(np.float64)
    fin = np.isfinite(f)
    assert np.array_equal(oracle.f64_to_bf16(f[fin]), h[fin])
    # positive finite ladder 0x0000 .. 0x7F7F
    lo = np.arange(0, 0x7F7F, dtype=np.uint32).astype(np.uint16)
    a = (lo.astype(np.uint32) << 16).view(np.float32).astype(np.float64)
    b = ((lo.astype(np.uint32) + 1) << 16).view(np.float32).astype(np.float64)
    mid = (a + b) / 2.0  # exact in fp64
    got = oracle.f64_to_bf16(mid)
    even = np.where(lo % 2 == 0, lo, lo + 1).astype(np.uint16)
    assert np.array_equal(got, even)
    up = oracle.f64_to_bf16(mid + (b - a) * 2.0 ** -20)
    dn = oracle.f64_to_bf16(mid - (b - a) * 2.0 ** -20)
    assert np.array_equal(up, (lo + 1).astype(np.uint16))
    assert np.array_equal(dn, lo)
    # signs and specials
    assert oracle.f64_to_bf16(np.array([-1.0]))[0] == 0xBF80
    assert oracle.f64_to_bf16(np.array([np.inf]))[0] == 0x7F80
    assert oracle.f64_to_bf16(np.array([-np.inf]))[0] == 0xFF80
    assert oracle.f64_to_bf16(np.array([3.5e38]))[0] == 0x7F80  # overflow after rounding


def test_bf16_round_matches_generator_rounding():
    """For fp32 inputs the oracle's direct fp64->bf16 rounding and the generator's
    bit-level fp32->bf16 rounding are independent implementations of the same RNE."""
    x = gen.normal_f32(7, "bf16check", (200000,), 3.0)
    x = np.concatenate([x, np.float32([1e-39, -2e-40, 1.0e-45, 3.0e38])])
    assert np.array_equal(oracle.f64_to_bf16(x.astype(np.float64)), gen.f32_to_bf16_bits(x))


# ---------------------------------------------------------------------------
# conv + SiLU
# ---------------------------------------------------------------------------
def test_silu_closed_forms():
    assert oracle.silu(0.0) == 0.0
    assert oracle.silu(1.0) == pytest.approx(1.0 / (1.0 + math.exp(-1.0)), rel=1e-15)
    for z in [-7.5, -1.0, 0.3, 2.0, 11.0]:
        # z*sig(z) - (-z)*sig(-z) = z
        assert oracle.silu(z) - oracle.silu(-z) == pytest.approx(z, rel=1e-14)
    assert oracle.silu(60.0) == pytest.approx(60.0, rel=1e-15)
    assert abs(oracle.silu(-60.0)) < 1e-20


def test_conv_golden_one_channel():
    g = read_golden("conv_one_channel.txt")
    x = _bf16(g["x"]).reshape(1, 2, 1)
    w = _bf16(g["w"]).reshape(1, 4)
    tail = _bf16(g["tail"]).reshape(1, 4, 1)
    y, tail2 = oracle.conv_linear(x, w, tail)
    for t, z in enumerate(g["z"]):
        assert y[0, t, 0] == pytest.approx(z / (1.0 + math.exp(-z)), rel=1e-15)
    assert np.array_equal(gen.bf16_bits_to_f32(tail2.ravel()), np.float32(g["tail_after"]))


def test_conv_tap_selection():
    """Taps (0,0,0,1) pass the newest input; (1,0,0,0) delay by three steps."""
    d = gen.conv_inputs(3, 2, 9, 40)
    silu = lambda z: z / (1.0 + np.exp(-z))
    xs = gen.bf16_bits_to_f32(d["x"]).astype(np.float64)
    ts = gen.bf16_bits_to_f32(d["tail"]).astype(np.float64)
    w = np.zeros((40, 4), np.float32)
    w[:, 3] = 1.0
    y, _ = oracle.conv_linear(d["x"], gen.f32_to_bf16_bits(w), d["tail"])
    np.testing.assert_allclose(y, silu(xs), rtol=1e-15, atol=0)
    w = np.zeros((40, 4), np.float32)
    w[:, 0] = 1.0
    y, _ = oracle.conv_linear(d["x"], gen.f32_to_bf16_bits(w), d["tail"])
    hist = np.concatenate([ts, xs], axis=1)  # [B, 4+T, C]
    np.testing.assert_allclose(y, silu(hist[:, 1:1 + 9]), rtol=1e-15, atol=0)


def test_conv_matches_numpy_correlate():
    """Pre-activation equals numpy's 'valid' cross-correlation of the history
    (tail ++ x) with the taps; the new tail is the last four inputs."""
    B, T, C = 2, 11, 17
    d = gen.conv_inputs(5, B, T, C)
    y, tail2 = oracle.conv_linear(d["x"], d["w"], d["tail"])
    xs = gen.bf16_bits_to_f32(d["x"]).astype(np.float64)
    ts = gen.bf16_bits_to_f32(d["tail"]).astype(np.float64)
    ws = gen.bf16_bits_to_f32(d["w"]).astype(np.float64)
    for b in range(B):
        for c in range(C):
            hist = np.concatenate([ts[b, :, c], xs[b, :, c]])
            z = np.correlate(hist, ws[c], mode="valid")[1:]
            np.testing.assert_allclose(y[b, :, c], z / (1.0 + np.exp(-z)), rtol=1e-13, atol=1e-15)
    assert np.array_equal(tail2, np.concatenate([d["tail"], d["x"]], axis=1)[:, -4:, :])


def test_conv_streaming_equals_one_call():
    d = gen.conv_inputs(9, 2, 7, 33)
    y_all, tail_all = oracle.conv_linear(d["x"], d["w"], d["tail"])
    tail = d["tail"]
    ys = []
    for t in range(7):
        y, tail = oracle.conv_linear(d["x"][:, t:t + 1], d["w"], tail)
        ys.append(y)
    assert np.array_equal(np.concatenate(ys, axis=1), y_all)
    assert np.array_equal(tail, tail_all)


def test_conv_tree_chain_and_replay():
    C = 24
    d = gen.conv_inputs(4, 1, 12, C)
    chain = np.arange(-1, 11, dtype=np.int32)
    y_lin, _ = oracle.conv_linear(d["x"], d["w"], d["tail"])
    y_tree = oracle.conv_tree(chain, d["x"][0], d["w"], d["tail"][0])
    assert np.array_equal(y_tree, y_lin[0])
    parents = gen.random_tree(11, 12, 5)
    y_tree = oracle.conv_tree(parents, d["x"][0], d["w"], d["tail"][0])
    for n in range(12):
        p = oracle.root_path(parents, n)
        y_path, _ = oracle.conv_linear(d["x"][:, p], d["w"], d["tail"])
        assert np.array_equal(y_tree[n], y_path[0, -1])


def test_conv_r32_closed_forms():
    """The binary32-decided conv on inputs whose outputs are known in closed
    form: SiLU(1) = 1/(1+e^-1) = 0.7310586 -> bf16 0.73046875 (0x3F3B),
    SiLU(-1) = -0.2689414 -> -0.26953125 (0xBE8A), SiLU(1+2) = 2.857722 ->
    2.859375 (0x4037), SiLU(0) = 0."""
    one, two = 0x3F80, 0x4000
    w = np.array([[0, 0, 0, one], [0, 0, 0, one], [0, 0, one, one], [one, one, one, one]], np.uint16)
    tail = np.zeros((1, 4, 4), np.uint16)
    tail[0, 3, 2] = one  # the newest tail input of channel 2
    x = np.array([[[one, 0xBF80, two, 0]]], np.uint16)  # 1, -1, 2, 0
    y, new_tail = oracle.conv_linear_r32(x, w, tail)
    assert y[0, 0].tolist() == [0x3F3B, 0xBE8A, 0x4037, 0]
    assert new_tail[0, 3].tolist() == x[0, 0].tolist()


def test_conv_r32_within_one_ulp_of_fp64():
    """Deciding the bf16 rounding in binary32 moves an output by at most one
    bf16 ulp from rounding the fp64 conv, and almost never (the binary32 value
    is within a few of its ulps of the exact one, and a bf16 midpoint lies
    between the two only rarely); the tail is the same."""
    d = gen.conv_inputs(12, 2, 48, 1024, tag="r32")
    y64, t64 = oracle.conv_linear(d["x"], d["w"], d["tail"])
    y16, t16 = oracle.conv_linear_r32(d["x"], d["w"], d["tail"])
    ref = oracle.f64_to_bf16(y64)
    key = lambda b: np.where(b.astype(np.int32) & 0x8000, -(b.astype(np.int32) & 0x7FFF), b.astype(np.int32))
    ulp = np.abs(key(ref) - key(y16))
    assert ulp.max() <= 1
    assert (ulp == 0).mean() > 0.999
    assert np.array_equal(t64, t16)


def test_conv_tree_r32_chain_and_root_paths():
    """The binary32-decided tree conv: a chain is the linear run, and every
    node of a random tree is the linear run over its root path."""
    C = 24
    d = gen.conv_inputs(5, 1, 12, C, tag="r32t")
    chain = np.arange(-1, 11, dtype=np.int32)
    y_lin, _ = oracle.conv_linear_r32(d["x"], d["w"], d["tail"])
    assert np.array_equal(oracle.conv_tree_r32(chain, d["x"][0], d["w"], d["tail"][0]), y_lin[0])
    parents = gen.random_tree(12, 12, 5)
    y_tree = oracle.conv_tree_r32(parents, d["x"][0], d["w"], d["tail"][0])
    for n in range(12):
        p = oracle.root_path(parents, n)
        y_path, _ = oracle.conv_linear_r32(d["x"][:, p], d["w"], d["tail"])
        assert np.array_equal(y_tree[n], y_path[0, -1])


# ---------------------------------------------------------------------------
# tree bookkeeping: brute force over every tree of up to 7 nodes
# ---------------------------------------------------------------------------
def _all_trees(N):
    for tail in itertools.product(*[range(i) for i in range(1, N)]):
        yield np.array((-1,) + tail, np.int32)


def test_tree_bookkeeping_brute_force():
    count = 0
    for N in range(1, 8):
        for parents in _all_trees(N):
            count += 1
            rc, depth = oracle.tree_check(parents)
            assert rc == 0
            paths = set()
            for n in range(N):
                p = oracle.root_path(parents, n)
                # walk by hand: consecutive parent links, starts at the root
                assert p[-1] == n and parents[p[0]] == -1
                assert all(parents[p[i]] == p[i - 1] for i in range(1, len(p)))
                assert len(p) == depth[n]
                for L in range(len(p) + 1):
                    paths.add(tuple(p[:L]))
            # every sequence of length <= 3 over the nodes: valid iff a root path
            if N <= 5:
                for L in range(0, 4):
                    for seq in itertools.product(range(N), repeat=L):
                        ok = oracle.path_check(parents, np.array(seq, np.int32)) == 0
                        assert ok == (tuple(seq) in paths), (parents, seq)
    assert count == sum(math.factorial(n - 1) for n in range(1, 8))


def test_tree_check_rejects():
    assert oracle.tree_check(np.array([0], np.int32))[0] < 0
    assert oracle.tree_check(np.array([-1, 1], np.int32))[0] < 0
    assert oracle.tree_check(np.array([-1, 0, -1], np.int32))[0] < 0
    assert oracle.tree_check(np.array([-1, 0, 3, 1], np.int32))[0] < 0
    assert oracle.tree_check(np.array([-1, -2], np.int32))[0] < 0


def test_random_tree_generator_shape():
    for seed in range(20):
        parents = gen.random_tree(seed, 32, 8)
        rc, depth = oracle.tree_check(parents)
        assert rc == 0 and len(parents) == 32 and depth.max() <= 8
        kids = np.bincount(parents[parents >= 0], minlength=32)
        assert kids.max() <= 4


# ---------------------------------------------------------------------------
# gated delta rule
# ---------------------------------------------------------------------------
def test_delta_golden_2x2():
    g = read_golden("delta_rule_2x2.txt")
    S0 = np.array(g["S0"]).reshape(2, 2)
    for matrix_form in (False, True):
        S1, o = oracle.delta_token(S0, g["k"], g["v"], g["q"], g["alpha"][0], g["beta"][0],
                                   matrix_form=matrix_form)
        np.testing.assert_allclose(S1.ravel(), g["S1"], rtol=0, atol=1e-15)
        np.testing.assert_allclose(o, g["o"], rtol=0, atol=1e-15)


def _textbook(S, k, v, q, alpha, beta):
    dk = len(k)
    S1 = alpha * S @ (np.eye(dk) - beta * np.outer(k, k)) + beta * np.outer(v, k)
    return S1, S1 @ q


@pytest.mark.parametrize("dk,dv", [(5, 3), (3, 7), (32, 32)])
def test_delta_row_form_vs_matrix_forms(dk, dv):
    rng_n = gen.normal(1, f"d{dk}{dv}", dv * dk + 3 * dk + dv)
    S = rng_n[: dv * dk].reshape(dv, dk)
    k = rng_n[dv * dk: dv * dk + dk]
    q = rng_n[dv * dk + dk: dv * dk + 2 * dk]
    v = rng_n[dv * dk + 2 * dk: dv * dk + 2 * dk + dv]
    k = k / np.linalg.norm(k)
    S_row, o_row = oracle.delta_token(S, k, v, q, 0.93, 0.61)
    S_mat, o_mat = oracle.delta_token(S, k, v, q, 0.93, 0.61, matrix_form=True)
    S_np, o_np = _textbook(S, k, v, q, 0.93, 0.61)
    np.testing.assert_allclose(S_row, S_np, rtol=0, atol=1e-13)
    np.testing.assert_allclose(S_mat, S_np, rtol=0, atol=1e-13)
    np.testing.assert_allclose(o_row, o_np, rtol=0, atol=1e-12)
    np.testing.assert_allclose(o_mat, o_np, rtol=0, atol=1e-12)


def test_delta_invariants():
    dk, dv = 16, 12
    n = gen.normal(2, "inv", dv * dk + 3 * dk + dv)
    S = n[: dv * dk].reshape(dv, dk)
    k = n[dv * dk: dv * dk + dk]
    k = k / np.linalg.norm(k)
    q = n[dv * dk + dk: dv * dk + 2 * dk]
    v = n[dv * dk + 2 * dk: dv * dk + 2 * dk + dv]
    # beta = 0, alpha = 1: state unchanged, o = S q
    S1, o = oracle.delta_token(S, k, v, q, 1.0, 0.0)
    assert np.array_equal(S1, S)
    np.testing.assert_allclose(o, S @ q, rtol=0, atol=1e-13)
    # beta = 0: pure decay
    S1, o = oracle.delta_token(S, k, v, q, 0.7, 0.0)
    np.testing.assert_allclose(S1, 0.7 * S, rtol=1e-15, atol=0)
    # alpha = 1, beta = 1, unit k: the new state maps k to v exactly
    S1, _ = oracle.delta_token(S, k, v, q, 1.0, 1.0)
    np.testing.assert_allclose(S1 @ k, v, rtol=0, atol=1e-13)
    # S0 = 0, one token: o = beta * v * (k . q)
    S1, o = oracle.delta_token(np.zeros_like(S), k, v, q, 0.9, 0.4)
    np.testing.assert_allclose(o, 0.4 * v * (k @ q), rtol=0, atol=1e-14)
    # rank-1 change: S1 - alpha*S has rank one, along k
    S1, _ = oracle.delta_token(S, k, v, q, 0.8, 0.3)
    sv = np.linalg.svd(S1 - 0.8 * S, compute_uv=False)
    assert sv[1] < 1e-12 * sv[0]


def test_l2norm():
    out = oracle.l2norm(np.array([3.0, 4.0]))
    np.testing.assert_allclose(out, np.array([3.0, 4.0]) / math.sqrt(25.0 + 1e-6), rtol=1e-15)
    assert np.array_equal(oracle.l2norm(np.zeros(8)), np.zeros(8))
    x = gen.normal(3, "l2", 128)
    np.testing.assert_allclose(np.linalg.norm(oracle.l2norm(x, eps=0.0)), 1.0, rtol=1e-14)


def _decode_textbook(d, shape, T, q_scale=1.0, normalize=True):
    """Independent numpy decode: matrix form, numpy norms, explicit head map
    (qkv as bf16 bits, or as fp32 values)."""
    B, Hk, Hv, dk, dv = shape.B, shape.Hk, shape.Hv, shape.dk, shape.dv
    qkv = d["qkv"].astype(np.float64) if d["qkv"].dtype == np.float32 else \
        gen.bf16_bits_to_f32(d["qkv"]).astype(np.float64)
    S = d["state"].astype(np.float64).copy()
    out = np.zeros((B, T, Hv, dv))
    for b in range(B):
        for t in range(T):
            row = qkv[b, t]
            qh = row[: Hk * dk].reshape(Hk, dk)
            kh = row[Hk * dk: 2 * Hk * dk].reshape(Hk, dk)
            vh = row[2 * Hk * dk:].reshape(Hv, dv)
            for h in range(Hv):
                g = h * Hk // Hv
                q, k = qh[g], kh[g]
                if normalize:
                    q = q / math.sqrt(q @ q + 1e-6)
                    k = k / math.sqrt(k @ k + 1e-6)
                S[b, h], out[b, t, h] = _textbook(S[b, h], k, vh[h], q * q_scale,
                                                  float(d["alpha"][b, t, h]), float(d["beta"][b, t, h]))
    return out, S


@pytest.mark.parametrize("shape", [gen.Shape(2, 2, 4, 8, 6), gen.Shape(1, 1, 3, 5, 4), gen.TINY])
def test_decode_vs_textbook(shape):
    T = 5
    d = gen.decode_inputs(21, shape, T)
    out, st = oracle.decode(d["qkv"], d["alpha"], d["beta"], d["state"], shape.Hk, shape.Hv,
                            shape.dk, shape.dv, q_scale=0.75)
    out_t, st_t = _decode_textbook(d, shape, T, q_scale=0.75)
    np.testing.assert_allclose(out, out_t, rtol=0, atol=1e-12)
    np.testing.assert_allclose(st, st_t, rtol=0, atol=1e-12)
    out, st = oracle.decode(d["qkv"], d["alpha"], d["beta"], d["state"], shape.Hk, shape.Hv,
                            shape.dk, shape.dv, normalize=False)
    out_t, st_t = _decode_textbook(d, shape, T, normalize=False)
    np.testing.assert_allclose(out, out_t, rtol=1e-12, atol=1e-10)


@pytest.mark.parametrize("shape", [gen.Shape(2, 2, 4, 8, 6), gen.TINY])
def test_decode_f32_vs_textbook(shape):
    """The fp32-activation decode against the independent numpy decode on fp32
    draws (values that bf16 cannot hold, so a stray rounding would show)."""
    T = 6
    d = gen.decode_inputs_f32(22, shape, T)
    assert not np.array_equal(gen.bf16_bits_to_f32(gen.f32_to_bf16_bits(d["qkv"])), d["qkv"])
    out, st = oracle.decode_f32(d["qkv"], d["alpha"], d["beta"], d["state"], shape.Hk, shape.Hv,
                                shape.dk, shape.dv, q_scale=0.75)
    out_t, st_t = _decode_textbook(d, shape, T, q_scale=0.75)
    np.testing.assert_allclose(out, out_t, rtol=0, atol=1e-12)
    np.testing.assert_allclose(st, st_t, rtol=0, atol=1e-12)


def test_decode_f32_equals_bf16_decode_on_bf16_values():
    """Widening is exact, so fp32 inputs that bf16 holds exactly give the bf16
    decode's results bit for bit."""
    s = gen.Shape(2, 2, 4, 16, 8)
    d = gen.decode_inputs(23, s, 4)
    out, st = oracle.decode(d["qkv"], d["alpha"], d["beta"], d["state"], s.Hk, s.Hv, s.dk, s.dv)
    out32, st32 = oracle.decode_f32(gen.bf16_bits_to_f32(d["qkv"]), d["alpha"], d["beta"], d["state"], s.Hk,
                                    s.Hv, s.dk, s.dv)
    assert np.array_equal(out, out32) and np.array_equal(st, st32)


def test_conv_f32_matches_numpy_correlate_and_bf16_conv():
    """The fp32 conv: numpy's cross-correlation of (tail ++ x) with the taps,
    then SiLU; the new tail is the last four inputs; on bf16-held values it is
    the bf16 conv exactly."""
    B, T, C = 2, 9, 16
    d = gen.conv_inputs_f32(6, B, T, C, zero_tail=False)
    y, tail2 = oracle.conv_linear_f32(d["x"], d["w"], d["tail"])
    for b in range(B):
        for c in range(C):
            hist = np.concatenate([d["tail"][b, :, c], d["x"][b, :, c]]).astype(np.float64)
            z = np.correlate(hist, d["w"][c].astype(np.float64), mode="valid")[1:]
            np.testing.assert_allclose(y[b, :, c], z / (1.0 + np.exp(-z)), rtol=1e-13, atol=1e-15)
    assert np.array_equal(tail2, np.concatenate([d["tail"], d["x"]], axis=1)[:, -4:, :])
    h = gen.conv_inputs(7, B, T, C)
    y16, t16 = oracle.conv_linear(h["x"], h["w"], h["tail"])
    y32, t32 = oracle.conv_linear_f32(gen.bf16_bits_to_f32(h["x"]), gen.bf16_bits_to_f32(h["w"]),
                                      gen.bf16_bits_to_f32(h["tail"]))
    assert np.array_equal(y16, y32) and np.array_equal(gen.bf16_bits_to_f32(t16), t32)


def test_decode_key_head_map():
    """Value heads 0,1 read key head 0 and heads 2,3 read key head 1 (Hk=2, Hv=4):
    changing key head 1's q and k moves only heads 2 and 3."""
    s = gen.TINY
    d = gen.decode_inputs(4, s, 3)
    out, _ = oracle.decode(d["qkv"], d["alpha"], d["beta"], d["state"], s.Hk, s.Hv, s.dk, s.dv)
    qkv2 = d["qkv"].copy()
    qkv2[..., s.dk: 2 * s.dk] = gen.normal_bf16(99, "q1", (1, 3, s.dk))
    qkv2[..., s.Hk * s.dk + s.dk: 2 * s.Hk * s.dk] = gen.normal_bf16(99, "k1", (1, 3, s.dk))
    out2, _ = oracle.decode(qkv2, d["alpha"], d["beta"], d["state"], s.Hk, s.Hv, s.dk, s.dv)
    assert np.array_equal(out2[:, :, :2], out[:, :, :2])
    assert np.abs(out2[:, :, 2:] - out[:, :, 2:]).min() > 0


def test_decode_streaming_and_batch_independence():
    s = gen.Shape(3, 2, 4, 8, 8)
    d = gen.decode_inputs(8, s, 6)
    out, st = oracle.decode(d["qkv"], d["alpha"], d["beta"], d["state"], 2, 4, 8, 8)
    o1, st1 = oracle.decode(d["qkv"][:, :2], d["alpha"][:, :2], d["beta"][:, :2], d["state"], 2, 4, 8, 8)
    o2, st2 = oracle.decode(d["qkv"][:, 2:], d["alpha"][:, 2:], d["beta"][:, 2:], st1, 2, 4, 8, 8)
    assert np.array_equal(np.concatenate([o1, o2], axis=1), out)
    assert np.array_equal(st2, st)
    ob, stb = oracle.decode(d["qkv"][1:2], d["alpha"][1:2], d["beta"][1:2], d["state"][1:2], 2, 4, 8, 8)
    assert np.array_equal(ob, out[1:2]) and np.array_equal(stb, st[1:2])


def test_tree_verify_equals_path_decode():
    s = gen.Shape(1, 2, 4, 8, 8)
    N = 14
    parents = gen.random_tree(6, N, 5)
    d = gen.decode_inputs(6, s.with_batch(1), N, tag="tree")
    qkv, al, be = d["qkv"][0], d["alpha"][0], d["beta"][0]
    out = oracle.tree_verify(parents, qkv, al, be, d["state"][0], 2, 4, 8, 8)
    for n in range(N):
        p = oracle.root_path(parents, n)
        o, _ = oracle.decode(qkv[None, p], al[None, p], be[None, p], d["state"], 2, 4, 8, 8)
        assert np.array_equal(out[n], o[0, -1])
    # a chain is plain decode
    chain = np.arange(-1, N - 1, dtype=np.int32)
    out = oracle.tree_verify(chain, qkv, al, be, d["state"][0], 2, 4, 8, 8)
    o, _ = oracle.decode(d["qkv"], d["alpha"], d["beta"], d["state"], 2, 4, 8, 8)
    assert np.array_equal(out, o[0])


def test_commit_equals_path_decode_and_tail():
    s = gen.Shape(1, 2, 4, 8, 8)
    N = 16
    parents = gen.random_tree(12, N, 6)
    d = gen.decode_inputs(12, s, N, tag="commit")
    c = gen.conv_inputs(12, 1, N, s.C)
    leaf = gen.random_leaf(12, parents)
    path = oracle.root_path(parents, leaf)
    for L in range(0, len(path) + 1):
        P = path[:L]
        st, tail = oracle.commit(parents, P, d["qkv"][0], d["alpha"][0], d["beta"][0], d["state"][0],
                                 2, 4, 8, 8, x_tree=c["x"][0], tail=c["tail"][0])
        _, st_ref = oracle.decode(d["qkv"][:, P], d["alpha"][:, P], d["beta"][:, P], d["state"], 2, 4, 8, 8)
        assert np.array_equal(st, st_ref[0])
        hist = np.concatenate([c["tail"][0], c["x"][0][P]], axis=0)
        assert np.array_equal(tail, hist[-4:])


def _chunk_form(qkv, alpha, beta, S0, Hk, Hv, dk, dv, chunk):
    """fp64 emulation of the WY/UT chunk form (Yang et al. 2024, 'Parallelizing
    Linear Transformers with the Delta Rule over Sequence Length', and the gated
    variant in 'Gated Delta Networks'): per chunk, gamma = cumprod(alpha),
    T = (I + L)^-1 with L_ts = beta_t (gamma_t/gamma_s) k_t.k_s (s < t),
    W = T diag(beta gamma) K, U~ = T diag(beta) V, U = U~ - W S0^T,
    O = diag(gamma) Q S0^T + (M o Q K^T) U, S_C = gamma_C S0 + U^T diag(gamma_C/gamma) K."""
    x = gen.bf16_bits_to_f32(qkv[0]).astype(np.float64)
    Tn = x.shape[0]
    Q = x[:, : Hk * dk].reshape(Tn, Hk, dk)
    K = x[:, Hk * dk: 2 * Hk * dk].reshape(Tn, Hk, dk)
    V = x[:, 2 * Hk * dk:].reshape(Tn, Hv, dv)
    Q = Q / np.sqrt((Q * Q).sum(-1, keepdims=True) + 1e-6)
    K = K / np.sqrt((K * K).sum(-1, keepdims=True) + 1e-6)
    S = S0[0].astype(np.float64).copy()
    out = np.zeros((Tn, Hv, dv))
    for h in range(Hv):
        g = h * Hk // Hv
        for c0 in range(0, Tn, chunk):
            c1 = min(Tn, c0 + chunk)
            n = c1 - c0
            q, k, v = Q[c0:c1, g], K[c0:c1, g], V[c0:c1, h]
            a = alpha[0, c0:c1, h].astype(np.float64)
            b = beta[0, c0:c1, h].astype(np.float64)
            gam = np.cumprod(a)
            ratio = gam[:, None] / gam[None, :]
            L = np.tril(b[:, None] * ratio * (k @ k.T), -1)
            Tm = np.linalg.solve(np.eye(n) + L, np.eye(n))
            W = Tm @ ((b * gam)[:, None] * k)
            Ut = Tm @ (b[:, None] * v)
            U = Ut - W @ S[h].T
            M = np.tril(ratio)
            out[c0:c1, h] = gam[:, None] * (q @ S[h].T) + (M * (q @ k.T)) @ U
            S[h] = gam[-1] * S[h] + U.T @ ((gam[-1] / gam)[:, None] * k)
    return out, S


@pytest.mark.parametrize("Tn,chunk", [(64, 16), (50, 16), (37, 64)])
def test_sequential_oracle_matches_chunk_form(Tn, chunk):
    """The sequential definition and the published chunk-parallel form agree in fp64."""
    s = gen.Shape(1, 2, 4, 16, 16)
    d = gen.decode_inputs(30, s, Tn, tag="prefill")
    out, st = oracle.prefill(d["qkv"], d["alpha"], d["beta"], d["state"], 2, 4, 16, 16)
    out_c, st_c = _chunk_form(d["qkv"], d["alpha"], d["beta"], d["state"], 2, 4, 16, 16, chunk)
    np.testing.assert_allclose(out[0], out_c, rtol=0, atol=1e-12)
    np.testing.assert_allclose(st[0], st_c, rtol=0, atol=1e-12)


# ---------------------------------------------------------------------------
# KDA variant: a decay per key channel
# ---------------------------------------------------------------------------
def _kda_textbook(S, k, v, q, alpha, beta):
    dk = len(k)
    S1 = S @ np.diag(alpha) @ (np.eye(dk) - beta * np.outer(k, k)) + beta * np.outer(v, k)
    return S1, S1 @ q


@pytest.mark.parametrize("dk,dv", [(5, 3), (3, 7), (32, 32)])
def test_kda_row_form_vs_matrix_forms(dk, dv):
    n = gen.normal(11, f"kda{dk}{dv}", dv * dk + 2 * dk + dv)
    S = n[: dv * dk].reshape(dv, dk)
    k = n[dv * dk: dv * dk + dk]
    k = k / np.linalg.norm(k)
    q = n[dv * dk + dk: dv * dk + 2 * dk]
    v = n[dv * dk + 2 * dk:]
    a = 0.8 + 0.2 * gen.uniform(11, f"kdaa{dk}", dk)
    S_row, o_row = oracle.kda_token(S, k, v, q, a, 0.7)
    S_mat, o_mat = oracle.kda_token(S, k, v, q, a, 0.7, matrix_form=True)
    S_np, o_np = _kda_textbook(S, k, v, q, a, 0.7)
    np.testing.assert_allclose(S_row, S_np, rtol=0, atol=1e-13)
    np.testing.assert_allclose(S_mat, S_np, rtol=0, atol=1e-13)
    np.testing.assert_allclose(o_row, o_np, rtol=0, atol=1e-12)
    np.testing.assert_allclose(o_mat, o_np, rtol=0, atol=1e-12)


def test_kda_invariants():
    dk, dv = 16, 12
    n = gen.normal(12, "kdainv", dv * dk + 2 * dk + dv)
    S = n[: dv * dk].reshape(dv, dk)
    k = n[dv * dk: dv * dk + dk]
    k = k / np.linalg.norm(k)
    q = n[dv * dk + dk: dv * dk + 2 * dk]
    v = n[dv * dk + 2 * dk:]
    a = 0.8 + 0.2 * gen.uniform(12, "kdaa", dk)
    # beta = 0: every column decays by its own gate
    S1, o = oracle.kda_token(S, k, v, q, a, 0.0)
    np.testing.assert_allclose(S1, S * a[None, :], rtol=1e-15, atol=0)
    np.testing.assert_allclose(o, (S * a[None, :]) @ q, rtol=0, atol=1e-13)
    # a gate of zero on a channel wipes that column before the write
    a0 = a.copy()
    a0[3] = 0.0
    S1, _ = oracle.kda_token(S, k, v, q, a0, 0.5)
    S_np, _ = _kda_textbook(S, k, v, q, a0, 0.5)
    np.testing.assert_allclose(S1, S_np, rtol=0, atol=1e-13)
    # all gates 1, beta 1, unit k: the new state maps k to v
    S1, _ = oracle.kda_token(S, k, v, q, np.ones(dk), 1.0)
    np.testing.assert_allclose(S1 @ k, v, rtol=0, atol=1e-13)
    # the decay comes first, the delta step second: read at k, the new state
    # moves beta of the way from the decayed read to v; read at any x
    # orthogonal to k, it is the decayed state alone.  Together these fix the
    # whole map, so they also catch the decay applied after the projection.
    beta = 0.35
    S1, _ = oracle.kda_token(S, k, v, q, a, beta)
    np.testing.assert_allclose(S1 @ k, (1 - beta) * ((S * a[None, :]) @ k) + beta * v, rtol=0, atol=1e-13)
    for t in range(3):
        x = gen.normal(12, f"kdaperp{t}", dk)
        x = x - (x @ k) * k
        np.testing.assert_allclose(S1 @ x, (S * a[None, :]) @ x, rtol=0, atol=1e-13)


def test_kda_with_equal_gates_is_gdn():
    """The same decay on every channel reduces KDA to the scalar-gated rule."""
    s = gen.Shape(2, 2, 4, 16, 8)
    d = gen.decode_inputs(13, s, 5, tag="kdagdn")
    a_vec = np.repeat(d["alpha"][..., None], s.dk, axis=-1)
    out_g, st_g = oracle.decode(d["qkv"], d["alpha"], d["beta"], d["state"], s.Hk, s.Hv, s.dk, s.dv)
    out_k, st_k = oracle.kda_decode(d["qkv"], a_vec, d["beta"], d["state"], s.Hk, s.Hv, s.dk, s.dv)
    np.testing.assert_allclose(out_k, out_g, rtol=0, atol=1e-13)
    np.testing.assert_allclose(st_k, st_g, rtol=0, atol=1e-13)


def test_kda_decode_vs_textbook():
    s = gen.Shape(2, 1, 3, 8, 6)
    T = 4
    d = gen.kda_inputs(14, s, T)
    out, st = oracle.kda_decode(d["qkv"], d["alpha"], d["beta"], d["state"], s.Hk, s.Hv, s.dk, s.dv)
    qkv = gen.bf16_bits_to_f32(d["qkv"]).astype(np.float64)
    S = d["state"].astype(np.float64).copy()
    for b in range(s.B):
        for t in range(T):
            row = qkv[b, t]
            q = row[: s.dk]
            k = row[s.dk: 2 * s.dk]
            q = q / math.sqrt(q @ q + 1e-6)
            k = k / math.sqrt(k @ k + 1e-6)
            for h in range(s.Hv):
                v = row[2 * s.dk + h * s.dv: 2 * s.dk + (h + 1) * s.dv]
                S[b, h], o = _kda_textbook(S[b, h], k, v, q, d["alpha"][b, t, h].astype(np.float64),
                                           float(d["beta"][b, t, h]))
                np.testing.assert_allclose(out[b, t, h], o, rtol=0, atol=1e-12)
    np.testing.assert_allclose(st, S, rtol=0, atol=1e-12)


# ---------------------------------------------------------------------------
# state snapshot / restore
# ---------------------------------------------------------------------------
def test_fnv1a64_published_vectors():
    # test vectors of the FNV-1a 64-bit hash (Fowler, Noll, Vo)
    assert oracle.fnv1a64(b"") == 0xCBF29CE484222325
    assert oracle.fnv1a64(b"a") == 0xAF63DC4C8601EC8C
    assert oracle.fnv1a64(b"foobar") == 0x85944171F73967E8


def test_mix64_is_splitmix64_output():
    # SplitMix64 seeded with 0: output n is mix64(n * golden gamma); its first
    # outputs are published with the generator
    g = 0x9E3779B97F4A7C15
    assert oracle.mix64(g) == 0xE220A8397B1DCDAF
    assert oracle.mix64(2 * g % 2 ** 64) == 0x6E789E6AA1B965F4
    assert oracle.mix64(3 * g % 2 ** 64) == 0x06C45D188009454F
    # and the seeded generator module's own implementation agrees
    z = np.array([5, 2 ** 63 + 7, 0xDEADBEEF], np.uint64)
    assert [oracle.mix64(int(x)) for x in z] == [int(v) for v in gen._mix64(z)]


def test_snapshot_checksum_special_cases():
    g = 0x9E3779B97F4A7C15
    assert oracle.snapshot_checksum(b"") == 0
    # all-zero payloads: the terms are SplitMix64's published outputs from seed 0
    assert oracle.snapshot_checksum(bytes(8)) == 0xE220A8397B1DCDAF
    assert oracle.snapshot_checksum(bytes(16)) == (0xE220A8397B1DCDAF + 0x6E789E6AA1B965F4) % 2 ** 64
    # one word: mix64 of the little-endian word plus the increment
    one = bytes([0x08, 0x07, 0x06, 0x05, 0x04, 0x03, 0x02, 0x01])
    assert oracle.snapshot_checksum(one) == oracle.mix64(0x0102030405060708 + g)
    # two words: the second is keyed by index 2
    two = bytes([3] + [0] * 7 + [9] + [0] * 7)
    assert oracle.snapshot_checksum(two) == (oracle.mix64(3 + g) + oracle.mix64(9 + 2 * g)) % 2 ** 64
    # position matters: swapping two different words changes the sum
    assert oracle.snapshot_checksum(bytes([9] + [0] * 7 + [3] + [0] * 7)) != oracle.snapshot_checksum(two)
    # changing one word moves the sum by exactly that word's term
    p = gen.uniform(3, "ck", 64)
    raw = bytearray(np.asarray(p * 2 ** 32, np.uint64).astype(np.uint32).tobytes())
    base = oracle.snapshot_checksum(raw)
    d_old = int.from_bytes(raw[40:48], "little")
    raw[40:48] = (d_old ^ 0x10).to_bytes(8, "little")
    delta = oracle.mix64(((d_old ^ 0x10) + 6 * g) % 2 ** 64) - oracle.mix64((d_old + 6 * g) % 2 ** 64)
    assert oracle.snapshot_checksum(raw) == (base + delta) % 2 ** 64


def _snap_arrays(seed, L, B, s):
    st = gen.normal(seed, "snap.state", L * B * s.Hv * s.dv * s.dk).astype(np.float32).reshape(L, B, s.Hv, s.dv, s.dk)
    tl = gen.normal_bf16(seed, "snap.tail", L * B * 4 * s.C).reshape(L, B, 4, s.C)
    return st, tl


def test_snapshot_format_and_round_trip():
    s = gen.Shape(1, 2, 4, 32, 64)
    L, B, seq = 3, 4, 2
    st, tl = _snap_arrays(5, L, B, s)
    blob = oracle.snapshot_save(st, tl, seq, s.Hk, s.Hv, s.dk, s.dv)
    assert blob.size == 64 + L * (s.Hv * s.dv * s.dk * 4 + 4 * s.C * 2)
    h = blob[:64].tobytes()
    assert h[:8] == b"GDNSNAP1"
    assert [int.from_bytes(h[o:o + 4], "little") for o in range(8, 32, 4)] == [1, L, s.Hk, s.Hv, s.dk, s.dv]
    text = f"gdn-snapshot/1;layers={L};state:f32[{s.Hv},{s.dv},{s.dk}];tail:bf16[4,{s.C}]".encode()
    assert int.from_bytes(h[32:40], "little") == oracle.fnv1a64(text)
    assert int.from_bytes(h[40:48], "little") == blob.size - 64
    assert int.from_bytes(h[56:64], "little") == 0
    # the payload is each layer's raw state bytes then raw tail bytes, in layer order
    want = b"".join(st[l, seq].tobytes() + tl[l, seq].tobytes() for l in range(L))
    assert blob[64:].tobytes() == want
    assert int.from_bytes(h[48:56], "little") == oracle.snapshot_checksum(want)
    # restore into other arrays: only sequence seq changes, bit for bit
    st0, tl0 = _snap_arrays(6, L, B, s)
    rc, st1, tl1 = oracle.snapshot_restore(blob, st0, tl0, seq, s.Hk, s.Hv, s.dk, s.dv)
    assert rc == 0
    assert st1[:, seq].tobytes() == st[:, seq].tobytes() and np.array_equal(tl1[:, seq], tl[:, seq])
    others = [b for b in range(B) if b != seq]
    assert np.array_equal(st1[:, others], st0[:, others]) and np.array_equal(tl1[:, others], tl0[:, others])


def test_snapshot_restore_refusals():
    s = gen.Shape(1, 2, 4, 32, 32)
    L, B = 2, 2
    st, tl = _snap_arrays(7, L, B, s)
    blob = oracle.snapshot_save(st, tl, 1, s.Hk, s.Hv, s.dk, s.dv)
    st0, tl0 = np.zeros_like(st), np.zeros_like(tl)
    bad = blob.copy()
    bad[64 + 1000] ^= 1                                  # one payload bit
    rc, st1, tl1 = oracle.snapshot_restore(bad, st0, tl0, 1, s.Hk, s.Hv, s.dk, s.dv)
    assert rc == 2 and not st1.any() and not tl1.any()
    bad = blob.copy()
    bad[0] ^= 1                                          # magic
    assert oracle.snapshot_restore(bad, st0, tl0, 1, s.Hk, s.Hv, s.dk, s.dv)[0] == 1
    # another model's shape: the signature and shape fields refuse it
    assert oracle.snapshot_restore(blob, np.zeros((L, B, 4, 64, 16), np.float32),
                                   np.zeros((L, B, 4, 2 * 2 * 16 + 4 * 64), np.uint16), 1, 2, 4, 16, 64)[0] == 1
    assert oracle.snapshot_signature(2, 2, 4, 32, 32) != oracle.snapshot_signature(3, 2, 4, 32, 32)
    assert oracle.snapshot_signature(2, 2, 4, 32, 32) != oracle.snapshot_signature(2, 1, 4, 32, 32)


# ---------------------------------------------------------------------------
# gate front end and gated-norm output
# ---------------------------------------------------------------------------
def test_softplus_and_sigmoid_closed_forms():
    assert oracle.softplus(0.0) == pytest.approx(math.log(2.0), rel=0, abs=1e-16)
    for x in (-40.0, -3.5, -0.25, 0.7, 5.0, 40.0):
        # softplus(x) - softplus(-x) = x; sigmoid(x) + sigmoid(-x) = 1
        assert oracle.softplus(x) - oracle.softplus(-x) == pytest.approx(x, rel=0, abs=1e-13)
        assert oracle.sigmoid(x) + oracle.sigmoid(-x) == pytest.approx(1.0, rel=0, abs=1e-15)
        # d/dx softplus = sigmoid (central difference)
        h = 1e-5
        assert (oracle.softplus(x + h) - oracle.softplus(x - h)) / (2 * h) == pytest.approx(oracle.sigmoid(x),
                                                                                            abs=1e-9)
    assert oracle.softplus(-40.0) == pytest.approx(math.exp(-40.0), rel=1e-12)
    assert oracle.sigmoid(0.0) == 0.5


def test_gates_special_values_and_power_form():
    Hv = 4
    bf = gen.f32_to_bf16_bits
    a = bf(np.array([[0.0, 0.0, 1.5, -2.0]], np.float32))
    b = bf(np.array([[0.0, 2.0, -1.0, 0.5]], np.float32))
    A_log = np.array([0.0, math.log(2.0), 0.3, 1.7], np.float32)
    dt_bias = np.array([0.0, 0.0, -4.0, 0.25], np.float32)
    al, be = oracle.gates_from_projections(a, b, A_log, dt_bias)
    assert al[0, 0] == pytest.approx(0.5, abs=1e-15)        # exp(-1 * ln 2)
    # A_log = ln 2 rounded to fp32: alpha = 2^-(e^A_log), about 1/4
    assert al[0, 1] == pytest.approx(2.0 ** -math.exp(float(A_log[1])), rel=1e-15)
    assert be[0, 0] == 0.5
    # alpha = (1 + e^(a + dt_bias)) ^ (-e^A_log); beta = 1 / (1 + e^-b)
    av = gen.bf16_bits_to_f32(a).astype(np.float64)[0]
    bv = gen.bf16_bits_to_f32(b).astype(np.float64)[0]
    for h in range(Hv):
        x = av[h] + float(dt_bias[h])
        assert al[0, h] == pytest.approx((1.0 + math.exp(x)) ** (-math.exp(float(A_log[h]))), rel=1e-13)
        assert be[0, h] == pytest.approx(1.0 / (1.0 + math.exp(-bv[h])), rel=1e-15)


def test_gated_rmsnorm_invariants():
    dv = 16
    o = gen.normal(21, "rms.o", dv)
    z = gen.normal_bf16(21, "rms.z", (dv,))
    w = (1.0 + 0.1 * gen.normal(21, "rms.w", dv)).astype(np.float32)
    zf = gen.bf16_bits_to_f32(z).astype(np.float64)
    g = w.astype(np.float64) * zf / (1.0 + np.exp(-zf))            # w * SiLU(z)
    y = oracle.gated_rmsnorm(o, z, w, eps=0.0)
    # with eps = 0: y / (w SiLU(z)) has unit root-mean-square and o's direction
    r = y / g
    assert np.sqrt(np.mean(r ** 2)) == pytest.approx(1.0, abs=1e-13)
    np.testing.assert_allclose(r * np.linalg.norm(o) / math.sqrt(dv), o, rtol=1e-12, atol=0)
    # scale invariance, and eps acting as an additive floor on the mean square
    np.testing.assert_allclose(oracle.gated_rmsnorm(7.5 * o, z, w, eps=0.0), y, rtol=1e-13, atol=0)
    c = np.full(dv, 0.01)
    y_c = oracle.gated_rmsnorm(c, z, w, eps=1e-4)
    np.testing.assert_allclose(y_c, 0.01 / math.sqrt(1e-4 + 1e-4) * g, rtol=1e-13, atol=0)
    # SiLU(0) = 0
    assert np.all(oracle.gated_rmsnorm(o, np.zeros(dv, np.uint16), w) == 0.0)


def test_layer_decode_is_conv_gates_decode_norm():
    """The composed oracle equals its parts: the pinned conv, the pinned decode
    (fed the gates rounded to fp32, hence the 1e-6 slack) and the norm."""
    s = gen.Shape(2, 2, 4, 32, 32)
    T = 3
    d = gen.layer_inputs(22, s, T)
    o, y, st, tl = oracle.layer_decode(d["x"], d["w"], d["tail"], d["a"], d["b"], d["A_log"], d["dt_bias"], d["z"],
                                       d["norm_w"], d["state"], s.Hk, s.Hv, s.dk, s.dv)
    yc, tail_ref = oracle.conv_linear(d["x"], d["w"], d["tail"])
    assert np.array_equal(tl, tail_ref)
    al, be = oracle.gates_from_projections(d["a"], d["b"], d["A_log"], d["dt_bias"])
    o_ref, st_ref = oracle.decode(oracle.f64_to_bf16(yc), al.astype(np.float32), be.astype(np.float32), d["state"],
                                  s.Hk, s.Hv, s.dk, s.dv)
    np.testing.assert_allclose(o, o_ref, rtol=0, atol=1e-6)
    np.testing.assert_allclose(st, st_ref, rtol=0, atol=1e-6)
    for b_ in range(s.B):
        for t in range(T):
            for h in range(s.Hv):
                np.testing.assert_array_equal(y[b_, t, h], oracle.gated_rmsnorm(o[b_, t, h], d["z"][b_, t, h],
                                                                                d["norm_w"]))
    # the gates the recipe draws decay (some heads strongly: A up to 16, dt up to 0.1)
    assert 0.0 < al.min() and al.max() < 1.0


def test_parallel_key_head_oracle_equals_serial():
    """The test helper that runs the oracle per key head on all cores gives the
    serial oracle's results bit for bit (key heads are independent problems)."""
    from gdn_testutil import oracle_decode_parallel
    s = gen.Shape(2, 3, 6, 8, 8)
    d = gen.decode_inputs(24, s, 5)
    out, st = oracle.decode(d["qkv"], d["alpha"], d["beta"], d["state"], s.Hk, s.Hv, s.dk, s.dv)
    out_p, st_p = oracle_decode_parallel(d["qkv"], d["alpha"], d["beta"], d["state"], s)
    assert np.array_equal(out, out_p) and np.array_equal(st, st_p)
    out_k, _ = oracle_decode_parallel(d["qkv"], d["alpha"], d["beta"], d["state"], s, keys=[1])
    assert np.array_equal(out_k[:, :, 2:4], out[:, :, 2:4]) and np.isnan(out_k[:, :, :2]).all()
