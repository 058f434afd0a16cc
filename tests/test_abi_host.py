"""C-ABI checks that need no GPU: the library builds and loads, exports every
symbol include/gdn.h declares, validates its arguments before touching the
device, and its host-side tree bookkeeping matches the oracle bit for bit.

Every call here is made with arguments that fail validation (or with host-only
entry points), so no kernel is ever launched from these tests."""
import ctypes
import itertools
import os
import re

import numpy as np
import pytest

import oracle
from hybrid_linear_attention_conv_gb300 import build as gbuild
from hybrid_linear_attention_conv_gb300 import gdn
from hybrid_linear_attention_conv_gb300 import inputs as gen

ROOT = os.path.dirname(os.path.dirname(os.path.abspath(__file__)))


@pytest.fixture(scope="module")
def lib():
    gbuild.build()
    return gdn.load()


def _header_symbols():
    txt = open(os.path.join(ROOT, "include", "gdn.h")).read()
    txt = re.sub(r"/\*.*?\*/", "", txt, flags=re.S)
    return sorted(set(re.findall(r"\b(gdn_[a-z_0-9]+)\s*\(", txt)))


def test_exports_every_declared_symbol(lib):
    syms = _header_symbols()
    assert sorted(gdn.EXPORTS) == syms
    for s in syms:
        assert hasattr(lib, s), s
    # the symbols are real dynamic exports of the .so (nm -D)
    import subprocess
    out = subprocess.run(["nm", "-D", "--defined-only", gdn.LIB_PATH], capture_output=True,
                         text=True, check=True).stdout
    exported = set(re.findall(r" T (gdn_\w+)", out))
    assert set(syms) <= exported


def test_abi_version(lib):
    assert gdn.abi_version() == 1


def test_state_bytes(lib):
    assert gdn.state_bytes(1, 16, 48, 128, 128) == 48 * 128 * 128 * 4 == 3145728
    assert gdn.state_bytes(64, 16, 48, 128, 128) == 64 * 3145728
    assert gdn.state_bytes(1, 16, 48, 100, 128) == 0  # unsupported head size


def _sh(B=1, Hk=16, Hv=48, dk=128, dv=128):
    return gdn.gdn_shape(B, Hk, Hv, dk, dv)


FAKE = 0x10000  # aligned, never dereferenced: every call below fails validation first


@pytest.mark.parametrize("fn", ["gdn_decode_step", "gdn_kda_decode_step"])
def test_decode_validation(lib, fn):
    P = ctypes.c_void_p
    step = getattr(lib, fn)
    cases = [
        (_sh(dk=100), 1, FAKE, -2),
        (_sh(dv=48), 1, FAKE, -2),
        (_sh(Hk=5), 1, FAKE, -2),           # 48 % 5 != 0
        (_sh(B=-1), 1, FAKE, -2),
        (_sh(), -3, FAKE, -1),
        (_sh(), 1, FAKE + 2, -6),           # misaligned qkv
    ]
    for sh, T, qkv, want in cases:
        rc = step(ctypes.byref(sh), T, P(qkv), P(FAKE), P(FAKE), P(FAKE), P(FAKE),
                                 1.0, 1, None)
        assert rc == want, (sh.dk, sh.dv, sh.Hk, T, gdn.last_error())
        assert gdn.last_error()
    # null state
    rc = step(ctypes.byref(_sh()), 1, P(FAKE), P(FAKE), P(FAKE), None, None, 1.0, 1, None)
    assert rc == -1
    # unknown flag
    rc = step(ctypes.byref(_sh()), 1, P(FAKE), P(FAKE), P(FAKE), P(FAKE), None, 1.0,
                             0x80, None)
    assert rc == -1
    # the prefill-only flag is unknown to the other entry points
    rc = step(ctypes.byref(_sh()), 1, P(FAKE), P(FAKE), P(FAKE), P(FAKE), None, 1.0,
              gdn.GDN_NORMALIZE_QK | gdn.GDN_PREFILL_TWO_LAUNCH, None)
    assert rc == -1


def test_conv_validation(lib):
    P = ctypes.c_void_p
    assert lib.gdn_conv_step(1, 1, 100, None, P(FAKE), P(FAKE), P(FAKE), P(FAKE), 0, None) == -2
    assert lib.gdn_conv_step(1, -1, 128, None, P(FAKE), P(FAKE), P(FAKE), P(FAKE), 0, None) == -1
    assert lib.gdn_conv_step(1, 1, 128, None, P(FAKE), P(FAKE + 8), P(FAKE), P(FAKE), 0, None) == -6
    bad = np.array([-1, 0, 5], np.int32)
    assert lib.gdn_conv_step(1, 3, 128, bad.ctypes.data_as(P), P(FAKE), P(FAKE), P(FAKE), P(FAKE), 0,
                             None) == -3


def _tree_call(lib, parents, sh=None, N=None):
    P = ctypes.c_void_p
    par = np.ascontiguousarray(parents, np.int32)
    sh = sh or _sh()
    return lib.gdn_tree_verify(ctypes.byref(sh), len(par) if N is None else N, par.ctypes.data_as(P),
                               P(FAKE), P(FAKE), P(FAKE), P(FAKE), P(FAKE), 1.0, 1, None)


def test_tree_validation(lib):
    assert _tree_call(lib, [0, 0]) == -3                  # root must be -1
    assert _tree_call(lib, [-1, 1]) == -3                 # parent must precede
    assert _tree_call(lib, [-1, 0, -1]) == -3             # a second root
    assert _tree_call(lib, [-1] + [0] * 64) == -3         # N = 65 > 64
    assert _tree_call(lib, [-1], N=0) == -3
    assert _tree_call(lib, [-1, 0], sh=_sh(B=2)) == -2    # one sequence only


def _nested_branch_tree(levels):
    """A spine where every spine node also has a leaf child: `levels` nested
    branching nodes on the deepest root path."""
    parents = [-1]
    spine = 0
    for _ in range(levels):
        parents.append(spine)          # next spine node (first child)
        nxt = len(parents) - 1
        parents.append(spine)          # a leaf sibling (second child)
        spine = nxt
    return np.array(parents, np.int32)


def test_tree_depth_exceeded(lib):
    # 9 nested branching nodes need 9 parked states: refused before any launch
    parents = _nested_branch_tree(9)
    assert _tree_call(lib, parents) == -5
    assert "branch" in gdn.last_error()


def test_commit_validation(lib):
    P = ctypes.c_void_p
    parents = np.array([-1, 0, 0, 1, 3], np.int32)

    def call(path, sh=None):
        pa = np.ascontiguousarray(path, np.int32)
        return lib.gdn_commit_path(ctypes.byref(sh or _sh()), len(parents), parents.ctypes.data_as(P),
                                   pa.ctypes.data_as(P) if pa.size else None, len(pa), P(FAKE), P(FAKE),
                                   P(FAKE), None, P(FAKE + 4), None, 1, None)

    assert call([1, 3]) == -4          # does not start at the root
    assert call([0, 2, 3]) == -4       # 3 is not a child of 2
    assert call([0, 7]) == -4          # out of range
    assert call([0, 1, 3], sh=_sh(dk=96)) == -2
    assert call([0, 1, 3]) == -6       # valid path, misaligned state pointer


def test_root_path_matches_oracle_brute_force(lib):
    """Bit-exact bookkeeping: every node of every tree with up to 7 nodes."""
    for N in range(1, 8):
        for tail in itertools.product(*[range(i) for i in range(1, N)]):
            parents = np.array((-1,) + tail, np.int32)
            for n in range(N):
                assert np.array_equal(gdn.tree_root_path(parents, n), oracle.root_path(parents, n))
    for seed in range(10):
        parents = gen.random_tree(seed, 64, 20)
        for n in range(64):
            assert np.array_equal(gdn.tree_root_path(parents, n), oracle.root_path(parents, n))


def test_root_path_rejects(lib):
    with pytest.raises(gdn.GdnError):
        gdn.tree_root_path(np.array([-1, 2, 0], np.int32), 1)
    with pytest.raises(gdn.GdnError):
        gdn.tree_root_path(np.array([-1, 0], np.int32), 5)


@pytest.mark.parametrize("fn", ["gdn_conv_decode_step", "gdn_kda_conv_decode_step"])
def test_conv_decode_validation(lib, fn):
    P = ctypes.c_void_p
    step = getattr(lib, fn)
    sh = _sh(B=2)
    args = lambda T, ti, to: (ctypes.byref(sh), T, P(FAKE), P(FAKE), P(ti), P(to), P(FAKE), P(FAKE), P(FAKE), None,
                              1.0, 1, None)
    assert step(*args(17, FAKE, FAKE)) == -2   # more than 16 tokens
    assert step(*args(1, FAKE, FAKE + 16)) == -1  # overlapping tails
    assert step(*args(1, FAKE, FAKE + 8)) == -6   # misaligned tail_out
    big = gdn.gdn_shape(1, 1, 16, 128, 128)  # 2*128 + 16*128 channels x 16 tokens > 48 KB staging
    assert step(ctypes.byref(big), 16, P(FAKE), P(FAKE), P(FAKE), P(FAKE), P(FAKE), P(FAKE),
                                     P(FAKE), None, 1.0, 1, None) == -2


def test_tree_verify_batched_validation(lib):
    P = ctypes.c_void_p

    def call(B, N, counts, parents):
        c = np.ascontiguousarray(counts, np.int32)
        pa = np.ascontiguousarray(parents, np.int32)
        sh = _sh(B=B)
        return lib.gdn_tree_verify_batched(ctypes.byref(sh), N, c.ctypes.data_as(P), pa.ctypes.data_as(P),
                                           P(FAKE), P(FAKE), P(FAKE), P(FAKE), P(FAKE), 1.0, 1, None)

    ok_tree = [-1, 0, 0, 1]
    assert call(33, 4, [4] * 33, ok_tree * 33) == -2            # more than 32 trees
    assert call(2, 4, [4, 0], ok_tree * 2) == -3                 # an empty tree
    assert call(2, 4, [4, 5], ok_tree * 2) == -3                 # more nodes than the capacity
    assert call(3, 4, [4, 4, 3], ok_tree + ok_tree + [-1, 2, 0, 9]) == -3  # tree 2: parent after child
    assert "tree 2" in gdn.last_error()
    assert call(2, 65, [1, 1], [-1] * 130) == -3                 # capacity above 64


# ---------------------------------------------------------------------------
# snapshot / restore (host side: sizes, signature, refusals)
# ---------------------------------------------------------------------------
@pytest.mark.parametrize("L,shape", [(1, (2, 4, 32, 32)), (48, (16, 48, 128, 128)), (3, (2, 4, 32, 64))])
def test_snapshot_sizes_and_signature_match_oracle(lib, L, shape):
    Hk, Hv, dk, dv = shape
    assert gdn.snapshot_bytes(L, Hk, Hv, dk, dv) == oracle.snapshot_bytes(L, Hk, Hv, dk, dv)
    assert gdn.snapshot_signature(L, Hk, Hv, dk, dv) == oracle.snapshot_signature(L, Hk, Hv, dk, dv)


def test_snapshot_validation(lib):
    P = ctypes.c_void_p
    sh = _sh(B=4)
    need = gdn.snapshot_bytes(2, sh.Hk, sh.Hv, sh.dk, sh.dv)
    s_el = 4 * sh.Hv * sh.dv * sh.dk
    t_el = 4 * 4 * (2 * sh.Hk * sh.dk + sh.Hv * sh.dv)

    def save(L=2, seq=1, ss=s_el, ts=t_el, dst=FAKE, n=need, ws=FAKE, wsn=256, shape=sh):
        return lib.gdn_snapshot_save(ctypes.byref(shape), L, seq, P(FAKE), ss, P(FAKE), ts, P(dst), n, P(ws), wsn,
                                     None)

    def restore(L=2, seq=1, ss=s_el, ts=t_el, src=FAKE, n=need, ws=FAKE, wsn=256):
        return lib.gdn_snapshot_restore(ctypes.byref(sh), L, seq, P(src), n, P(FAKE), ss, P(FAKE), ts, P(ws), wsn,
                                        None)

    assert save(L=0) == -1
    assert save(seq=4) == -1 and "seq" in gdn.last_error()
    assert save(seq=-1) == -1
    assert save(ss=s_el - 4) == -1                      # layers would overlap
    assert save(ts=t_el + 4) == -6                      # 8 bytes: not a multiple of 16
    assert save(n=need - 1) == -1 and "needs" in gdn.last_error()
    assert save(dst=FAKE + 8) == -6
    assert save(ws=0) == -9
    assert save(ws=FAKE + 16) == -6
    assert save(wsn=255) == -9
    assert save(shape=_sh(dk=100)) == -2
    assert restore(n=need - 16) == -1
    assert restore(seq=9) == -1
    assert gdn.snapshot_bytes(1, 2, 4, 100, 32) == 0    # bad shape


def test_layer_step_and_gates_validation(lib):
    P = ctypes.c_void_p
    sh = _sh(B=2)

    def layer(T=1, flags=1, eps=1e-6, a=FAKE, y=FAKE, shape=sh, tail_out=FAKE):
        return lib.gdn_layer_decode_step(ctypes.byref(shape), T, P(FAKE), P(FAKE), P(FAKE), P(tail_out), P(a),
                                         P(FAKE), P(FAKE), P(FAKE), P(FAKE), P(FAKE), eps, P(FAKE), None, P(y), 1.0,
                                         flags, None)

    assert layer(flags=1 | 2) == -1 and "GDN_OUT_BF16" in gdn.last_error()
    assert layer(eps=-1.0) == -1
    assert layer(eps=float("nan")) == -1
    assert layer(T=-1) == -1
    assert layer(T=17) == -2                          # the fused step's token limit
    assert layer(a=FAKE + 2) == -6
    assert layer(y=0) == -1
    assert layer(tail_out=FAKE + 16) == -1            # overlapping tails
    assert layer(shape=_sh(dv=48)) == -2
    assert layer(T=0) == 0                            # no-op
    assert lib.gdn_gates(-1, 4, P(FAKE), P(FAKE), P(FAKE), P(FAKE), P(FAKE), P(FAKE), None) == -1
    assert lib.gdn_gates(4, 0, P(FAKE), P(FAKE), P(FAKE), P(FAKE), P(FAKE), P(FAKE), None) == -1
    assert lib.gdn_gates(4, 4, P(FAKE), P(FAKE), P(FAKE), P(FAKE), P(FAKE + 4), P(FAKE), None) == -6
    assert lib.gdn_gates(0, 4, None, None, None, None, None, None, None) == 0


def test_prefill_workspace_holds_the_prepass_records(lib):
    P = ctypes.c_void_p
    sh = gdn.gdn_shape(1, 16, 48, 128, 128)
    # the status word, one 50,432-byte record per (chunk of 64, value head), then
    # one int32 ready flag per (chunk, value head), padded to 16 bytes
    assert gdn.prefill_workspace_bytes(8192, 16, 48, 128, 128) == 256 + 128 * 48 * 50432 + 128 * 48 * 4
    assert gdn.prefill_workspace_bytes(65, 16, 48, 128, 128) == 256 + 2 * 48 * 50432 + 2 * 48 * 4
    assert gdn.prefill_workspace_bytes(65, 1, 3, 128, 128) == 256 + 2 * 3 * 50432 + 32
    assert gdn.prefill_workspace_bytes(100, 2, 4, 32, 32) == 256     # narrow heads: no records
    rc = lib.gdn_chunk_prefill(ctypes.byref(sh), 64, 64, P(FAKE), P(FAKE), P(FAKE), P(FAKE), P(FAKE), P(FAKE * 256),
                               256, 1.0, 1, None)
    assert rc == -9 and "needed" in gdn.last_error()


def test_fp32_activation_flag_validation(lib):
    """GDN_IN_F32 is accepted by the conv and the plain decode, refused by the
    other entry points; the conv refuses the decode-only flags."""
    P = ctypes.c_void_p
    F32 = gdn.GDN_IN_F32
    rc = lib.gdn_kda_decode_step(ctypes.byref(_sh()), 1, P(FAKE), P(FAKE), P(FAKE), P(FAKE), None, 1.0, 1 | F32, None)
    assert rc == -1 and "flag" in gdn.last_error()
    rc = lib.gdn_conv_decode_step(ctypes.byref(_sh()), 1, P(FAKE), P(FAKE), P(FAKE), P(FAKE), P(FAKE), P(FAKE),
                                  P(FAKE), None, 1.0, 1 | F32, None)
    assert rc == -1
    rc = _tree_call_flags(lib, 1 | F32)
    assert rc == -1
    # the flag passes the decode's flag check: the (misaligned) qkv is what fails
    rc = lib.gdn_decode_step(ctypes.byref(_sh()), 1, P(FAKE + 4), P(FAKE), P(FAKE), P(FAKE), None, 1.0, 1 | F32,
                             None)
    assert rc == -6
    assert lib.gdn_conv_step(1, 1, 128, None, P(FAKE), P(FAKE + 8), P(FAKE), P(FAKE), F32, None) == -6
    assert lib.gdn_conv_step(1, 1, 128, None, P(FAKE), P(FAKE), P(FAKE), P(FAKE), gdn.GDN_NORMALIZE_QK, None) == -1


def _tree_call_flags(lib, flags):
    P = ctypes.c_void_p
    par = np.array([-1, 0], np.int32)
    return lib.gdn_tree_verify(ctypes.byref(_sh()), 2, par.ctypes.data_as(P), P(FAKE), P(FAKE), P(FAKE), P(FAKE),
                               P(FAKE), 1.0, flags, None)


def test_wait_limit_setter_and_status_validation(lib):
    """The wait-limit setter returns the previous limit and clamps at 10 s; the
    status readers refuse a missing or misaligned workspace before touching
    the device."""
    prev = gdn.set_wait_limit_ns(12345)
    try:
        assert prev == 200_000_000
        assert gdn.set_wait_limit_ns(10**12) == 12345
        assert gdn.set_wait_limit_ns(0) == 10_000_000_000
    finally:
        gdn.set_wait_limit_ns(prev)
    word = ctypes.c_int32(7)
    assert lib.gdn_prefill_status(None, None, ctypes.byref(word)) == -1
    assert lib.gdn_prefill_status(ctypes.c_void_p(FAKE + 16), None, ctypes.byref(word)) == -6
    assert word.value == 7


def test_commit_batched_validation(lib):
    """Every tree and path is checked before anything is enqueued; a call in
    which no sequence accepted anything is a no-op."""
    P = ctypes.c_void_p
    N = 5
    parents = np.array([[-1, 0, 0, 1, 3], [-1, 0, 1, -7, -7]], np.int32)
    counts = np.array([5, 3], np.int32)

    def call(paths, lengths, sh=None, flags=1, cnt=counts, par=parents):
        pa = np.ascontiguousarray(paths, np.int32)
        ln = np.ascontiguousarray(lengths, np.int32)
        return lib.gdn_commit_path_batched(ctypes.byref(sh or _sh(B=2)), N, cnt.ctypes.data_as(P),
                                           par.ctypes.data_as(P), pa.ctypes.data_as(P), ln.ctypes.data_as(P),
                                           P(FAKE), P(FAKE), P(FAKE), None, P(FAKE), None, flags, None)

    ok = [[0, 1, 3, 4, 0], [0, 1, 2, 0, 0]]
    assert call(ok, [0, 0]) == 0                       # nothing accepted: a no-op
    assert call([[1, 3, 0, 0, 0], [0, 0, 0, 0, 0]], [2, 0]) == -4   # does not start at the root
    assert call([[0, 1, 3, 0, 0], [0, 2, 0, 0, 0]], [3, 2]) == -4   # 2 is not a child of 0 in tree 1
    assert call(ok, [4, 4]) == -4                      # tree 1 has 3 nodes
    assert call(ok, [4, 3], sh=_sh(B=0)) == -2
    assert call(ok, [4, 3], sh=_sh(B=33)) == -2
    assert call(ok, [4, 3], flags=1 | gdn.GDN_OUT_BF16) == -1
    assert call(ok, [4, 3], cnt=np.array([5, 6], np.int32)) == -3
    bad = parents.copy()
    bad[1, 1] = 2
    assert call(ok, [4, 3], par=bad) == -3
    assert "tree 1" in gdn.last_error()


def test_conv_fused_round_validation(lib):
    """The verify and commit with the conv fused in refuse what the unfused
    calls refuse, plus missing conv inputs and overlapping tails.  Every call
    fails validation (the last argument checked is a misaligned state), so
    nothing is launched."""
    P = ctypes.c_void_p
    parents = np.array([-1, 0, 0, 1, 3], np.int32)
    far = FAKE + (1 << 20)  # a second buffer, clear of the first tail

    def verify(x=FAKE, w=FAKE, tail=FAKE, sh=None, par=parents, flags=1, state=FAKE + 4):
        return lib.gdn_conv_tree_verify(ctypes.byref(sh or _sh()), len(par), par.ctypes.data_as(P), P(x), P(w),
                                        P(tail), P(FAKE), P(FAKE), P(state), P(FAKE), 1.0, flags, None)

    assert verify(x=None) == -1
    assert verify(w=None) == -1
    assert verify(tail=None) == -1
    assert verify(x=FAKE + 2) == -6
    assert verify(par=np.array([0, 0], np.int32)) == -3
    assert verify(sh=_sh(B=2)) == -2
    assert verify(flags=0x40) == -1
    assert verify() == -6 and "state" in gdn.last_error()

    def commit(path=(0, 1, 3), w=FAKE, tin=FAKE, tout=far, sh=None, flags=1, state=FAKE + 4):
        pa = np.ascontiguousarray(path, np.int32)
        return lib.gdn_conv_commit_path(ctypes.byref(sh or _sh()), len(parents), parents.ctypes.data_as(P),
                                        pa.ctypes.data_as(P) if pa.size else None, len(pa), P(FAKE), P(w), P(tin),
                                        P(tout), P(FAKE), P(FAKE), P(state), flags, None)

    assert commit(w=None) == -1
    assert commit(tin=None) == -1
    assert commit(tout=None) == -1
    assert commit(tout=FAKE + 16) == -1 and "overlap" in gdn.last_error()
    assert commit(tout=FAKE + 8) == -6
    assert commit(path=(1, 3)) == -4
    assert commit(flags=1 | gdn.GDN_OUT_BF16) == -1
    assert commit(sh=_sh(B=2)) == -2
    assert commit() == -6 and "state" in gdn.last_error()
    assert commit(path=()) == -6  # nothing accepted still validates everything (the tail is still copied)

    N = 5
    par2 = np.array([[-1, 0, 0, 1, 3], [-1, 0, 1, -7, -7]], np.int32)
    counts = np.array([5, 3], np.int32)

    def vbatch(x=FAKE, sh=None, par=par2, state=FAKE + 4):
        return lib.gdn_conv_tree_verify_batched(ctypes.byref(sh or _sh(B=2)), N, counts.ctypes.data_as(P),
                                                par.ctypes.data_as(P), P(x), P(FAKE), P(FAKE), P(FAKE), P(FAKE),
                                                P(state), P(FAKE), 1.0, 1, None)

    assert vbatch(x=None) == -1
    assert vbatch(sh=_sh(B=33)) == -2
    bad = par2.copy()
    bad[1, 2] = 2
    assert vbatch(par=bad, state=FAKE) == -3 and "tree 1" in gdn.last_error()  # pointers pass, the tree does not
    assert vbatch() == -6

    def cbatch(lengths=(3, 2), tout=far, w=FAKE, state=FAKE + 4):
        paths = np.array([[0, 1, 3, 0, 0], [0, 1, 2, 0, 0]], np.int32)
        ln = np.ascontiguousarray(lengths, np.int32)
        return lib.gdn_conv_commit_path_batched(ctypes.byref(_sh(B=2)), N, counts.ctypes.data_as(P),
                                                par2.ctypes.data_as(P), paths.ctypes.data_as(P),
                                                ln.ctypes.data_as(P), P(FAKE), P(w), P(FAKE), P(tout), P(FAKE),
                                                P(FAKE), P(state), 1, None)

    assert cbatch(w=None) == -1
    assert cbatch(tout=FAKE + 2 * 4 * 10240 * 2 - 16) == -1  # overlaps the last sequence's tail_in
    assert cbatch(lengths=(3, 4)) == -4
    assert cbatch() == -6
    assert cbatch(lengths=(0, 0)) == -6  # no sequence accepted anything: still validated


def test_kda_round_validation(lib):
    """The KDA tree verify and commit validate like the plain ones; nothing is launched."""
    P = ctypes.c_void_p
    parents = np.array([-1, 0, 0, 1, 3], np.int32)

    def verify(alpha=FAKE, sh=None, par=parents, state=FAKE + 4):
        return lib.gdn_kda_tree_verify(ctypes.byref(sh or _sh()), len(par), par.ctypes.data_as(P), P(FAKE),
                                       P(alpha), P(FAKE), P(state), P(FAKE), 1.0, 1, None)

    assert verify(alpha=None) == -1
    assert verify(alpha=FAKE + 4) == -6
    assert verify(sh=_sh(B=2)) == -2
    assert verify(par=np.array([-1, 1], np.int32)) == -3
    assert verify() == -6 and "state" in gdn.last_error()

    par2 = np.array([[-1, 0, 0, 1, 3], [-1, 0, 1, -7, -7]], np.int32)
    counts = np.array([5, 3], np.int32)

    def vbatch(sh=None, alpha=FAKE, state=FAKE + 4, par=par2):
        return lib.gdn_kda_tree_verify_batched(ctypes.byref(sh or _sh(B=2)), 5, counts.ctypes.data_as(P),
                                               par.ctypes.data_as(P), P(FAKE), P(alpha), P(FAKE), P(state), P(FAKE),
                                               1.0, 1, None)

    assert vbatch(sh=_sh(B=33)) == -2
    assert vbatch(alpha=None) == -1
    bad = par2.copy()
    bad[1, 2] = 2
    assert vbatch(par=bad, state=FAKE) == -3
    assert vbatch() == -6

    def commit(path=(0, 1, 3), state=FAKE + 4, flags=1):
        pa = np.ascontiguousarray(path, np.int32)
        return lib.gdn_kda_commit_path(ctypes.byref(_sh()), len(parents), parents.ctypes.data_as(P),
                                       pa.ctypes.data_as(P) if pa.size else None, len(pa), P(FAKE), P(FAKE),
                                       P(FAKE), None, P(state), None, flags, None)

    assert commit(path=(1, 3)) == -4
    assert commit(flags=1 | gdn.GDN_OUT_BF16) == -1
    assert commit() == -6
