"""GPU parity for the snapshot / restore of a sequence's recurrent sections:
the blob is byte-identical to the oracle's, a restore is bit-exact and
touches only its sequence, and a corrupted or foreign blob is refused on the
device with nothing written.  Blobs in device memory and in pinned host
memory (written and read by the kernels directly)."""
import numpy as np
import pytest
import torch

from gdn_testutil import bf16, gdn, gen, host, oracle

pytestmark = pytest.mark.gpu


@pytest.fixture(scope="module", autouse=True)
def _built():
    from hybrid_linear_attention_conv_gb300 import build
    build.build()
    gdn.load()
    assert torch.cuda.is_available()


def _arrays(seed, L, B, s):
    st = gen.normal(seed, "snapg.state", L * B * s.Hv * s.dv * s.dk).astype(np.float32).reshape(
        L, B, s.Hv, s.dv, s.dk)
    tl = gen.normal_bf16(seed, "snapg.tail", L * B * 4 * s.C).reshape(L, B, 4, s.C)
    return st, tl


def _dev(st, tl):
    return torch.from_numpy(st).cuda(), bf16(tl)


@pytest.mark.parametrize("shape,L,B,seq", [
    (gen.Shape(1, 2, 4, 32, 64), 3, 4, 2),
    (gen.Shape(1, 16, 48, 128, 128), 4, 3, 0),
    (gen.TINY, 1, 1, 0),
])
def test_save_equals_oracle_blob_and_restore_is_exact(shape, L, B, seq):
    s = shape
    st, tl = _arrays(61, L, B, s)
    st_d, tl_d = _dev(st, tl)
    blob = gdn.snapshot_save(st_d, tl_d, seq, s.Hk, s.Hv, s.dk, s.dv)
    torch.cuda.synchronize()
    want = oracle.snapshot_save(st, tl, seq, s.Hk, s.Hv, s.dk, s.dv)
    assert np.array_equal(blob.cpu().numpy(), want)
    # restore into other arrays: sequence seq becomes the saved one, bit for bit
    st2, tl2 = _arrays(62, L, B, s)
    st2_d, tl2_d = _dev(st2, tl2)
    assert gdn.snapshot_restore(blob, st2_d, tl2_d, seq, s.Hk, s.Hv, s.dk, s.dv) == 0
    rc, st_ref, tl_ref = oracle.snapshot_restore(want, st2, tl2, seq, s.Hk, s.Hv, s.dk, s.dv)
    assert rc == 0
    assert np.array_equal(st2_d.cpu().numpy().view(np.uint32), st_ref.view(np.uint32))
    assert np.array_equal(host(tl2_d), tl_ref)


def test_strided_layers():
    """Layers spaced apart by more than one layer's array (a view of a bigger
    allocation) are read and written at their own stride."""
    s = gen.Shape(1, 2, 4, 32, 32)
    L, B, seq = 3, 2, 1
    st, tl = _arrays(63, L, B + 1, s)
    st_big, tl_big = _dev(st, tl)
    st_v, tl_v = st_big[:, :B], tl_big[:, :B]
    blob = gdn.snapshot_save(st_v, tl_v, seq, s.Hk, s.Hv, s.dk, s.dv)
    torch.cuda.synchronize()
    want = oracle.snapshot_save(np.ascontiguousarray(st[:, :B]), np.ascontiguousarray(tl[:, :B]), seq, s.Hk, s.Hv,
                                s.dk, s.dv)
    assert np.array_equal(blob.cpu().numpy(), want)
    before_st, before_tl = st_big.clone(), tl_big.clone()
    st_big[:, seq].zero_()
    tl_big[:, seq].zero_()
    gdn.snapshot_restore(blob, st_v, tl_v, seq, s.Hk, s.Hv, s.dk, s.dv)
    assert torch.equal(st_big, before_st) and torch.equal(tl_big, before_tl)


def test_corrupted_and_foreign_blobs_are_refused_untouched():
    s = gen.Shape(1, 2, 4, 32, 64)
    L, B, seq = 2, 2, 1
    st, tl = _arrays(64, L, B, s)
    st_d, tl_d = _dev(st, tl)
    blob = gdn.snapshot_save(st_d, tl_d, seq, s.Hk, s.Hv, s.dk, s.dv)
    st2_d, tl2_d = _dev(*_arrays(65, L, B, s))
    keep_st, keep_tl = st2_d.clone(), tl2_d.clone()
    # one flipped payload bit: the checksum refuses it (status 2)
    bad = blob.clone()
    bad[64 + 12345] ^= 4
    with pytest.raises(gdn.GdnError, match="checksum"):
        gdn.snapshot_restore(bad, st2_d, tl2_d, seq, s.Hk, s.Hv, s.dk, s.dv)
    assert torch.equal(st2_d, keep_st) and torch.equal(tl2_d, keep_tl)
    # the same bytes read as another model (dk and dv swapped: equal sizes,
    # another signature): the header refuses it (status 1)
    o = gen.Shape(1, 2, 4, 64, 32)
    assert gdn.snapshot_bytes(L, o.Hk, o.Hv, o.dk, o.dv) == blob.numel()
    st3 = torch.zeros((L, B, o.Hv, o.dv, o.dk), dtype=torch.float32, device="cuda")
    tl3 = torch.zeros((L, B, 4, o.C), dtype=torch.bfloat16, device="cuda")
    with pytest.raises(gdn.GdnError, match="header"):
        gdn.snapshot_restore(blob, st3, tl3, seq, o.Hk, o.Hv, o.dk, o.dv)
    assert not st3.any() and not tl3.any()
    # a restore after refusals still works (the workspace status is per call)
    assert gdn.snapshot_restore(blob, st2_d, tl2_d, seq, s.Hk, s.Hv, s.dk, s.dv) == 0
    assert torch.equal(st2_d[:, seq], st_d[:, seq]) and torch.equal(tl2_d[:, seq], tl_d[:, seq])


def test_pinned_host_blob_and_file_round_trip(tmp_path):
    """The kernels write the blob straight into pinned host memory and read it
    back from there; a blob written to a file restores the same."""
    s = gen.Shape(1, 16, 48, 128, 128)
    L, B, seq = 2, 2, 1
    st, tl = _arrays(66, L, B, s)
    st_d, tl_d = _dev(st, tl)
    blob_h = gdn.snapshot_save(st_d, tl_d, seq, s.Hk, s.Hv, s.dk, s.dv, host=True)
    torch.cuda.synchronize()
    assert not blob_h.is_cuda and blob_h.is_pinned()
    want = oracle.snapshot_save(st, tl, seq, s.Hk, s.Hv, s.dk, s.dv)
    assert np.array_equal(blob_h.numpy(), want)
    path = str(tmp_path / "seq.gdnsnap")
    gdn.write_snapshot_file(blob_h, path)
    back = gdn.read_snapshot_file(path)
    st2_d, tl2_d = _dev(*_arrays(67, L, B, s))
    gdn.snapshot_restore(back, st2_d, tl2_d, seq, s.Hk, s.Hv, s.dk, s.dv)
    assert torch.equal(st2_d[:, seq], st_d[:, seq]) and torch.equal(tl2_d[:, seq], tl_d[:, seq])


def test_full_model_state_of_one_sequence():
    """48 layers x 64 sequences at the 27B head shape (9.66 GB of state):
    snapshot sequence 63 and restore it into sequence 5; the blob equals the
    oracle's, computed from host copies of that sequence's sections."""
    s = gen.Shape(64, 16, 48, 128, 128)
    L = 48
    g = torch.Generator(device="cuda")
    g.manual_seed(68)
    st_d = torch.randn((L, s.B, s.Hv, s.dv, s.dk), generator=g, device="cuda")
    tl_d = torch.randn((L, s.B, 4, s.C), generator=g, device="cuda").to(torch.bfloat16)
    blob = gdn.snapshot_save(st_d, tl_d, 63, s.Hk, s.Hv, s.dk, s.dv)
    torch.cuda.synchronize()
    st_h = st_d[:, 63:64].cpu().numpy()
    tl_h = host(tl_d[:, 63:64].contiguous())
    want = oracle.snapshot_save(st_h, tl_h, 0, s.Hk, s.Hv, s.dk, s.dv)
    assert np.array_equal(blob.cpu().numpy(), want)
    neighbour = st_d[:, 4].clone()
    gdn.snapshot_restore(blob, st_d, tl_d, 5, s.Hk, s.Hv, s.dk, s.dv)
    assert torch.equal(st_d[:, 5], st_d[:, 63]) and torch.equal(tl_d[:, 5], tl_d[:, 63])
    assert torch.equal(st_d[:, 4], neighbour)
