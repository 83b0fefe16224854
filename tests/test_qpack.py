"""The on-disk expert container (moe_qpack_*), CPU only: blobs written by the library's packer
read back bit for bit, through direct and buffered reads, and malformed files are refused."""
import os

import numpy as np
import pytest

from int4_routed_expert_05_b300 import moe, synth


def _aligned(nbytes: int, align: int = 4096) -> np.ndarray:
    raw = np.empty(nbytes + align, dtype=np.uint8)
    off = (-raw.ctypes.data) % align
    return raw[off: off + nbytes]


def _blob(mshape, sh, seed, l, e):
    return moe.pack_expert(mshape, synth.expert_tensors(sh, seed, l, e))


@pytest.mark.parametrize("bits", [4, 8])
def test_roundtrip(tmp_path, bits):
    sh = synth.Shape(256, 16, 2, 64, 64, bits=bits)
    mshape = moe.make_shape(256, 16, 2, 64, 64, bits)
    L, path = 3, str(tmp_path / "experts.qpack")
    q = moe.Qpack.create(path, mshape, L)
    blobs = {}
    for l in range(L):
        for e in range(sh.n_experts):
            if (l, e) == (1, 7):
                continue  # left unwritten: reads as zeros
            blobs[l, e] = _blob(mshape, sh, 4, l, e)
            q.write(l, e, blobs[l, e])
    q.close()
    stride = moe.expert_stride(mshape)
    assert os.path.getsize(path) == 4096 + L * sh.n_experts * stride
    for direct in (True, False):
        r = moe.Qpack.open(path, direct=direct, n_threads=2)
        s2, nl, st, _ = r.info()
        assert (s2.hidden, s2.n_experts, s2.top_k, s2.inter, s2.bits) == (256, 16, 2, 64, bits)
        assert nl == L and st == stride
        buf = _aligned(stride)
        for (l, e), b in blobs.items():
            r.read(l, e, buf)
            assert np.array_equal(buf, b), (l, e, direct)
        r.read(1, 7, buf)
        assert not buf.any()
        with pytest.raises(moe.MoeError):
            r.read(L, 0, buf)
        with pytest.raises(moe.MoeError):
            r.read(0, sh.n_experts, buf)
        r.close()


def test_refuses_truncated_and_foreign_files(tmp_path):
    mshape = moe.make_shape(256, 16, 2, 64, 64, 4)
    path = str(tmp_path / "x.qpack")
    moe.Qpack.create(path, mshape, 2).close()
    size = os.path.getsize(path)
    with open(path, "r+b") as f:  # one byte short
        f.truncate(size - 1)
    with pytest.raises(moe.MoeError):
        moe.Qpack.open(path)
    with open(path, "wb") as f:  # not a container
        f.write(b"\0" * size)
    with pytest.raises(moe.MoeError):
        moe.Qpack.open(path)
    with pytest.raises(moe.MoeError):
        moe.Qpack.open(str(tmp_path / "missing.qpack"))


def test_direct_reads_need_an_aligned_destination(tmp_path):
    mshape = moe.make_shape(256, 16, 2, 64, 64, 4)
    path = str(tmp_path / "a.qpack")
    moe.Qpack.create(path, mshape, 1).close()
    r = moe.Qpack.open(path, direct=True)
    if not r.info()[3]:
        r.close()
        pytest.skip("the file system here does not take O_DIRECT: reads are buffered")
    stride = moe.expert_stride(mshape)
    raw = _aligned(stride + 64)
    with pytest.raises(moe.MoeError):
        r.read(0, 0, raw[16: 16 + stride])
    r.close()
