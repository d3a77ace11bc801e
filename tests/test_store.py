"""The expert container (routed blobs on disk, one positioned read per blob):
layout against its documented header, round trip of the packer's bytes, and
errors on bad calls and malformed files.  Host only."""
import os
import struct

import numpy as np
import pytest

import synth

moe = pytest.importorskip("int4_expert_streaming_gb300")
from int4_expert_streaming_gb300 import workload  # noqa: E402

TINY2 = synth.Workload("tiny2", n_layers=2, hidden=256, n_experts=16, top_k=2, inter=128, shared_inter=128,
                       router_sigma=synth.CONFIGS["tiny"].router_sigma)


@pytest.fixture(scope="module")
def lib():
    moe.build()
    return moe.load_library()


def test_header_layout_and_size(lib, tmp_path):
    """The 4096-byte little-endian header as documented: magic, version 1,
    shape, group 64, stride, data offset 4096; the file holds every blob."""
    p = tmp_path / "c.bin"
    moe.moe_store_create(p, 3, 16, 256, 128, 4)
    stride = moe.moe_blob_stride(256, 128, 4)
    raw = p.read_bytes()
    assert len(raw) == 4096 + 3 * 16 * stride and stride % 4096 == 0
    assert raw[:8] == b"MOEXPRT1"
    assert struct.unpack_from("<7I", raw, 8) == (1, 3, 16, 256, 128, 4, 64)
    assert struct.unpack_from("<2Q", raw, 40) == (stride, 4096)
    assert raw[56:4096] == bytes(4096 - 56) and raw[4096:] == bytes(len(raw) - 4096)  # unwritten blobs are zeros
    assert moe.moe_store_info(p) == dict(n_layers=3, n_experts=16, hidden=256, inter=128, bits=4, stride=stride)


@pytest.mark.parametrize("bits", [4, 8])
def test_round_trip_of_packed_layers(lib, tmp_path, bits):
    p = tmp_path / f"w{bits}.bin"
    workload.write_store(TINY2, p, bits=bits)
    stride = moe.moe_blob_stride(TINY2.hidden, TINY2.inter, bits)
    raw = p.read_bytes()
    for layer in range(TINY2.n_layers):
        blobs, *_ = workload.layer_blobs(TINY2, layer, bits)
        for e in (0, 7, 15):
            want = blobs[e * stride:(e + 1) * stride]
            assert np.array_equal(moe.moe_store_read(p, layer, e, stride), want)
            off = 4096 + (layer * TINY2.n_experts + e) * stride  # the documented position
            assert raw[off:off + stride] == want.tobytes()


def test_errors(lib, tmp_path):
    p = tmp_path / "c.bin"
    stride = moe.moe_blob_stride(256, 128, 4)
    with pytest.raises(moe.MoeError) as e:
        moe.moe_store_create(p, 2, 16, 256, 128, 3)  # bits
    assert e.value.code == moe.MOE_EINVAL
    with pytest.raises(moe.MoeError) as e:
        moe.moe_store_info(tmp_path / "missing.bin")
    assert e.value.code == moe.MOE_EIO
    moe.moe_store_create(p, 2, 16, 256, 128, 4)
    for layer, expert in ((2, 0), (-1, 0), (0, 16)):
        with pytest.raises(moe.MoeError) as e:
            moe.moe_store_read(p, layer, expert, stride)
        assert e.value.code == moe.MOE_EINVAL
    with pytest.raises(moe.MoeError) as e:
        moe.moe_store_write_layer(p, 0, np.zeros(16 * 4096, np.uint8), 4096)  # wrong stride
    assert e.value.code == moe.MOE_EINVAL
    with pytest.raises(moe.MoeError) as e:
        moe.moe_store_write_layer(p, 2, np.zeros(16 * stride, np.uint8), stride)  # layer out of range
    assert e.value.code == moe.MOE_EINVAL
    # truncated: shorter than its header says
    with open(p, "r+b") as f:
        f.truncate(4096 + stride)
    with pytest.raises(moe.MoeError) as e:
        moe.moe_store_read(p, 0, 0, stride)
    assert e.value.code == moe.MOE_EIO
    # a foreign file
    q = tmp_path / "foreign.bin"
    q.write_bytes(os.urandom(8192))
    with pytest.raises(moe.MoeError) as e:
        moe.moe_store_info(q)
    assert e.value.code == moe.MOE_EIO


def test_create_rejects_store_path_for_resident_or_bad_flags(lib, tmp_path):
    """Checked before any GPU work."""
    p = tmp_path / "c.bin"
    moe.moe_store_create(p, 2, 16, 256, 128, 4)
    for kw in (dict(store_path=p), dict(store_path=p, pool_slots=4, store_flags=0x2)):
        cfg = moe.make_config(2, 256, 16, 2, 128, 128, **kw)
        with pytest.raises(moe.MoeError) as e:
            moe.moe_create(cfg)
        assert e.value.code == moe.MOE_EINVAL
