"""Host-side checks of libmoe.so that need no GPU: the library loads and exports
every symbol include/moe.h declares, the packer's bytes equal the oracle
packer's, the slot-pool policy replays the oracle pool simulator, and invalid
arguments fail cleanly."""
import os
import re

import numpy as np
import pytest

import int4_expert_streaming_gb300 as moe
import oracle
import synth

ROOT = os.path.dirname(os.path.dirname(os.path.abspath(__file__)))


@pytest.fixture(scope="module")
def lib():
    moe.build()
    return moe.load_library()


def _declared():
    text = open(os.path.join(ROOT, "include", "moe.h")).read()
    text = re.sub(r"/\*.*?\*/", "", text, flags=re.S)
    return sorted(set(re.findall(r"\b(moe_[a-z_]+)\s*\(", text)))


def test_library_exports_every_declared_symbol(lib):
    declared = _declared()
    assert len(declared) >= 16
    missing = [n for n in declared if not hasattr(lib, n)]
    assert not missing, missing
    assert sorted(moe.EXPORTS) == declared


@pytest.mark.parametrize("bits,H,I", [(4, 256, 128), (8, 256, 128), (4, 2048, 512), (8, 2048, 512), (4, 256, 64)])
def test_packer_bytes_equal_oracle_packer(lib, bits, H, I):
    d = synth.expert(5, 3, 7, H, I, bits)
    ours = moe.moe_pack_expert(H, I, bits, d)
    ref = oracle.pack_blob(d, H, I, bits)
    assert ours.nbytes == ref.nbytes == moe.moe_blob_stride(H, I, bits)
    assert np.array_equal(ours, ref)
    assert moe.moe_blob_bytes(H, I, bits) == oracle.blob_bytes(H, I, bits)


def test_packer_rejects_bad_input(lib):
    d = synth.expert(1, 0, 0, 256, 64, 4)
    bad = dict(d)
    bad["q_up"] = d["q_up"].copy()
    bad["q_up"][0, 0] = 16  # does not fit in 4 bits
    with pytest.raises(moe.MoeError) as e:
        moe.moe_pack_expert(256, 64, 4, bad)
    assert e.value.code == moe.MOE_EINVAL
    with pytest.raises(moe.MoeError):
        moe.moe_pack_expert(256, 64, 4, d, out=np.empty(100, np.uint8))
    assert moe.moe_blob_stride(100, 64, 4) == 0 and moe.moe_blob_stride(256, 64, 3) == 0


@pytest.mark.parametrize("policy", [moe.MOE_EVICT_LFU_RECENCY, moe.MOE_EVICT_LRU, moe.MOE_EVICT_LFU_PERSIST,
                                    moe.MOE_EVICT_LFU_AGED])
@pytest.mark.parametrize("slots,E,kmax", [(4, 16, 3), (128, 512, 10), (8, 8, 8), (2, 6, 2)])
def test_slotpool_replays_oracle_pool_sim(lib, policy, slots, E, kmax):
    """Random Zipf-skewed request streams: events identical to the oracle simulator
    (aging every 7 calls, so the aged policy halves many times in 400 calls)."""
    rng = np.random.default_rng(slots * 1000 + E + policy)
    p = 1.0 / np.arange(1, E + 1) ** 1.1
    p /= p.sum()
    pool = moe.moe_slotpool_create(slots, E, policy, aging_period=7)
    sim = oracle.PoolSim(slots, E, policy, aging_period=7)
    try:
        for _ in range(400):
            n = int(rng.integers(1, min(kmax, slots) + 1))
            req = sorted(set(int(v) for v in rng.choice(E, size=n, p=p)))
            assert moe.moe_slotpool_request(pool, req) == sim.request(req)
    finally:
        moe.moe_slotpool_destroy(pool)


def test_slotpool_errors(lib):
    pool = moe.moe_slotpool_create(2, 6)
    try:
        with pytest.raises(moe.MoeError) as e:
            moe.moe_slotpool_request(pool, [0, 1, 2])
        assert e.value.code == moe.MOE_EPOOL
        with pytest.raises(moe.MoeError) as e:
            moe.moe_slotpool_request(pool, [3, 1])
        assert e.value.code == moe.MOE_EINVAL
        with pytest.raises(moe.MoeError):
            moe.moe_slotpool_request(pool, [6])
        assert moe.moe_slotpool_request(pool, []) == []
    finally:
        moe.moe_slotpool_destroy(pool)
    with pytest.raises(moe.MoeError):
        moe.moe_slotpool_create(0, 4)
    with pytest.raises(moe.MoeError):
        moe.moe_slotpool_create(2, 4, 4)


def test_slotpool_default_aging_period_is_64(lib):
    """aging_period <= 0 means 64: identical events to an explicit 64."""
    rng = np.random.default_rng(3)
    a = moe.moe_slotpool_create(6, 24, moe.MOE_EVICT_LFU_AGED, 0)
    b = moe.moe_slotpool_create(6, 24, moe.MOE_EVICT_LFU_AGED, 64)
    sim = oracle.PoolSim(6, 24, oracle.POLICY_LFU_AGED, aging_period=64)
    try:
        for _ in range(300):
            req = sorted(int(v) for v in rng.choice(24, size=3, replace=False))
            want = sim.request(req)
            assert moe.moe_slotpool_request(a, req) == want == moe.moe_slotpool_request(b, req)
    finally:
        moe.moe_slotpool_destroy(a)
        moe.moe_slotpool_destroy(b)


@pytest.mark.parametrize("field,value", [("hidden", 100), ("bits", 3), ("group_size", 32), ("top_k", 0),
                                         ("top_k", 17), ("pool_slots", 1), ("max_batch", 65), ("inter", 96),
                                         ("policy", 4), ("policy", -1)])
def test_create_rejects_bad_config_before_any_gpu_work(lib, field, value):
    cfg = moe.make_config(2, 256, 16, 2, 128, 128)
    setattr(cfg, field, value)
    with pytest.raises(moe.MoeError) as e:
        moe.moe_create(cfg)
    assert e.value.code == moe.MOE_EINVAL
    assert moe.moe_last_error(None)


@pytest.mark.parametrize("kw", [dict(layer_bits=[4, 3]), dict(layer_bits=[8, 4], inter=1024),
                                dict(layer_bits=[4, 8], pool_slots=4, store_path="/nonexistent/c.bin")])
def test_create_rejects_bad_layer_bits_before_any_gpu_work(lib, kw):
    """Widths other than 4 or 8, a row too long for a layer's width, and a
    mixed stack with an expert container (which holds one width)."""
    args = dict(n_layers=2, hidden=256, n_experts=16, top_k=2, inter=128, shared_inter=128)
    args.update(kw)
    cfg = moe.make_config(**args)
    with pytest.raises(moe.MoeError) as e:
        moe.moe_create(cfg)
    assert e.value.code == moe.MOE_EINVAL
    assert "layer_bits" in moe.moe_last_error(None) or "width" in moe.moe_last_error(None)


def test_binding_rejects_host_tensors_for_device_args(lib):
    import torch
    with pytest.raises(ValueError):
        moe.moe_forward_decode(0, 0, torch.zeros(4), 1, torch.zeros(4))
