"""A mixed int4/int8 store (moe_config.layer_bits): each layer's blobs packed
for its own width, every slot sized for the widest layer.

Every layer is checked against the oracle at that layer's own width (decode
at 1 and 5 tokens, prefill), a streaming context must give the resident
context's bits with pool events equal to the oracle simulator, and one
full-size case (hidden 2048, 512 experts, int8 then int4) catches pitch and
stride mistakes that the tiny shapes could hide."""
import dataclasses
import os

import numpy as np
import pytest

import oracle
import synth
from _common import assert_close, oracle_layer

torch = pytest.importorskip("torch")
pytestmark = [pytest.mark.gpu,
              pytest.mark.skipif(not torch.cuda.is_available(), reason="needs a CUDA GPU")]

import int4_expert_streaming_gb300 as moe  # noqa: E402
from int4_expert_streaming_gb300 import workload  # noqa: E402

BITS = [4, 8, 4]
W = dataclasses.replace(synth.CONFIGS["tiny"], n_layers=3, zipf_s=1.1)
THREADS = max(1, os.cpu_count() or 1)


@pytest.fixture(scope="module", autouse=True)
def _built():
    moe.build()
    moe.load_library()


def _stack(ctx, w, x_np):
    L, B = w.n_layers, x_np.shape[0]
    x = torch.from_numpy(x_np).cuda()
    y = torch.empty_like(x)
    xt = torch.empty((L, B, w.hidden), device="cuda")
    yt = torch.empty((L, B, w.hidden), device="cuda")
    it = torch.empty((L, B, w.top_k), dtype=torch.int32, device="cuda")
    moe.moe_forward_decode_stack(ctx, 0, L, x, B, y, 1e-6, xt, it, yt, torch.cuda.current_stream())
    torch.cuda.synchronize()
    assert torch.equal(y, yt[L - 1])
    return xt.cpu().numpy(), it.cpu().numpy(), yt.cpu().numpy()


def _check_layers(w, bits, xt, it, yt):
    for l in range(w.n_layers):
        orc = oracle_layer(w, l, experts=np.unique(it[l]), bits=bits[l])
        ref = orc.tokens(xt[l], threads=THREADS)
        assert np.array_equal(it[l], ref["idx"]), f"layer {l} ({bits[l]}-bit): chosen experts differ"
        assert_close(yt[l], ref["y"], what=f"y layer {l} ({bits[l]}-bit)")


@pytest.mark.parametrize("B", [1, 5])
def test_mixed_store_decode_each_layer_at_its_width(B):
    ctx = workload.create_loaded(W, max_batch=B, layer_bits=BITS)
    try:
        x = synth.tokens(W.seed, 60 + B, B, W.hidden)
        xt, it, yt = _stack(ctx, W, x)
        _check_layers(W, BITS, xt, it, yt)
        # single-layer calls give the stack's bits
        for l in range(W.n_layers):
            xl = torch.from_numpy(np.ascontiguousarray(xt[l])).cuda()
            yl = torch.empty_like(xl)
            il = torch.empty((B, W.top_k), dtype=torch.int32, device="cuda")
            moe.moe_forward_decode(ctx, l, xl, B, yl, il)
            torch.cuda.synchronize()
            assert np.array_equal(il.cpu().numpy(), it[l]) and np.array_equal(yl.cpu().numpy(), yt[l]), l
    finally:
        moe.moe_destroy(ctx)


@pytest.mark.parametrize("B", [2, 5])
def test_mixed_store_streaming_equals_resident(B):
    """6 of 16 slots per layer: misses copy each layer's own stride into
    slots sized for the widest layer."""
    res = workload.create_loaded(W, max_batch=B, layer_bits=BITS)
    st = workload.create_loaded(W, max_batch=B, pool_slots=6, layer_bits=BITS)
    try:
        sims = [oracle.PoolSim(6, W.n_experts) for _ in range(W.n_layers)]
        for step in range(6):
            x = synth.tokens(W.seed, 70 + step, B, W.hidden)
            xa, ia, ya = _stack(res, W, x)
            xb, ib, yb = _stack(st, W, x)
            assert np.array_equal(ia, ib) and np.array_equal(ya, yb), step
            tr = moe.moe_pool_trace(st)
            for l in range(W.n_layers):
                want = sims[l].request(ib[l].reshape(-1))
                got = [tuple(int(v) for v in r[2:]) for r in tr if int(r[0]) == step and int(r[1]) == l]
                assert got == want, (step, l)
        s = moe.moe_pool_stats(st)
        assert s["misses"] > 0
        strides = [moe.moe_blob_stride(W.hidden, W.inter, b) for b in BITS]
        per_layer = [moe.moe_pool_stats(st, l) for l in range(W.n_layers)]
        for l in range(W.n_layers):
            assert per_layer[l]["h2d_bytes"] == per_layer[l]["misses"] * strides[l], l
    finally:
        moe.moe_destroy(res)
        moe.moe_destroy(st)


def test_mixed_store_prefill_each_layer_at_its_width():
    T = 300
    ctx = workload.create_loaded(W, max_tokens=T, layer_bits=BITS)
    try:
        for l in range(W.n_layers):
            x_np = synth.tokens(W.seed, 80 + l, T, W.hidden)
            x = torch.from_numpy(x_np).cuda()
            y = torch.full_like(x, float("nan"))
            idx = torch.empty((T, W.top_k), dtype=torch.int32, device="cuda")
            wt = torch.empty((T, W.top_k), dtype=torch.float32, device="cuda")
            moe.moe_forward_prefill(ctx, l, x, T, y, idx, wt, torch.cuda.current_stream())
            torch.cuda.synchronize()
            ref = oracle_layer(W, l, bits=BITS[l]).tokens(x_np, prefill=True, threads=THREADS)
            assert np.array_equal(idx.cpu().numpy(), ref["idx"]), l
            np.testing.assert_allclose(wt.cpu().numpy(), ref["w"], rtol=2e-6, atol=1e-7)
            assert_close(y.cpu().numpy(), ref["y"], what=f"prefill y layer {l} ({BITS[l]}-bit)")
    finally:
        moe.moe_destroy(ctx)


@pytest.mark.parametrize("B", [1, 8])
def test_mixed_store_full_size(B):
    """80B layer shapes, int8 layer then int4 layer."""
    w = dataclasses.replace(synth.CONFIGS["80b"], n_layers=2)
    bits = [8, 4]
    ctx = workload.create_loaded(w, max_batch=B, layer_bits=bits)
    try:
        x = synth.tokens(w.seed, 90 + B, B, w.hidden)
        xt, it, yt = _stack(ctx, w, x)
        _check_layers(w, bits, xt, it, yt)
    finally:
        moe.moe_destroy(ctx)
