"""Decode parity at the full 80B and 35B layer shapes (hidden 2048,
intermediate 512, group 64), a few layers deep.

The batched per-layer kernels that run 4 tokens and more only take their
multi-chunk form (several 16-byte code chunks per lane) at hidden 2048; the
tiny shapes never reach it.  Here every layer of a 3-layer 80B-shaped stack
(512 experts, top-10, Zipf router bias, router weights ~ N(0, 1/H)) is
checked against the oracle fed the GPU's own layer input, at 8 and 64 tokens,
int4 and int8, on resident and streaming contexts; and the persistent
decode-stack kernel (1-3 tokens) at the 35B and 80B shapes.  Tolerances are
the layer contract's: chosen experts bit-exact, rel-L2 <= 1e-4 and max-abs
<= 1e-3 * max|y|."""
import concurrent.futures as cf
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

L = 3
W80 = dataclasses.replace(synth.CONFIGS["80b"], n_layers=L)
W35 = dataclasses.replace(synth.CONFIGS["35b"], n_layers=L)
THREADS = max(1, os.cpu_count() or 1)


@pytest.fixture(scope="module", autouse=True)
def _built():
    moe.build()
    moe.load_library()


@pytest.fixture(scope="module", params=[4, 8], ids=["int4", "int8"])
def ctx80(request):
    bits = request.param
    ctx = workload.create_loaded(W80, bits, max_batch=64)
    yield bits, ctx
    moe.moe_destroy(ctx)


def _run_stack(ctx, w, x_np, stream=None):
    B = x_np.shape[0]
    x = torch.from_numpy(x_np).cuda()
    y = torch.empty_like(x)
    xt = torch.empty((L, B, w.hidden), device="cuda")
    yt = torch.empty((L, B, w.hidden), device="cuda")
    it = torch.empty((L, B, w.top_k), dtype=torch.int32, device="cuda")
    moe.moe_forward_decode_stack(ctx, 0, L, x, B, y, 1e-6, xt, it, yt, stream or torch.cuda.current_stream())
    torch.cuda.synchronize()
    assert torch.equal(y, yt[L - 1])
    return xt.cpu().numpy(), it.cpu().numpy(), yt.cpu().numpy()


def _check_stack_vs_oracle(w, bits, xt, it, yt):
    """Every layer against the oracle holding only the experts the GPU chose
    (any other choice by the oracle fails its lookup as well as the index
    comparison)."""
    for l in range(L):
        orc = oracle_layer(w, l, experts=np.unique(it[l]), bits=bits)
        ref = orc.tokens(xt[l], threads=THREADS)
        assert np.array_equal(it[l], ref["idx"]), f"layer {l}: chosen experts differ"
        assert_close(yt[l], ref["y"], what=f"y layer {l}")
        if l + 1 < L:
            assert_close(xt[l + 1], oracle.renorm(yt[l]), rel_l2=1e-6, max_abs_frac=1e-6, what="renorm")


@pytest.mark.parametrize("B", [8, 64])
def test_80b_batched_decode_full_size(ctx80, B):
    """4+ tokens run the per-layer kernels (router, top-k, dispatch, batched
    gate/up, batched down, combine) at hidden 2048: two (int4) or four (int8)
    code chunks per lane on the gate/up rows."""
    bits, ctx = ctx80
    x = synth.tokens(W80.seed, 1000 + B, B, W80.hidden)
    xt, it, yt = _run_stack(ctx, W80, x)
    _check_stack_vs_oracle(W80, bits, xt, it, yt)


@pytest.mark.parametrize("B", [1, 3])
def test_80b_persistent_stack_full_size(ctx80, B):
    """1-3 tokens run the persistent decode-stack kernel at the 80B shape."""
    bits, ctx = ctx80
    x = synth.tokens(W80.seed, 2000 + B, B, W80.hidden)
    xt, it, yt = _run_stack(ctx, W80, x)
    _check_stack_vs_oracle(W80, bits, xt, it, yt)


def test_80b_single_layer_decode_full_size_equals_stack(ctx80):
    """moe_forward_decode of one layer at 64 tokens gives the stack's bits
    for that layer (same kernels), and the routing weights match the oracle."""
    bits, ctx = ctx80
    B = 64
    xt, it, yt = _run_stack(ctx, W80, synth.tokens(W80.seed, 3000, B, W80.hidden))
    l = 1
    x = torch.from_numpy(np.ascontiguousarray(xt[l])).cuda()
    y = torch.empty_like(x)
    idx = torch.empty((B, W80.top_k), dtype=torch.int32, device="cuda")
    wt = torch.empty((B, W80.top_k), dtype=torch.float32, device="cuda")
    moe.moe_forward_decode(ctx, l, x, B, y, idx, wt)
    torch.cuda.synchronize()
    assert np.array_equal(idx.cpu().numpy(), it[l])
    assert np.array_equal(y.cpu().numpy(), yt[l])
    orc = oracle_layer(W80, l, experts=np.unique(it[l]), bits=bits)
    ref = orc.tokens(xt[l], threads=THREADS)
    np.testing.assert_allclose(wt.cpu().numpy(), ref["w"], rtol=2e-6, atol=1e-7)


def test_35b_persistent_stack_full_size():
    """The 35B decode stack's kernel at its own shape (256 experts, top-8),
    1 token, int4: the headline workload, three layers deep."""
    ctx = workload.create_loaded(W35, max_batch=1)
    try:
        x = synth.tokens(W35.seed, 4000, 1, W35.hidden)
        xt, it, yt = _run_stack(ctx, W35, x)
        _check_stack_vs_oracle(W35, 4, xt, it, yt)
    finally:
        moe.moe_destroy(ctx)


@pytest.mark.parametrize("B", [8])
def test_80b_streaming_batched_full_size(B):
    """A streaming context (128 of 512 slots per layer, cold pool, LFU +
    recency) at 8 tokens: outputs bitwise those of the resident context over
    several calls, pool events equal to the oracle simulator replayed on the
    routing, and the first call's layers against the oracle."""
    w = W80
    res = workload.create_loaded(w, max_batch=B)
    st = workload.create_loaded(w, max_batch=B, pool_slots=128)
    try:
        sims = [oracle.PoolSim(128, w.n_experts) for _ in range(L)]
        for step in range(4):
            x = synth.tokens(w.seed, 5000 + step, B, w.hidden)
            xa, ia, ya = _run_stack(res, w, x)
            xb, ib, yb = _run_stack(st, w, x)
            assert np.array_equal(ia, ib) and np.array_equal(ya, yb) and np.array_equal(xa, xb), step
            if step == 0:
                _check_stack_vs_oracle(w, w.bits, xb, ib, yb)
            tr = moe.moe_pool_trace(st)
            for l in range(L):
                want = sims[l].request(ib[l].reshape(-1))
                got = [tuple(int(v) for v in r[2:]) for r in tr if int(r[0]) == step and int(r[1]) == l]
                assert got == want, (step, l)
        s = moe.moe_pool_stats(st)
        assert s["misses"] > 0 and s["calls"] == 4 * L
    finally:
        moe.moe_destroy(res)
        moe.moe_destroy(st)
