"""Prefill parity: the tensor-core grouped-GEMM path through the C ABI against
the CPU oracle's prefill definition (bf16 operands, fp64 accumulation):
chosen experts bit-exact, routing weights to fp32 rounding, layer output
within the layer tolerance."""
import dataclasses
import math

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

TINY = synth.CONFIGS["tiny"]
# tiny dims with the 80B-style router (logits ~ N(0,1) plus a Zipf(1.1) popularity bias):
# skewed counts, so some experts fill several 256-row chunks and many get none
TINY_ZIPF = dataclasses.replace(TINY, router_sigma=1.0 / math.sqrt(256), zipf_s=1.1)
# one layer with the real hidden/intermediate sizes and fewer experts
WIDE = synth.Workload("wide", n_layers=1, hidden=2048, n_experts=64, top_k=4, inter=512, shared_inter=512,
                      router_sigma=1.0 / math.sqrt(2048), zipf_s=1.1, renorm=False)


@pytest.fixture(scope="module", autouse=True)
def _built():
    moe.build()
    moe.load_library()


def _prefill(ctx, w, x_np, layer=0):
    T = x_np.shape[0]
    x = torch.from_numpy(x_np).cuda()
    y = torch.full_like(x, float("nan"))  # the call must overwrite every element
    idx = torch.empty((T, w.top_k), dtype=torch.int32, device="cuda")
    wt = torch.empty((T, w.top_k), dtype=torch.float32, device="cuda")
    moe.moe_forward_prefill(ctx, layer, x, T, y, idx, wt, torch.cuda.current_stream())
    torch.cuda.synchronize()
    return y.cpu().numpy(), idx.cpu().numpy(), wt.cpu().numpy()


def _check(w, x_np, y, idx, wt, rows=None, norm_topk=True, threads=8):
    orc = oracle_layer(w, 0, norm_topk=norm_topk)
    rows = np.arange(x_np.shape[0]) if rows is None else np.asarray(rows)
    ref = orc.tokens(x_np[rows], prefill=True, threads=threads)
    assert np.array_equal(idx[rows], ref["idx"])
    np.testing.assert_allclose(wt[rows], ref["w"], rtol=2e-6, atol=1e-7)
    return assert_close(y[rows], ref["y"])


@pytest.mark.parametrize("T", [1, 37, 300, 1200])
def test_tiny_prefill_matches_oracle(T):
    w = TINY
    ctx = workload.create_loaded(w, max_tokens=T)
    try:
        x = synth.tokens(w.seed, 3, T, w.hidden)
        _check(w, x, *_prefill(ctx, w, x))
    finally:
        moe.moe_destroy(ctx)


def test_tiny_prefill_zipf_skew_full_and_partial_chunks():
    w = TINY_ZIPF
    T = 1500
    ctx = workload.create_loaded(w, max_tokens=T)
    try:
        x = synth.tokens(w.seed, 5, T, w.hidden)
        y, idx, wt = _prefill(ctx, w, x)
        counts = np.bincount(idx.ravel(), minlength=w.n_experts)
        assert counts.max() > 2 * 256 and (counts % 256 != 0).any()  # several full chunks and ragged tails
        _check(w, x, y, idx, wt)
    finally:
        moe.moe_destroy(ctx)


def test_two_stage_router_small():
    """128 experts (a multiple of 128): the router runs as tensor-core approximate
    logits plus exact logits of the candidates the error bound leaves; the
    chosen experts and weights must still equal the exact router's."""
    w = dataclasses.replace(TINY_ZIPF, n_experts=128, top_k=6)
    T = 700
    ctx = workload.create_loaded(w, max_tokens=T)
    try:
        x = synth.tokens(w.seed, 21, T, w.hidden)
        y, idx, wt = _prefill(ctx, w, x)
        _check(w, x, y, idx, wt)
        _prefill(ctx, w, x[:5])  # a second call reports any failed device-side check of the first
    finally:
        moe.moe_destroy(ctx)


def test_tiny_prefill_int8():
    w = dataclasses.replace(TINY, bits=8)
    ctx = workload.create_loaded(w, max_tokens=300)
    try:
        x = synth.tokens(w.seed, 7, 300, w.hidden)
        _check(w, x, *_prefill(ctx, w, x))
    finally:
        moe.moe_destroy(ctx)


def test_tiny_prefill_full_softmax_weights():
    w = TINY
    ctx = workload.create_loaded(w, max_tokens=64, norm_topk=False)
    try:
        x = synth.tokens(w.seed, 9, 64, w.hidden)
        _check(w, x, *_prefill(ctx, w, x), norm_topk=False)
    finally:
        moe.moe_destroy(ctx)


def test_tiny_prefill_without_shared_expert():
    w = dataclasses.replace(TINY, shared_inter=0)
    ctx = workload.create_loaded(w, max_tokens=200)
    try:
        x = synth.tokens(w.seed, 11, 200, w.hidden)
        _check(w, x, *_prefill(ctx, w, x))
    finally:
        moe.moe_destroy(ctx)


def test_tiny_prefill_fewer_tokens_than_max_and_repeat():
    """A context sized for 1000 tokens serves smaller calls; repeated calls agree bitwise
    in the chosen experts and to fp32-reduction order in y."""
    w = TINY
    ctx = workload.create_loaded(w, max_tokens=1000)
    try:
        x = synth.tokens(w.seed, 13, 129, w.hidden)
        y1, i1, w1 = _prefill(ctx, w, x)
        y2, i2, w2 = _prefill(ctx, w, x)
        assert np.array_equal(i1, i2) and np.array_equal(w1, w2)
        assert_close(y2, y1, rel_l2=1e-6, max_abs_frac=1e-5)
        _check(w, x, y1, i1, w1)
    finally:
        moe.moe_destroy(ctx)


def test_prefill_single_token_equals_decode_to_bf16():
    """T = 1: the prefill path (bf16 operands) and the decode path (exact
    dequantised weights) agree to the bf16 rounding of the operands (unit
    roundoff 2^-9 per operand, three chained products: rel-L2 below 2^-7)."""
    w = TINY
    ctx = workload.create_loaded(w, max_tokens=1, max_batch=1)
    try:
        x_np = synth.tokens(w.seed, 15, 1, w.hidden)
        y_p, i_p, _ = _prefill(ctx, w, x_np)
        x = torch.from_numpy(x_np).cuda()
        y = torch.empty_like(x)
        idx = torch.empty((1, w.top_k), dtype=torch.int32, device="cuda")
        moe.moe_forward_decode(ctx, 0, x, 1, y, idx, None, torch.cuda.current_stream())
        torch.cuda.synchronize()
        assert np.array_equal(i_p, idx.cpu().numpy())
        assert_close(y_p, y.cpu().numpy(), rel_l2=2.0 ** -7, max_abs_frac=2.0 ** -5)
    finally:
        moe.moe_destroy(ctx)


@pytest.mark.parametrize("w,T", [(TINY_ZIPF, 200), (WIDE, 160)])
def test_prefill_equals_decode_batches(w, T):
    """One prefill of T tokens against the same tokens decoded in batches of up
    to 64 (the full-sequence against incremental check, for the MoE layer):
    identical experts, routing weights to a few fp32 roundings, outputs within the
    bf16 rounding of the prefill operands (rel-L2 below 2^-7)."""
    ctx = workload.create_loaded(w, max_tokens=T, max_batch=64)
    try:
        x_np = synth.tokens(w.seed, 21, T, w.hidden)
        y_p, i_p, w_p = _prefill(ctx, w, x_np)
        ys, idxs, ws = [], [], []
        for t0 in range(0, T, 64):
            xb = torch.from_numpy(x_np[t0:t0 + 64]).cuda()
            B = xb.shape[0]
            y = torch.empty_like(xb)
            idx = torch.empty((B, w.top_k), dtype=torch.int32, device="cuda")
            wt = torch.empty((B, w.top_k), dtype=torch.float32, device="cuda")
            moe.moe_forward_decode(ctx, 0, xb, B, y, idx, wt, torch.cuda.current_stream())
            torch.cuda.synchronize()
            ys.append(y.cpu().numpy()), idxs.append(idx.cpu().numpy()), ws.append(wt.cpu().numpy())
        assert np.array_equal(i_p, np.concatenate(idxs))
        np.testing.assert_allclose(w_p, np.concatenate(ws), rtol=5e-6, atol=2e-7)  # each is within 2e-6 of the oracle
        assert_close(y_p, np.concatenate(ys), rel_l2=2.0 ** -7, max_abs_frac=2.0 ** -5)
    finally:
        moe.moe_destroy(ctx)


def test_wide_prefill_sampled_rows():
    """Hidden 2048 / inter 512 (the 80B expert shape), 64 experts, Zipf-skewed
    routing; 600 tokens, oracle on a seeded sample of 48 rows plus all routes."""
    w = WIDE
    T = 600
    ctx = workload.create_loaded(w, max_tokens=T)
    try:
        x = synth.tokens(w.seed, 1, T, w.hidden)
        y, idx, wt = _prefill(ctx, w, x)
        orc = oracle_layer(w, 0)
        routes = [orc.route(x[t]) for t in range(T)]
        assert np.array_equal(idx, np.stack([r[1] for r in routes]))
        rows = np.sort(np.random.default_rng(17).choice(T, 48, replace=False))
        _check(w, x, y, idx, wt, rows=rows)
    finally:
        moe.moe_destroy(ctx)


def test_prefill_rejects_bad_calls():
    w = TINY
    ctx = workload.create_loaded(w, max_tokens=8)
    try:
        x = torch.zeros((16, w.hidden), device="cuda")
        y = torch.empty_like(x)
        with pytest.raises(moe.MoeError) as e:
            moe.moe_forward_prefill(ctx, 0, x, 16, y)  # T > max_tokens
        assert e.value.code == moe.MOE_EINVAL
        with pytest.raises(moe.MoeError) as e:
            moe.moe_forward_prefill(ctx, 0, x, 0, y)
        assert e.value.code == moe.MOE_EINVAL
        with pytest.raises(moe.MoeError) as e:
            moe.moe_forward_prefill(ctx, 0, x, 4, x)  # y aliases x
        assert e.value.code == moe.MOE_EINVAL
    finally:
        moe.moe_destroy(ctx)
    ctx = workload.create_loaded(w)  # no prefill scratch
    try:
        x = torch.zeros((1, w.hidden), device="cuda")
        with pytest.raises(moe.MoeError) as e:
            moe.moe_forward_prefill(ctx, 0, x, 1, torch.empty_like(x))
        assert e.value.code == moe.MOE_ESTATE
    finally:
        moe.moe_destroy(ctx)


def test_80b_prefill_full_size_sampled():
    """The full 80B-shaped prefill layer (512 experts, top-10, 4096 tokens):
    every token's experts bit-exact against the oracle router, the sorted
    dispatch consistent, and a seeded sample of 32 output rows within the
    layer tolerance."""
    import concurrent.futures as cf
    w = synth.CONFIGS["80b-prefill"]
    T = w.prefill_tokens
    ctx = workload.create_loaded(w, max_tokens=T)
    try:
        x = synth.tokens(w.seed, 0, T, w.hidden)
        y, idx, wt = _prefill(ctx, w, x)
        router = oracle_layer(w, 0, experts=[])
        with cf.ThreadPoolExecutor(16) as ex:
            routes = list(ex.map(lambda t: router.route(x[t]), range(T)))
        assert np.array_equal(idx, np.stack([r[1] for r in routes]))
        np.testing.assert_allclose(wt, np.stack([r[2] for r in routes]), rtol=2e-6, atol=1e-7)
        counts = np.bincount(idx.ravel(), minlength=w.n_experts)
        assert counts.sum() == T * w.top_k and counts.max() > 256  # Zipf-skewed: hot experts span chunks
        _prefill(ctx, w, x[:8])  # reports any failed device-side check of the full call
        rows = np.sort(np.random.default_rng(23).choice(T, 32, replace=False))
        orc = oracle_layer(w, 0, experts=np.unique(idx[rows]))
        ref = orc.tokens(x[rows], prefill=True, threads=16)
        assert np.array_equal(idx[rows], ref["idx"])
        assert_close(y[rows], ref["y"])
    finally:
        moe.moe_destroy(ctx)
