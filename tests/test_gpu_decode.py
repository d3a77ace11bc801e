"""Decode parity: the CUDA path through the C ABI against the CPU oracle on the
tiny workload and its variants (batch sizes, int8, full-softmax weights, Zipf
router bias, multi-layer stacks, streaming slot pool)."""
import dataclasses

import numpy as np
import pytest

import oracle
import synth
from _common import assert_close, oracle_layer, seed_with_gap

torch = pytest.importorskip("torch")
pytestmark = [pytest.mark.gpu,
              pytest.mark.skipif(not torch.cuda.is_available(), reason="needs a CUDA GPU")]

import int4_expert_streaming_gb300 as moe  # noqa: E402
from int4_expert_streaming_gb300 import workload  # noqa: E402

TINY = synth.CONFIGS["tiny"]


@pytest.fixture(scope="module", autouse=True)
def _built():
    moe.build()
    moe.load_library()


def _ctx(w, **kw):
    return workload.create_loaded(w, **kw)


def _decode(ctx, w, x_np, layer=0):
    B = x_np.shape[0]
    x = torch.from_numpy(x_np).cuda()
    y = torch.empty_like(x)
    idx = torch.empty((B, w.top_k), dtype=torch.int32, device="cuda")
    wt = torch.empty((B, w.top_k), dtype=torch.float32, device="cuda")
    moe.moe_forward_decode(ctx, layer, x, B, y, idx, wt, torch.cuda.current_stream())
    torch.cuda.synchronize()
    return y.cpu().numpy(), idx.cpu().numpy(), wt.cpu().numpy()


def _check_layer(w, x_np, y, idx, wt, layer=0, norm_topk=True, orc=None):
    orc = orc or oracle_layer(w, layer, norm_topk=norm_topk)
    ref = orc.tokens(x_np)
    assert np.array_equal(idx, ref["idx"]), (idx, ref["idx"])
    np.testing.assert_allclose(wt, ref["w"], rtol=2e-6, atol=1e-7)
    return assert_close(y, ref["y"])


@pytest.mark.parametrize("B", [1, 3, 8])
def test_tiny_decode_matches_oracle(B):
    w = seed_with_gap(TINY, B)
    ctx = _ctx(w, max_batch=B)
    try:
        x = synth.tokens(w.seed, 0, B, w.hidden)
        _check_layer(w, x, *_decode(ctx, w, x))
    finally:
        moe.moe_destroy(ctx)


def test_tiny_decode_max_batch_64_all_experts_active():
    w = TINY
    ctx = _ctx(w, max_batch=64)
    try:
        x = synth.tokens(w.seed, 1, 64, w.hidden)
        y, idx, wt = _decode(ctx, w, x)
        assert len(np.unique(idx)) == w.n_experts  # every expert is routed to by someone
        _check_layer(w, x, y, idx, wt)
    finally:
        moe.moe_destroy(ctx)


def test_tiny_decode_int8():
    w = dataclasses.replace(seed_with_gap(TINY, 4), bits=8)
    ctx = _ctx(w, max_batch=4)
    try:
        x = synth.tokens(w.seed, 0, 4, w.hidden)
        _check_layer(w, x, *_decode(ctx, w, x))
    finally:
        moe.moe_destroy(ctx)


def test_tiny_decode_full_softmax_weights():
    w = seed_with_gap(TINY, 2)
    ctx = _ctx(w, max_batch=2, norm_topk=False)
    try:
        x = synth.tokens(w.seed, 0, 2, w.hidden)
        _check_layer(w, x, *_decode(ctx, w, x), norm_topk=False)
    finally:
        moe.moe_destroy(ctx)


def test_tiny_decode_with_zipf_router_bias_and_wider_shapes():
    """E = 64, k = 10, Zipf(1.1) bias, router weights ~ N(0, 1/H) (the 80B
    recipe at tiny width), hidden 512, intermediate 192 (three groups)."""
    w = dataclasses.replace(TINY, n_experts=64, top_k=10, hidden=512, inter=192, shared_inter=64,
                            router_sigma=1.0 / np.sqrt(512), zipf_s=1.1)
    w = seed_with_gap(w, 5)
    ctx = _ctx(w, max_batch=5)
    try:
        x = synth.tokens(w.seed, 0, 5, w.hidden)
        _check_layer(w, x, *_decode(ctx, w, x))
    finally:
        moe.moe_destroy(ctx)


def test_tiny_stack_layer_by_layer():
    """Three-layer stack with renormalisation: each layer checked against the
    oracle fed the GPU's own layer input; the renormalisation checked too."""
    w = dataclasses.replace(TINY, n_layers=3)
    B = 4
    ctx = _ctx(w, max_batch=B)
    try:
        x = torch.from_numpy(synth.tokens(w.seed, 0, B, w.hidden)).cuda()
        y = torch.empty_like(x)
        xt = torch.empty((3, B, w.hidden), device="cuda")
        yt = torch.empty((3, B, w.hidden), device="cuda")
        it = torch.empty((3, B, w.top_k), dtype=torch.int32, device="cuda")
        moe.moe_forward_decode_stack(ctx, 0, 3, x, B, y, 1e-6, xt, it, yt, torch.cuda.current_stream())
        torch.cuda.synchronize()
        xt, yt, it = xt.cpu().numpy(), yt.cpu().numpy(), it.cpu().numpy()
        assert np.array_equal(xt[0], x.cpu().numpy())
        assert np.array_equal(yt[2], y.cpu().numpy())
        for l in range(3):
            orc = oracle_layer(w, l)
            ref = orc.tokens(xt[l])
            assert np.array_equal(it[l], ref["idx"]), l
            assert_close(yt[l], ref["y"], what=f"y layer {l}")
            if l + 1 < 3:
                assert_close(xt[l + 1], oracle.renorm(yt[l]), rel_l2=1e-6, max_abs_frac=1e-6, what="renorm")
    finally:
        moe.moe_destroy(ctx)


def test_streaming_pool_trace_and_placement_invariance():
    """A pool of 4 slots for 16 experts: the pool events equal the oracle pool
    simulator replayed on the GPU's routing, and every output is bitwise equal
    to the all-resident context's (an expert's answer does not depend on
    whether it came from the pool or was just fetched from the host store)."""
    w = TINY
    B, steps = 2, 12
    res = _ctx(w, max_batch=B)
    st = _ctx(w, max_batch=B, pool_slots=4)
    sim = oracle.PoolSim(4, w.n_experts)
    try:
        for step in range(steps):
            x = synth.tokens(w.seed, 100 + step, B, w.hidden)
            y0, i0, w0 = _decode(res, w, x)
            y1, i1, w1 = _decode(st, w, x)
            assert np.array_equal(i0, i1) and np.array_equal(y0, y1) and np.array_equal(w0, w1)
            want = sim.request(i1.reshape(-1))
            tr = moe.moe_pool_trace(st)
            got = [tuple(r[2:]) for r in tr if r[0] == step]
            assert got == want, step
        s = moe.moe_pool_stats(st, 0)
        tr = moe.moe_pool_trace(st)
        assert s["hits"] == int((tr[:, 3] == 0).sum()) and s["misses"] == int((tr[:, 3] == 1).sum())
        assert s["h2d_bytes"] == s["misses"] * moe.moe_blob_stride(w.hidden, w.inter, w.bits)
        assert s["resident"] == 4 and s["calls"] == steps and s["evictions"] > 0
        rs = moe.moe_pool_stats(res, 0)
        assert rs["resident"] == w.n_experts and rs["misses"] == 0 and rs["hits"] == s["hits"] + s["misses"]
    finally:
        moe.moe_destroy(res)
        moe.moe_destroy(st)


@pytest.mark.parametrize("B,L,max_batch,slots", [(3, 2, 3, 6), (1, 4, 1, 6), (2, 3, 8, 6), (5, 2, 8, 12)])
def test_streaming_stack_matches_resident_stack(B, L, max_batch, slots):
    """Whole-stack calls of a streaming context equal the resident context's
    bitwise: up to 3 tokens (pool >= B * top_k slots) through one persistent
    launch per call that waits at layers with a miss, more through the
    per-layer kernels.  The pool events of every (call, layer) equal the
    oracle simulator fed the resident context's routing."""
    w = dataclasses.replace(TINY, n_layers=L)
    res = _ctx(w, max_batch=max_batch)
    st = _ctx(w, max_batch=max_batch, pool_slots=slots, policy=moe.MOE_EVICT_LRU)
    sims = [oracle.PoolSim(slots, w.n_experts, moe.MOE_EVICT_LRU) for _ in range(L)]
    one_launch = B <= 3
    try:
        idx_tr = torch.empty((L, B, w.top_k), dtype=torch.int32, device="cuda")
        for step in range(6):
            x = torch.from_numpy(synth.tokens(w.seed, 7 + step, B, w.hidden)).cuda()
            ya, yb = torch.empty_like(x), torch.empty_like(x)
            moe.moe_forward_decode_stack(res, 0, L, x, B, ya, 1e-6, None, idx_tr, None)
            n0 = moe.moe_launch_count(st)
            moe.moe_forward_decode_stack(st, 0, L, x, B, yb)
            torch.cuda.synchronize()
            assert torch.equal(ya, yb), step
            if one_launch:
                assert moe.moe_launch_count(st) - n0 == 1, step
            tr = moe.moe_pool_trace(st)
            for l in range(L):
                want = sims[l].request(idx_tr[l].cpu().numpy().reshape(-1))
                got = [tuple(int(v) for v in r[2:]) for r in tr if r[0] == step and r[1] == l]
                assert got == want, (step, l)
        s = moe.moe_pool_stats(st)
        assert s["misses"] > 0 and s["calls"] == 6 * L
        assert s["h2d_bytes"] == s["misses"] * moe.moe_blob_stride(w.hidden, w.inter, w.bits)
        if not one_launch:
            assert s["h2d_ms"] > 0.0  # the per-layer path's copies are timed by events
        # a call over the upper layers only
        x = torch.from_numpy(synth.tokens(w.seed, 99, B, w.hidden)).cuda()
        ya, yb = torch.empty_like(x), torch.empty_like(x)
        moe.moe_forward_decode_stack(res, 1, L - 1, x, B, ya)
        moe.moe_forward_decode_stack(st, 1, L - 1, x, B, yb)
        torch.cuda.synchronize()
        assert torch.equal(ya, yb)
    finally:
        moe.moe_destroy(res)
        moe.moe_destroy(st)


@pytest.mark.parametrize("slots,policy,aging", [(8, 0, 0), (5, 1, 0), (6, 2, 0), (4, 3, 3)])
def test_pool_reset_size_and_policy_replay_oracle(slots, policy, aging):
    """moe_pool_reset re-sizes and re-polices a loaded streaming context: after
    a first run under LFU + recency on all 8 reserved slots, the reset starts
    every layer cold; then, over whole-stack calls (the graph path), the pool
    events of each (call, layer) equal the oracle simulator under the new
    size, policy and aging period fed the routing of an all-resident context,
    and every output is bitwise the resident context's."""
    w = dataclasses.replace(TINY, n_layers=2, zipf_s=1.1)
    B, L, k = 2, 2, TINY.top_k
    res = _ctx(w, max_batch=B)
    st = _ctx(w, max_batch=B, pool_slots=8)
    try:
        def step(s, ctx, idx_tr=None):
            x = torch.from_numpy(synth.tokens(w.seed, 300 + s, B, w.hidden)).cuda()
            y = torch.empty_like(x)
            moe.moe_forward_decode_stack(ctx, 0, L, x, B, y, 1e-6, None, idx_tr, None)
            return y

        for s in range(5):
            step(s, st)
        moe.moe_pool_reset(st, slots, policy, aging)
        z = moe.moe_pool_stats(st)
        assert (z["hits"], z["misses"], z["calls"], z["resident"]) == (0, 0, 0, 0)
        assert len(moe.moe_pool_trace(st)) == 0
        sims = [oracle.PoolSim(slots, w.n_experts, policy, aging_period=aging if aging > 0 else 64)
                for _ in range(L)]
        idx_tr = torch.empty((L, B, k), dtype=torch.int32, device="cuda")
        routes = []
        for s in range(16):
            ya = step(s, res, idx_tr)
            yb = step(s, st)
            torch.cuda.synchronize()
            assert torch.equal(ya, yb), s
            routes.append(idx_tr.cpu().numpy().copy())
        tr = moe.moe_pool_trace(st)
        tr = tr[np.lexsort((tr[:, 1], tr[:, 0]))]
        pos = 0
        for s in range(16):
            for l in range(L):
                want = sims[l].request(routes[s][l].reshape(-1))
                rows = tr[pos:pos + len(want)]
                assert all(int(r[0]) == s and int(r[1]) == l for r in rows), (s, l)
                assert [tuple(int(v) for v in r[2:]) for r in rows] == want, (s, l)
                pos += len(want)
        assert pos == len(tr)
        st1 = moe.moe_pool_stats(st)
        assert st1["misses"] > 0 and st1["resident"] <= L * slots and st1["calls"] == 16 * L
    finally:
        moe.moe_destroy(res)
        moe.moe_destroy(st)


@pytest.mark.parametrize("flags,B", [(0, 1), (moe.MOE_STORE_DIRECT, 2), (0, 5)])
def test_streaming_from_expert_container_equals_pinned_store(tmp_path, flags, B):
    """Misses read from the expert container (one positioned read per blob
    into the staging ring, then the copy) give the pinned store's outputs and
    pool trace exactly; the container's bytes are the packer's."""
    w = dataclasses.replace(TINY, n_layers=3, zipf_s=1.1)
    path = tmp_path / "experts.bin"
    workload.write_store(w, path)
    a = _ctx(w, max_batch=8, pool_slots=10)
    b = _ctx(w, max_batch=8, pool_slots=10, store_path=path, store_flags=flags)
    try:
        for step in range(8):
            x = torch.from_numpy(synth.tokens(w.seed, 400 + step, B, w.hidden)).cuda()
            ya, yb = torch.empty_like(x), torch.empty_like(x)
            moe.moe_forward_decode_stack(a, 0, w.n_layers, x, B, ya)
            moe.moe_forward_decode_stack(b, 0, w.n_layers, x, B, yb)
            torch.cuda.synchronize()
            assert torch.equal(ya, yb), step
        assert np.array_equal(moe.moe_pool_trace(a), moe.moe_pool_trace(b))
        sa, sb = moe.moe_pool_stats(a), moe.moe_pool_stats(b)
        assert sb["misses"] == sa["misses"] > 0 and sb["h2d_bytes"] == sa["h2d_bytes"]
        with pytest.raises(moe.MoeError) as e:  # the container holds the routed blobs
            blobs, shared, wr, wsg, beta = workload.layer_blobs(w, 0)
            moe.moe_load_experts(b, 0, blobs, moe.moe_blob_stride(w.hidden, w.inter, w.bits), shared, wr, wsg, beta)
        assert e.value.code == moe.MOE_EINVAL
    finally:
        moe.moe_destroy(a)
        moe.moe_destroy(b)
    bad = tmp_path / "other.bin"
    moe.moe_store_create(bad, w.n_layers, w.n_experts, w.hidden, w.inter, 8)  # int8 container for an int4 config
    with pytest.raises(moe.MoeError) as e:
        moe.moe_create(workload.config_for(w, pool_slots=10, store_path=bad))
    assert e.value.code == moe.MOE_EIO


def test_pool_reset_errors():
    w = TINY
    st = _ctx(w, max_batch=1, pool_slots=6)
    res = _ctx(w, max_batch=1)
    try:
        for args in ((7, 0, 0), (w.top_k - 1, 0, 0), (6, 4, 0), (6, -1, 0)):
            with pytest.raises(moe.MoeError) as e:
                moe.moe_pool_reset(st, *args)
            assert e.value.code == moe.MOE_EINVAL, args
        with pytest.raises(moe.MoeError) as e:
            moe.moe_pool_reset(res, 6, 0, 0)
        assert e.value.code == moe.MOE_ESTATE
        moe.moe_pool_reset(st, 6, moe.MOE_EVICT_LFU_AGED, 0)  # still usable after refused resets
    finally:
        moe.moe_destroy(st)
        moe.moe_destroy(res)


def test_router_bias_updates_all_layers_at_once():
    """moe_set_router_bias_all equals one moe_set_router_bias per layer (the
    staged copies run in stream order), on a streaming and on a resident
    context; a context with a layer not yet loaded refuses it."""
    w = dataclasses.replace(TINY, n_layers=3, zipf_s=1.1)
    B = 2
    a = _ctx(w, max_batch=B, pool_slots=5)
    b = _ctx(w, max_batch=B, pool_slots=5)
    r = _ctx(w, max_batch=B)
    rng = np.random.default_rng(41)
    try:
        for step in range(6):
            bias = (rng.standard_normal((w.n_layers, w.n_experts)) * 2.0).astype(np.float32)
            for l in range(w.n_layers):
                moe.moe_set_router_bias(a, l, np.ascontiguousarray(bias[l]))
            moe.moe_set_router_bias_all(b, bias)
            moe.moe_set_router_bias_all(r, bias)
            bias[:] = 0.0  # the host buffer may be reused at once
            x = torch.from_numpy(synth.tokens(w.seed, 50 + step, B, w.hidden)).cuda()
            ya, yb, yr = torch.empty_like(x), torch.empty_like(x), torch.empty_like(x)
            moe.moe_forward_decode_stack(a, 0, w.n_layers, x, B, ya)
            moe.moe_forward_decode_stack(b, 0, w.n_layers, x, B, yb)
            moe.moe_forward_decode_stack(r, 0, w.n_layers, x, B, yr)
            torch.cuda.synchronize()
            assert torch.equal(ya, yb) and torch.equal(ya, yr)
        assert np.array_equal(moe.moe_pool_trace(a), moe.moe_pool_trace(b))
    finally:
        for c in (a, b, r):
            moe.moe_destroy(c)
    part = workload.create_loaded(w, max_batch=B, layers=[0])
    try:
        with pytest.raises(moe.MoeError) as e:
            moe.moe_set_router_bias_all(part, np.zeros((w.n_layers, w.n_experts), np.float32))
        assert e.value.code == moe.MOE_ESTATE
    finally:
        moe.moe_destroy(part)


def test_decode_argument_errors():
    w = dataclasses.replace(TINY, n_layers=2)
    ctx = workload.create_loaded(w, max_batch=2, layers=[0])
    try:
        x = torch.zeros((2, w.hidden), device="cuda")
        y = torch.zeros_like(x)
        for args, code in [((0, x, 0, y), moe.MOE_EINVAL), ((0, x, 3, y), moe.MOE_EINVAL),
                           ((5, x, 1, y), moe.MOE_EINVAL), ((1, x, 1, y), moe.MOE_ESTATE),
                           ((0, x, 1, x), moe.MOE_EINVAL)]:
            with pytest.raises(moe.MoeError) as e:
                moe.moe_forward_decode(ctx, *args)
            assert e.value.code == code, args
        moe.moe_forward_decode(ctx, 0, x, 2, y)  # still usable
        torch.cuda.synchronize()
    finally:
        moe.moe_destroy(ctx)


def test_injected_faults_fail_cleanly():
    w = TINY
    with pytest.raises(moe.MoeError) as e:
        workload.create_loaded(w, pool_slots=4, fault_flags=moe.MOE_FAULT_PINNED_ALLOC)
    assert e.value.code == moe.MOE_ENOMEM
    x = torch.from_numpy(synth.tokens(w.seed, 0, 1, w.hidden)).cuda()
    y = torch.empty_like(x)
    ctx = workload.create_loaded(w, pool_slots=4, fault_flags=moe.MOE_FAULT_WAIT_TIMEOUT)
    try:
        with pytest.raises(moe.MoeError) as e:
            moe.moe_forward_decode(ctx, 0, x, 1, y)
        assert e.value.code == moe.MOE_ETIMEOUT
        moe.moe_forward_decode(ctx, 0, x, 1, y)  # the timeout is not sticky
        torch.cuda.synchronize()
    finally:
        moe.moe_destroy(ctx)
    ctx = workload.create_loaded(w, pool_slots=4, fault_flags=moe.MOE_FAULT_MISS_COPY, fault_arg=1)
    try:
        with pytest.raises(moe.MoeError) as e:
            moe.moe_forward_decode(ctx, 0, x, 1, y)
        assert e.value.code == moe.MOE_ECUDA
        with pytest.raises(moe.MoeError) as e:
            moe.moe_forward_decode(ctx, 0, x, 1, y)
        assert e.value.code == moe.MOE_ESTATE  # poisoned
    finally:
        moe.moe_destroy(ctx)


def test_streaming_stack_abandoned_by_a_failed_copy_ends_cleanly():
    """The host's service of a missed expert fails (injected) while the
    persistent kernel runs the layer: the call returns MOE_ECUDA, the host
    marks the layer abandoned, the kernel sees it when it asks for the slots
    and ends at once (the stream synchronises well before any device-side wait
    could run out), and the context is poisoned."""
    import time
    w = dataclasses.replace(TINY, n_layers=3)
    x = torch.from_numpy(synth.tokens(w.seed, 5, 1, w.hidden)).cuda()
    y = torch.empty_like(x)
    ctx = _ctx(w, max_batch=1, pool_slots=6, fault_flags=moe.MOE_FAULT_MISS_COPY, fault_arg=1)
    try:
        n0 = moe.moe_launch_count(ctx)
        t0 = time.perf_counter()
        with pytest.raises(moe.MoeError) as e:
            moe.moe_forward_decode_stack(ctx, 0, 3, x, 1, y)
        assert e.value.code == moe.MOE_ECUDA
        torch.cuda.synchronize()
        assert time.perf_counter() - t0 < 0.5
        assert moe.moe_launch_count(ctx) - n0 == 1  # it was the persistent kernel
        with pytest.raises(moe.MoeError) as e:
            moe.moe_forward_decode_stack(ctx, 0, 3, x, 1, y)
        assert e.value.code == moe.MOE_ESTATE
    finally:
        moe.moe_destroy(ctx)
    torch.cuda.synchronize()


def test_device_wait_runs_out_and_reports_timeout():
    """MOE_FAULT_DEVICE_WAIT: in the next multi-layer persistent launch one CTA
    withholds its outputs of the first layer and every device-side wait is
    bounded by 1 ms.  The other CTAs' waits run out, the kernel ends normally
    (no GPU fault: the stream synchronises cleanly), the next call reports
    MOE_ETIMEOUT and poisons the context; a fresh context then runs clean."""
    w = dataclasses.replace(TINY, n_layers=3)
    x = torch.from_numpy(synth.tokens(w.seed, 11, 1, w.hidden)).cuda()
    y = torch.empty_like(x)
    ctx = _ctx(w, max_batch=1, fault_flags=moe.MOE_FAULT_DEVICE_WAIT)
    try:
        moe.moe_forward_decode_stack(ctx, 0, 3, x, 1, y)  # asynchronous: the launch itself succeeds
        torch.cuda.synchronize()
        with pytest.raises(moe.MoeError) as e:
            moe.moe_forward_decode_stack(ctx, 0, 3, x, 1, y)
        assert e.value.code == moe.MOE_ETIMEOUT
        with pytest.raises(moe.MoeError) as e:
            moe.moe_forward_decode(ctx, 0, x, 1, y)
        assert e.value.code == moe.MOE_ESTATE  # poisoned
    finally:
        moe.moe_destroy(ctx)
    torch.cuda.synchronize()
    fresh = _ctx(w, max_batch=1)
    try:
        xt = torch.empty((3, 1, w.hidden), device="cuda")
        yt = torch.empty((3, 1, w.hidden), device="cuda")
        it = torch.empty((3, 1, w.top_k), dtype=torch.int32, device="cuda")
        for _ in range(2):
            moe.moe_forward_decode_stack(fresh, 0, 3, x, 1, y, 1e-6, xt, it, yt)
        torch.cuda.synchronize()
        for l in range(3):
            ref = oracle_layer(w, l).tokens(xt[l].cpu().numpy())
            assert np.array_equal(it[l].cpu().numpy(), ref["idx"])
            assert_close(yt[l].cpu().numpy(), ref["y"], what=f"layer {l}")
    finally:
        moe.moe_destroy(fresh)


@pytest.mark.parametrize("B,bits", [(1, 4), (2, 4), (3, 4), (5, 4), (1, 8), (3, 8), (12, 4)])
def test_stack_kernel_equals_per_layer_kernels(B, bits):
    """The persistent stack kernel (B <= 3, all resident) and the batched
    per-layer kernels share one arithmetic: every layer's routing and output
    agree bit for bit; and each layer matches the oracle fed the GPU's own
    layer input (larger B: the per-layer path on both sides)."""
    w = dataclasses.replace(TINY, n_layers=3, bits=bits)
    L = w.n_layers
    ctx = _ctx(w, max_batch=B)
    try:
        x = torch.from_numpy(synth.tokens(w.seed, 3, B, w.hidden)).cuda()
        y = torch.empty_like(x)
        xt = torch.empty((L, B, w.hidden), device="cuda")
        yt = torch.empty((L, B, w.hidden), device="cuda")
        it = torch.empty((L, B, w.top_k), dtype=torch.int32, device="cuda")
        n0 = moe.moe_launch_count(ctx)
        moe.moe_forward_decode_stack(ctx, 0, L, x, B, y, 1e-6, xt, it, yt, torch.cuda.current_stream())
        torch.cuda.synchronize()
        launches = moe.moe_launch_count(ctx) - n0
        assert launches == (1 if B <= 3 else 6 * L + L - 1)
        for l in range(L):
            yl = torch.empty_like(x)
            il = torch.empty((B, w.top_k), dtype=torch.int32, device="cuda")
            moe.moe_forward_decode(ctx, l, xt[l].contiguous(), B, yl, il)
            torch.cuda.synchronize()
            assert torch.equal(il, it[l]), l
            assert torch.equal(yl, yt[l]), l
            ref = oracle_layer(w, l).tokens(xt[l].cpu().numpy())
            assert np.array_equal(it[l].cpu().numpy(), ref["idx"])
            assert_close(yt[l].cpu().numpy(), ref["y"], what=f"layer {l}")
        assert torch.equal(y, yt[L - 1])
    finally:
        moe.moe_destroy(ctx)


def test_stack_kernel_wider_shapes():
    """Hidden 512, 64 experts top-10, intermediate 192 and shared 64 (ragged
    chunk counts), Zipf router bias, 4 layers, B = 3."""
    w = dataclasses.replace(TINY, n_layers=4, n_experts=64, top_k=10, hidden=512, inter=192, shared_inter=64,
                            router_sigma=1.0 / np.sqrt(512), zipf_s=1.1)
    B, L = 3, 4
    ctx = _ctx(w, max_batch=B)
    try:
        x = torch.from_numpy(synth.tokens(w.seed, 0, B, w.hidden)).cuda()
        y = torch.empty_like(x)
        xt = torch.empty((L, B, w.hidden), device="cuda")
        yt = torch.empty((L, B, w.hidden), device="cuda")
        it = torch.empty((L, B, w.top_k), dtype=torch.int32, device="cuda")
        moe.moe_forward_decode_stack(ctx, 0, L, x, B, y, 1e-6, xt, it, yt)
        torch.cuda.synchronize()
        for l in range(L):
            ref = oracle_layer(w, l).tokens(xt[l].cpu().numpy())
            assert np.array_equal(it[l].cpu().numpy(), ref["idx"]), l
            assert_close(yt[l].cpu().numpy(), ref["y"], what=f"layer {l}")
            if l + 1 < L:
                assert_close(xt[l + 1].cpu().numpy(), oracle.renorm(yt[l].cpu().numpy()), rel_l2=1e-6,
                             max_abs_frac=1e-6, what="renorm")
    finally:
        moe.moe_destroy(ctx)


def test_stack_repeated_launches_are_deterministic():
    """The barrier counters reset at the end of every launch: 50 launches in a
    row give identical results and no device-side wait runs out."""
    w = dataclasses.replace(TINY, n_layers=2)
    ctx = _ctx(w, max_batch=2)
    try:
        x = torch.from_numpy(synth.tokens(w.seed, 9, 2, w.hidden)).cuda()
        y0 = torch.empty_like(x)
        moe.moe_forward_decode_stack(ctx, 0, 2, x, 2, y0)
        y = torch.empty_like(x)
        for _ in range(50):
            moe.moe_forward_decode_stack(ctx, 0, 2, x, 2, y)
        torch.cuda.synchronize()
        assert torch.equal(y, y0)
        moe.moe_forward_decode_stack(ctx, 0, 2, x, 2, y)  # would raise MOE_ETIMEOUT after a timed-out launch
        torch.cuda.synchronize()
    finally:
        moe.moe_destroy(ctx)
