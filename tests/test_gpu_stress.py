"""The streaming stress workload at full size: the 48-layer 80B-shaped stack,
128 of 512 slots per layer in HBM, the store in pinned host memory, Zipf
routing with drift, a cold pool.

Every pool event (hit / miss, slot, evicted expert) of every layer and step
must equal the oracle pool simulator replayed on the GPU's routing; on
sampled steps every layer's chosen experts must equal the oracle router fed
the GPU's layer input (with that step's drifted bias), and the layer output
must be within the layer tolerance."""
import concurrent.futures as cf
import dataclasses

import numpy as np
import pytest

import oracle
import synth
from _common import assert_close

torch = pytest.importorskip("torch")
pytestmark = [pytest.mark.gpu,
              pytest.mark.skipif(not torch.cuda.is_available(), reason="needs a CUDA GPU")]

import int4_expert_streaming_gb300 as moe  # noqa: E402
from int4_expert_streaming_gb300 import workload  # noqa: E402


@pytest.fixture(scope="module", autouse=True)
def _built():
    moe.build()
    moe.load_library()


def _oracle_layer(w, layer, bits, bias, experts):
    wr, wsg, _ = synth.layer_inputs(w, layer)
    ex = {int(e): synth.expert(w.seed, layer, int(e), w.hidden, w.inter, bits, w.sigma) for e in experts}
    shared = synth.expert(w.seed, layer, synth.SHARED, w.hidden, w.shared_inter, bits, w.sigma)
    return oracle.Layer(w.hidden, w.n_experts, w.top_k, w.inter, w.shared_inter, wr, wsg, ex, shared=shared,
                        router_bias=bias)


@pytest.mark.parametrize("bits,steps", [(4, 1024), (8, 128)])
def test_stress_pool_trace_and_sampled_layers(bits, steps):
    w = dataclasses.replace(synth.CONFIGS["stress"], bits=bits)
    L, H, k = w.n_layers, w.hidden, w.top_k
    ctx = workload.create_loaded(w, bits, max_batch=1)
    try:
        drift = workload.Drift(w)
        st = torch.cuda.current_stream()
        rng = np.random.default_rng(31)
        sampled = set(range(4)) | set(int(s) for s in rng.choice(np.arange(4, steps), 4, replace=False))
        y = torch.empty((1, H), device="cuda")
        idx_tr = torch.empty((L, 1, k), dtype=torch.int32, device="cuda")
        x_tr = torch.empty((L, 1, H), device="cuda")
        y_tr = torch.empty((L, 1, H), device="cuda")
        routes, checks = [], []
        for s in range(steps):
            if s > 0:
                drift.advance(ctx, st)
            x = torch.from_numpy(synth.tokens(w.seed, s, 1, H)).cuda()
            if s in sampled:
                biases = [drift.bias(l) for l in range(L)]
                moe.moe_forward_decode_stack(ctx, 0, L, x, 1, y, 1e-6, x_tr, idx_tr, y_tr, st)
                torch.cuda.synchronize()
                checks.append((s, biases, x_tr.cpu().numpy()[:, 0], idx_tr.cpu().numpy()[:, 0], y_tr.cpu().numpy()[:, 0]))
            else:
                moe.moe_forward_decode_stack(ctx, 0, L, x, 1, y, 1e-6, None, idx_tr, None, st)
            routes.append(idx_tr.cpu().numpy()[:, 0].copy())
        # pool events of every (step, layer) against the oracle simulator
        tr = moe.moe_pool_trace(ctx)
        sims = [oracle.PoolSim(w.pool_slots, w.n_experts) for _ in range(L)]
        order = np.lexsort((tr[:, 1], tr[:, 0]))  # by call number, then layer (stable within a call)
        tr = tr[order]
        pos = 0
        for s in range(steps):
            for l in range(L):
                want = sims[l].request(routes[s][l])
                got = [tuple(int(v) for v in r[2:]) for r in tr[pos:pos + len(want)]]
                assert all(int(r[0]) == s and int(r[1]) == l for r in tr[pos:pos + len(want)]), (s, l)
                assert got == want, (s, l)
                pos += len(want)
        assert pos == len(tr)
        stats = moe.moe_pool_stats(ctx)
        assert stats["misses"] == int((tr[:, 3] == 1).sum()) and stats["hits"] == int((tr[:, 3] == 0).sum())
        assert stats["h2d_bytes"] == stats["misses"] * moe.moe_blob_stride(H, w.inter, bits)
        distinct = [len(np.unique(np.concatenate([routes[s][l] for s in range(steps)]))) for l in range(L)]
        assert stats["resident"] == sum(min(w.pool_slots, d) for d in distinct)
        assert stats["evictions"] == int(((tr[:, 3] == 1) & (tr[:, 5] >= 0)).sum())

        # sampled steps: every layer against the oracle fed the GPU's layer input
        def one(item):
            s, biases, xs, idxs, ys, l = item
            lay = _oracle_layer(w, l, bits, biases[l], idxs[l])
            ref = lay.token(xs[l])
            return s, l, ref, idxs[l], ys[l]

        items = [(s, b, xs, ids, ys, l) for (s, b, xs, ids, ys) in checks for l in range(L)]
        with cf.ThreadPoolExecutor(16) as ex:
            for s, l, ref, idx, yg in ex.map(one, items):
                assert np.array_equal(idx, ref["idx"]), (s, l)
                assert_close(yg, ref["y"], what=f"y step {s} layer {l}")
    finally:
        moe.moe_destroy(ctx)
