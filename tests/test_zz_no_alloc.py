"""moe_route_noalloc (routing with its scratch in a fixed device array) gives
the same experts and weights as the routing inside moe_forward_decode, on two
calls in a row, and rejects a request larger than its array."""
import math

import numpy as np
import pytest

import synth

torch = pytest.importorskip("torch")
pytestmark = [pytest.mark.gpu,
              pytest.mark.skipif(not torch.cuda.is_available(), reason="needs a CUDA GPU")]

import int4_expert_streaming_gb300 as moe  # noqa: E402
from int4_expert_streaming_gb300 import workload  # noqa: E402


@pytest.fixture(scope="module", autouse=True)
def _built():
    moe.build()
    moe.load_library()


def _decode_routing(ctx, w, x):
    B = x.shape[0]
    y = torch.empty_like(x)
    idx = torch.empty((B, w.top_k), dtype=torch.int32, device="cuda")
    wt = torch.empty((B, w.top_k), dtype=torch.float32, device="cuda")
    moe.moe_forward_decode(ctx, 0, x, B, y, idx, wt, torch.cuda.current_stream())
    return idx, wt


@pytest.mark.parametrize("name", ["tiny", "80b-prefill"])
def test_route_noalloc_matches_decode_two_calls(name):
    w = synth.CONFIGS[name]
    B = 8
    ctx = workload.create_loaded(w, max_batch=B)
    try:
        for step in (0, 1):  # two calls in a row, different tokens
            x = torch.from_numpy(synth.tokens(w.seed, 40 + step, B, w.hidden)).cuda()
            ref_i, ref_w = _decode_routing(ctx, w, x)
            got_i = torch.full((B, w.top_k), -1, dtype=torch.int32, device="cuda")
            got_w = torch.full((B, w.top_k), float("nan"), device="cuda")
            moe.moe_route_noalloc(ctx, 0, x, B, got_i, got_w, torch.cuda.current_stream())
            torch.cuda.synchronize()
            assert torch.equal(got_i, ref_i)
            assert torch.equal(got_w, ref_w)
    finally:
        moe.moe_destroy(ctx)


def test_route_noalloc_rejects_oversize():
    # 1024 experts x 64 tokens of logits alone exceed the fixed 256 KiB array
    w = synth.Workload("wide-router", n_layers=1, hidden=256, n_experts=1024, top_k=2, inter=64, shared_inter=64,
                       router_sigma=1.0 / math.sqrt(256))
    ctx = workload.create_loaded(w, max_batch=64)
    try:
        x = torch.zeros((64, w.hidden), device="cuda")
        i = torch.empty((64, w.top_k), dtype=torch.int32, device="cuda")
        wt = torch.empty((64, w.top_k), device="cuda")
        with pytest.raises(moe.MoeError) as e:
            moe.moe_route_noalloc(ctx, 0, x, 64, i, wt)
        assert e.value.code == moe.MOE_EINVAL
        moe.moe_route_noalloc(ctx, 0, x[:8], 8, i[:8], wt[:8])  # 8 tokens fit
        torch.cuda.synchronize()
        assert np.all((i[:8].cpu().numpy() >= 0) & (i[:8].cpu().numpy() < 1024))
    finally:
        moe.moe_destroy(ctx)
