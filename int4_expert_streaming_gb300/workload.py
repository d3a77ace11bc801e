"""Load the seeded synthetic workloads (package ``synth``) into a context
through the C ABI: draw and quantise each expert, pack it with
``moe_pack_expert`` and hand whole layers to ``moe_load_experts``."""
from __future__ import annotations

import concurrent.futures as cf
import os

import numpy as np

import synth

from . import (make_config, moe_blob_stride, moe_create, moe_load_experts, moe_pack_expert, moe_store_create,
               moe_store_write_layer)


def _threads(n=None):
    return n or max(1, os.cpu_count() or 1)


def layer_blobs(w: "synth.Workload", layer: int, bits: int | None = None, threads: int | None = None,
                out: np.ndarray | None = None, routed: bool = True):
    """Packed routed blobs [E*stride] (uint8; None when routed is False), the
    shared blob, router weights (bf16 bits), shared-gate weights (bf16 bits)
    and router bias (fp32 or None)."""
    bits = bits or w.bits
    stride = moe_blob_stride(w.hidden, w.inter, bits)
    E = w.n_experts
    blobs = None
    if routed:
        blobs = out if out is not None else np.empty(E * stride, np.uint8)
        assert blobs.nbytes >= E * stride

        def one(e):
            d = synth.expert(w.seed, layer, e, w.hidden, w.inter, bits, w.sigma)
            moe_pack_expert(w.hidden, w.inter, bits, d, out=blobs[e * stride:(e + 1) * stride])

        with cf.ThreadPoolExecutor(_threads(threads)) as ex:
            list(ex.map(one, range(E)))
        blobs = blobs[:E * stride]
    shared = None
    if w.shared_inter > 0:
        shared = moe_pack_expert(w.hidden, w.shared_inter, bits,
                                 synth.expert(w.seed, layer, synth.SHARED, w.hidden, w.shared_inter, bits, w.sigma))
    wr, wsg, beta = synth.layer_inputs(w, layer)
    return blobs, shared, wr, wsg, beta


def config_for(w: "synth.Workload", bits: int | None = None, max_batch: int = 1, max_tokens: int = 0,
               pool_slots: int | None = None, n_layers: int | None = None, **kw):
    return make_config(n_layers or w.n_layers, w.hidden, w.n_experts, w.top_k, w.inter, w.shared_inter,
                       bits=bits or w.bits,
                       pool_slots=pool_slots if pool_slots is not None else (w.pool_slots or w.n_experts),
                       max_batch=max_batch, max_tokens=max_tokens, **kw)


def create_loaded(w: "synth.Workload", bits: int | None = None, max_batch: int = 1, max_tokens: int = 0,
                  pool_slots: int | None = None, layers=None, threads: int | None = None, **kw):
    """Create a context for workload w and load every layer (or `layers`).
    With store_path=... (an expert container written by write_store) the
    routed blobs stay on disk and only the dense parts are loaded."""
    bits = bits or w.bits
    cfg = config_for(w, bits, max_batch, max_tokens, pool_slots, **kw)
    from_file = cfg.store_path is not None
    lbits = kw.get("layer_bits") or [bits] * cfg.n_layers  # layer_bits=[...]: a mixed store
    ctx = moe_create(cfg)
    strides = [moe_blob_stride(w.hidden, w.inter, b) for b in lbits]
    buf = None if from_file else np.empty(w.n_experts * max(strides), np.uint8)
    for layer in (range(cfg.n_layers) if layers is None else layers):
        blobs, shared, wr, wsg, beta = layer_blobs(w, layer, lbits[layer], threads, out=buf, routed=not from_file)
        moe_load_experts(ctx, layer, blobs, strides[layer], shared, wr, wsg if shared is not None else None, beta)
    return ctx


def write_store(w: "synth.Workload", path, bits: int | None = None, n_layers: int | None = None,
                threads: int | None = None) -> None:
    """Write the routed blobs of the workload's layers into an expert container."""
    bits = bits or w.bits
    L = n_layers or w.n_layers
    moe_store_create(path, L, w.n_experts, w.hidden, w.inter, bits)
    stride = moe_blob_stride(w.hidden, w.inter, bits)
    buf = np.empty(w.n_experts * stride, np.uint8)
    for layer in range(L):
        blobs, *_ = layer_blobs(w, layer, bits, threads, out=buf)
        moe_store_write_layer(path, layer, blobs, stride)


class Drift:
    """Temporally correlated popularity drift of a Zipf-biased workload.

    Each layer keeps the rank permutation its router bias is drawn from
    (beta_e = ln p(rank(e)), p(r) ~ r^-s).  Before decode step s >= 1,
    ``advance`` applies the workload's adjacent-rank swaps of step s to every
    layer and sends the new bias to the context with moe_set_router_bias;
    step 0 runs with the bias the layer was loaded with.  ``bias(layer)``
    gives the current bias, so a checker can rebuild the router of any step.
    """

    def __init__(self, w: "synth.Workload"):
        self.w = w
        self.perm = [synth.rank_permutation(w.seed, l, w.n_experts) for l in range(w.n_layers)]
        self.step = 0

    def bias(self, layer: int) -> np.ndarray:
        return synth.zipf_bias(self.perm[layer], self.w.zipf_s)

    def biases(self) -> np.ndarray:
        """The current bias of every layer, fp32 [n_layers, n_experts]."""
        return np.stack([self.bias(l) for l in range(self.w.n_layers)]).astype(np.float32)

    def advance(self, ctx=None, stream=None) -> None:
        from . import moe_set_router_bias
        self.step += 1
        for l in range(self.w.n_layers):
            synth.drift_step(self.w.seed, l, self.step, self.perm[l], self.w.drift_swaps)
            if ctx is not None:
                moe_set_router_bias(ctx, l, self.bias(l), stream)

    def schedule(self, n_steps: int) -> np.ndarray:
        """Advances n_steps times without a context and returns the biases of
        those steps, fp32 [n_steps, n_layers, n_experts] (inputs computed ahead,
        like the token batches; send step i with moe_set_router_bias_all)."""
        out = np.empty((n_steps, self.w.n_layers, self.w.n_experts), np.float32)
        for i in range(n_steps):
            self.advance()
            out[i] = self.biases()
        return out
