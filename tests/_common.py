"""Shared helpers of the tests: tolerances, oracle layers built from the
generator, and the router-gap seed search of the tiny workload."""
from __future__ import annotations

import dataclasses

import numpy as np

import oracle
import synth

# Tolerances on floating-point layer outputs (the decode definition is fp64,
# the kernels accumulate in fp32): relative L2 and max-abs against max|y|.
REL_L2 = 1e-4
MAX_ABS_FRAC = 1e-3


def assert_close(got, ref, rel_l2=REL_L2, max_abs_frac=MAX_ABS_FRAC, what="y"):
    got = np.asarray(got, np.float64)
    ref = np.asarray(ref, np.float64)
    assert got.shape == ref.shape, (got.shape, ref.shape)
    assert np.all(np.isfinite(got)), f"{what}: non-finite values"
    nr = np.linalg.norm(ref)
    rel = np.linalg.norm(got - ref) / (nr if nr > 0 else 1.0)
    mx = np.abs(got - ref).max() if got.size else 0.0
    lim = max_abs_frac * (np.abs(ref).max() if ref.size else 0.0)
    assert rel <= rel_l2 and mx <= lim, f"{what}: rel-L2 {rel:.3e} (<= {rel_l2}), max-abs {mx:.3e} (<= {lim:.3e})"
    return rel, mx


def oracle_layer(w: synth.Workload, layer: int, experts=None, bits=None, norm_topk=True):
    """oracle.Layer for one layer of workload w holding the given experts
    (default: all), drawn from the same generator streams as the GPU side."""
    bits = bits or w.bits
    ids = range(w.n_experts) if experts is None else sorted(set(int(e) for e in experts))
    ex = {e: synth.expert(w.seed, layer, e, w.hidden, w.inter, bits, w.sigma) for e in ids}
    shared = synth.expert(w.seed, layer, synth.SHARED, w.hidden, w.shared_inter, bits, w.sigma) \
        if w.shared_inter else None
    wr, wsg, beta = synth.layer_inputs(w, layer)
    return oracle.Layer(w.hidden, w.n_experts, w.top_k, w.inter, w.shared_inter, wr, wsg, ex, shared=shared,
                        router_bias=beta, norm_topk=norm_topk)


def topk_gap(logits: np.ndarray, k: int) -> float:
    s = np.sort(np.asarray(logits, np.float64))[::-1]
    return float(s[k - 1] - s[k]) if k < s.shape[0] else float("inf")


def seed_with_gap(w: synth.Workload, n_tokens: int, gap: float = 1e-3, layer: int = 0, max_tries: int = 200):
    """First seed from w.seed upward whose router logits (oracle, tokens of
    step 0) keep >= gap between the k-th and (k+1)-th expert of every token."""
    for s in range(w.seed, w.seed + max_tries):
        ws = dataclasses.replace(w, seed=s)
        wr, _, beta = synth.layer_inputs(ws, layer)
        x = synth.tokens(s, 0, n_tokens, w.hidden)
        if all(topk_gap(oracle.router_logits(wr, x[t], beta), w.top_k) >= gap for t in range(n_tokens)):
            return ws
    raise RuntimeError("no seed with the requested router gap")
