"""Pins of the CPU oracle against facts that do not come from the oracle itself:
hand-derived examples, closed forms, textbook special cases, error bounds and
invariants.  CPU only."""
import math
import os
from collections import Counter, OrderedDict

import numpy as np
import pytest
import torch

import oracle
import synth

GOLDEN = os.path.join(os.path.dirname(__file__), "golden")


def f16(v):
    return int(np.array(v, np.float16).view(np.uint16))


def bf16(v):
    return int(torch.tensor([v], dtype=torch.float32).to(torch.bfloat16).view(torch.int16).item()) & 0xFFFF


# --------------------------------------------------------------------------
# number formats
# --------------------------------------------------------------------------

def test_half_to_double_all_patterns():
    """Every non-NaN fp16 pattern widens exactly (numpy's float16 is the reference)."""
    bits = np.arange(65536, dtype=np.uint16)
    ref = bits.view(np.float16).astype(np.float64)
    got = np.array([oracle.half_to_double(int(b)) for b in bits])
    ok = ~np.isnan(ref)
    assert np.array_equal(got[ok], ref[ok])
    assert np.all(np.isnan(got[~ok]))


def test_float_to_bf16_round_to_nearest_even():
    """bf16 rounding matches torch's RNE conversion, including exact ties."""
    rng = np.random.default_rng(0)
    vals = list(rng.standard_normal(2000).astype(np.float32))
    # exact ties between two bf16 neighbours: 1 + 2^-8 (tie, even -> 1), 1 + 3*2^-8 (tie, odd -> up)
    vals += [np.float32(1 + 2 ** -8), np.float32(1 + 3 * 2 ** -8), np.float32(-(1 + 2 ** -8)), np.float32(0.0)]
    for v in vals:
        assert oracle.float_to_bf16(float(v)) == bf16(float(v)), v


# --------------------------------------------------------------------------
# dequantisation and the blob packer
# --------------------------------------------------------------------------

@pytest.mark.parametrize("bits", [4, 8])
def test_pack_unpack_every_code_bit_exact(bits):
    """Brute force: every code value in every position survives pack -> unpack."""
    H, I = 64, 64
    n = 1 << bits
    rng = np.random.default_rng(bits)
    e = {}
    for name, (r, c) in {"gate": (I, H), "up": (I, H), "down": (H, I)}.items():
        q = (np.arange(r * c) % n).astype(np.uint8).reshape(r, c)
        e["q_" + name] = np.ascontiguousarray(rng.permutation(q.reshape(-1)).reshape(r, c))
        e["sb_" + name] = rng.integers(0, 0x7BFF, size=(r, c // 64, 2)).astype(np.uint16)
    blob = oracle.pack_blob(e, H, I, bits)
    assert blob.nbytes == oracle.blob_stride(H, I, bits)
    back = oracle.unpack_blob(blob, H, I, bits)
    for k in e:
        assert np.array_equal(back[k], e[k]), k


def test_blob_layout_low_nibble_first():
    """Byte-level layout: codes 1..8 in columns 0..7 of the first gate row give the
    word 0x87654321 (low nibble first, little-endian); sections follow in the
    order gate.q, up.q, down.q, gate.sb, up.sb, down.sb; padding is zero."""
    H, I = 64, 64
    e = {k: np.zeros((I, H) if k.endswith(("gate", "up")) else (H, I), np.uint8)
         for k in ("q_gate", "q_up", "q_down")}
    e.update({k: np.zeros((64, 1, 2), np.uint16) for k in ("sb_gate", "sb_up", "sb_down")})
    e["q_gate"][0, :8] = np.arange(1, 9)
    e["q_up"][0, 0] = 0xA
    e["q_down"][0, 1] = 0xB
    e["sb_gate"][0, 0] = (0x1234, 0x5678)
    e["sb_down"][63, 0] = (0x9ABC, 0xDEF0)
    blob = oracle.pack_blob(e, H, I, 4)
    assert bytes(blob[:4]) == bytes([0x21, 0x43, 0x65, 0x87])
    qbytes = H * I // 2
    assert blob[qbytes] == 0x0A                    # up.q starts right after gate.q
    assert blob[2 * qbytes] == 0xB0                # down.q: column 1 = high nibble of byte 0
    sb0 = 3 * qbytes
    assert bytes(blob[sb0:sb0 + 4]) == bytes([0x34, 0x12, 0x78, 0x56])   # scale low half, bias high half
    sb_down_last = sb0 + 2 * I * 4 + 63 * 4
    assert bytes(blob[sb_down_last:sb_down_last + 4]) == bytes([0xBC, 0x9A, 0xF0, 0xDE])
    total = oracle.blob_bytes(H, I, 4)
    assert total == 3 * qbytes + 3 * 64 * 4 and not blob[total:].any()


def test_blob_stride_sizes():
    """Stride arithmetic for the two shapes in use: 1 769 472 B (int4, H 2048,
    I 512, already a multiple of 4096) and 3 342 336 B (int8)."""
    assert oracle.blob_bytes(2048, 512, 4) == 1769472 == oracle.blob_stride(2048, 512, 4)
    assert oracle.blob_stride(2048, 512, 8) == 3342336
    assert oracle.blob_bytes(256, 128, 4) == 55296 and oracle.blob_stride(256, 128, 4) == 57344


@pytest.mark.parametrize("bits", [4, 8])
def test_dequant_exact_on_fp16_grid(bits):
    """w = scale*q + bias exactly, for every code and a grid of fp16 scale/bias
    patterns including negatives and subnormals (numpy float16 widening)."""
    scales = [0.0, 2 ** -24, 3 * 2 ** -24, 2 ** -14, 0.0078125, 0.013, 0.5, 1.0, 3.75, -0.25]
    biases = [0.0, -2 ** -24, -0.048, 0.02, -1.0, 7.5, -65504.0 / 4096]
    n = 1 << bits
    rows = len(scales) * len(biases)
    q = np.tile((np.arange(64) % n).astype(np.uint8), (rows, 1))
    sb = np.zeros((rows, 1, 2), np.uint16)
    ref = np.zeros((rows, 64))
    for i, (s, b) in enumerate((s, b) for s in scales for b in biases):
        sb[i, 0] = (f16(s), f16(b))
        s16, b16 = float(np.float16(s)), float(np.float16(b))
        ref[i] = [s16 * c + b16 for c in q[i]]
    assert np.array_equal(oracle.dequant(q, sb), ref)


# --------------------------------------------------------------------------
# router
# --------------------------------------------------------------------------

def test_router_unit_vector_gives_weight_column():
    """x = e_j makes every logit the bf16 weight W[e][j] plus its bias exactly."""
    E, H = 16, 256
    w = synth.router_weights(7, 0, E, H, 0.02)
    bias = np.linspace(-1, 1, E).astype(np.float32)
    for j in (0, 7, 8, 255):
        x = np.zeros(H, np.float32)
        x[j] = 1.0
        got = oracle.router_logits(w, x, bias)
        want = synth.bf16_to_f32(w[:, j]) + bias
        assert np.array_equal(got, want.astype(np.float32))


def test_router_fixed_summation_order():
    """The fp32 order is pinned by hand: partial sums by (h/8) mod 32, butterfly 16..1.
    1 + 2^-24 + 2^-24: with the two tiny terms in lanes 1 and 17 they meet first (offset
    16) and survive, giving 1 + 2^-23; in lanes 1 and 2 each meets 1 alone and is
    rounded away (ties to even), giving 1."""
    H = 256
    tiny = 2.0 ** -24
    w = np.zeros((2, H), np.uint16)
    w[:, 0] = bf16(1.0)
    w[0, 8] = bf16(tiny)      # lane 1
    w[0, 136] = bf16(tiny)    # lane 17
    w[1, 8] = bf16(tiny)      # lane 1
    w[1, 16] = bf16(tiny)     # lane 2
    x = np.ones(H, np.float32)
    got = oracle.router_logits(w, x)
    assert got[0] == np.float32(1 + 2 ** -23)
    assert got[1] == np.float32(1.0)


def test_router_within_fp32_error_bound():
    """|l_fp32 - l_exact| <= (H/32 + 5) * 2^-24 * sum|w x| (sequential FMA per lane
    then 5 pairwise levels; standard forward error bound)."""
    E, H = 64, 2048
    w = synth.router_weights(3, 1, E, H, 0.02)
    x = synth.tokens(3, 0, 1, H)[0]
    got = oracle.router_logits(w, x).astype(np.float64)
    wf = synth.bf16_to_f32(w).astype(np.float64)
    exact = wf @ x.astype(np.float64)
    bound = (H / 32 + 5) * 2.0 ** -24 * (np.abs(wf) @ np.abs(x.astype(np.float64)))
    assert np.all(np.abs(got - exact) <= bound)


def test_topk_forced_order_and_ties():
    """Logits forced through x = e_0: known order, ties broken by the lower index."""
    vals = [0.5, 2.0, -1.0, 2.0, 0.25, 3.0, 0.5, -3.0]
    E, H = len(vals), 256
    w = np.zeros((E, H), np.uint16)
    for e, v in enumerate(vals):
        w[e, 0] = bf16(v)
    x = np.zeros(H, np.float32)
    x[0] = 1.0
    logits = oracle.router_logits(w, x)
    assert list(oracle.topk(logits, 5)) == [5, 1, 3, 0, 6]


def test_topk_weights_textbook_softmax():
    """k = E: renormalised top-k weights are the textbook softmax; norm_topk = 0
    gives full-softmax probabilities (scipy reference)."""
    from scipy.special import softmax
    rng = np.random.default_rng(5)
    logits = rng.standard_normal(32).astype(np.float32)
    idx = oracle.topk(logits, 32)
    assert np.allclose(oracle.topk_weights(logits, idx, True), softmax(logits.astype(np.float64))[idx],
                       rtol=1e-13, atol=0)
    idx4 = oracle.topk(logits, 4)
    full = softmax(logits.astype(np.float64))
    assert np.allclose(oracle.topk_weights(logits, idx4, False), full[idx4], rtol=1e-13, atol=0)
    renorm = full[idx4] / full[idx4].sum()
    assert np.allclose(oracle.topk_weights(logits, idx4, True), renorm, rtol=1e-13, atol=0)


def test_shared_gate_closed_form():
    H = 128
    w = np.zeros(H, np.uint16)
    w[0] = bf16(0.5)
    w[5] = bf16(-2.0)
    x = np.zeros(H, np.float32)
    x[0], x[5] = 1.0, 0.25
    assert oracle.shared_gate(w, x) == pytest.approx(1 / (1 + math.exp(-(0.5 - 0.5))), abs=0)
    x[5] = 1.0
    assert oracle.shared_gate(w, x) == pytest.approx(1 / (1 + math.exp(1.5)), rel=1e-15)


# --------------------------------------------------------------------------
# the quantiser (input generator) closed form
# --------------------------------------------------------------------------

@pytest.mark.parametrize("bits,step", [(4, 0.125), (8, 2.0 ** -7)])
def test_quantiser_exact_grid_closed_form(bits, step):
    """A group that lies exactly on an fp16 grid m + step*k (k = 0..2^b-1 all
    present) quantises to scale = step, bias = m, q = k."""
    n = 1 << bits
    m = -1.0
    ks = np.arange(64) % n
    if n > 64:
        ks = (np.arange(64) * (n - 1)) // 63   # 0 .. n-1, both ends present
    w = (m + step * ks).astype(np.float32)[None, :]
    q, sb = synth.quantize_affine(w, bits)
    assert np.array_equal(q[0], ks.astype(np.uint8))
    assert synth.f16_to_f32(int(sb[0, 0, 0])) == step and synth.f16_to_f32(int(sb[0, 0, 1])) == m


def test_quantiser_round_trip_error_bound():
    """|w - (scale*q + bias)| <= scale/2 + (fp16 rounding of bias) + (2^b-1)*(fp16 rounding of scale)."""
    w = synth.normal_matrix(11, 0, 1, 0, 32, 256, 0.02)
    for bits in (4, 8):
        q, sb = synth.quantize_affine(w, bits)
        wh = oracle.dequant(q, sb)
        for g in range(4):
            blk = w[:, g * 64:(g + 1) * 64].astype(np.float64)
            mn, mx = blk.min(1), blk.max(1)
            s = sb[:, g, 0].view(np.float16).astype(np.float64)
            b = sb[:, g, 1].view(np.float16).astype(np.float64)
            qmax = (1 << bits) - 1
            bound = s / 2 + np.abs(b - mn) + qmax * np.abs(s - (mx - mn) / qmax) + 1e-12
            err = np.abs(blk - wh[:, g * 64:(g + 1) * 64]).max(1)
            assert np.all(err <= bound)


# --------------------------------------------------------------------------
# the two-expert worked example
# --------------------------------------------------------------------------

def _read_golden(name):
    vals = {}
    for line in open(os.path.join(GOLDEN, name)):
        line = line.strip()
        if line and not line.startswith("#"):
            k, v = line.split()
            vals[k] = float(v)
    return vals


def _hand_expert(c, u, d, H=64, I=64, col=0, d_rows=None):
    """Quantised arrays written by hand for gate[:, col] = c, up[:, col] = u (other
    columns 0) and down[j][:] = d * d_rows[j] (a constant group per output row)."""
    def one_col(v):
        q = np.zeros((I, H), np.uint8)
        sb = np.zeros((I, 1, 2), np.uint16)
        if v > 0:
            q[:, col] = 15
            sb[:, 0] = (f16(v / 15), f16(0.0))
        else:
            q[:, :] = 15
            q[:, col] = 0
            sb[:, 0] = (f16(-v / 15), f16(v))
        return q, sb
    qg, sbg = one_col(c)
    qu, sbu = one_col(u)
    qd = np.zeros((H, I), np.uint8)
    sbd = np.zeros((H, 1, 2), np.uint16)
    for j in range(H):
        sbd[j, 0] = (f16(0.0), f16(d * (1.0 if d_rows is None else d_rows[j])))
    return {"q_gate": qg, "sb_gate": sbg, "q_up": qu, "sb_up": sbu, "q_down": qd, "sb_down": sbd}


def _worked_layer():
    v = _read_golden("worked_example.txt")
    H = 64
    rw = np.zeros((2, H), np.uint16)
    rw[0, 0] = bf16(1.0)
    wsg = np.zeros(H, np.uint16)
    wsg[0] = bf16(v["g"])
    experts = {0: _hand_expert(v["c0"], v["u0"], v["d0"]), 1: _hand_expert(v["c1"], v["u1"], v["d1"])}
    layer = oracle.Layer(H, 2, 2, 64, 64, rw, wsg, experts, shared=_hand_expert(v["cs"], v["us"], v["ds"]))
    x = np.zeros(H, np.float32)
    x[0] = 1.0
    return v, layer, x


def _silu(z):
    return z / (1 + math.exp(-z))


def test_worked_example_two_experts():
    v, layer, x = _worked_layer()
    out = layer.token(x)
    e = math.e
    want = (e / (1 + e)) * 64 * v["d0"] * v["u0"] * _silu(v["c0"]) \
        + (1 / (1 + e)) * 64 * v["d1"] * v["u1"] * _silu(v["c1"]) \
        + (1 / (1 + math.exp(-v["g"]))) * 64 * v["ds"] * v["us"] * _silu(v["cs"])
    assert list(out["idx"]) == [0, 1]
    assert out["w"] == pytest.approx([e / (1 + e), 1 / (1 + e)], rel=1e-15)
    assert np.allclose(out["y"], want, rtol=1e-7, atol=0)
    assert want == pytest.approx(v["y"], abs=1e-9)


def test_worked_example_row_dependent_down_and_other_column():
    """Same example with the active input column at 37 and a down matrix whose
    value depends on the output row j (d * (j % 8 + 1) / 8): y_j scales with that
    factor, so a transposed down matrix or a wrong input column fails."""
    v = _read_golden("worked_example.txt")
    H, col = 64, 37
    rows = [(j % 8 + 1) / 8 for j in range(H)]
    rw = np.zeros((2, H), np.uint16)
    rw[0, col] = bf16(1.0)
    wsg = np.zeros(H, np.uint16)
    wsg[col] = bf16(v["g"])
    mk = lambda c, u, d: _hand_expert(c, u, d, col=col, d_rows=rows)
    layer = oracle.Layer(H, 2, 2, 64, 64, rw, wsg, {0: mk(v["c0"], v["u0"], v["d0"]), 1: mk(v["c1"], v["u1"], v["d1"])},
                         shared=mk(v["cs"], v["us"], v["ds"]))
    x = np.zeros(H, np.float32)
    x[col] = 1.0
    out = layer.token(x)
    e = math.e
    base = (e / (1 + e)) * 64 * v["d0"] * v["u0"] * _silu(v["c0"]) \
        + (1 / (1 + e)) * 64 * v["d1"] * v["u1"] * _silu(v["c1"]) \
        + (1 / (1 + math.exp(-v["g"]))) * 64 * v["ds"] * v["us"] * _silu(v["cs"])
    assert np.allclose(out["y"], base * np.array(rows), rtol=1e-7, atol=0)


def test_worked_example_prefill_rounds_x_and_weights_only():
    """Prefill emulation on the worked example with x0 = 1 + 2^-10 (fp32) and expert 0's
    down value d0' = d0 (1 + 2^-10) (fp16-exact, not bf16-exact).  The expert FFNs see
    bf16(x0) = 1 and bf16(d0') = d0; the router and the shared gate see the fp32 x0; the
    SwiGLU output silu(c) u is used unrounded.  The decode definition sees x0 and d0'
    as they are."""
    v = _read_golden("worked_example.txt")
    eps = 2.0 ** -10
    H = 64
    x0 = 1.0 + eps
    d0p = v["d0"] * (1.0 + eps)
    assert f16(d0p) != f16(v["d0"]) and bf16(d0p) == bf16(v["d0"])
    rw = np.zeros((2, H), np.uint16)
    rw[0, 0] = bf16(1.0)
    wsg = np.zeros(H, np.uint16)
    wsg[0] = bf16(v["g"])
    experts = {0: _hand_expert(v["c0"], v["u0"], d0p), 1: _hand_expert(v["c1"], v["u1"], v["d1"])}
    layer = oracle.Layer(H, 2, 2, 64, 64, rw, wsg, experts, shared=_hand_expert(v["cs"], v["us"], v["ds"]))
    x = np.zeros(H, np.float32)
    x[0] = x0
    l0 = x0  # fp32 router logit of expert 0; expert 1's is 0
    w0, w1 = math.exp(l0) / (math.exp(l0) + 1), 1 / (math.exp(l0) + 1)
    sig = 1 / (1 + math.exp(-v["g"] * x0))
    want_p = w0 * 64 * v["d0"] * v["u0"] * _silu(v["c0"]) \
        + w1 * 64 * v["d1"] * v["u1"] * _silu(v["c1"]) \
        + sig * 64 * v["ds"] * v["us"] * _silu(v["cs"])
    want_d = w0 * 64 * d0p * v["u0"] * x0 * _silu(v["c0"] * x0) \
        + w1 * 64 * v["d1"] * v["u1"] * x0 * _silu(v["c1"] * x0) \
        + sig * 64 * v["ds"] * v["us"] * x0 * _silu(v["cs"] * x0)
    p = layer.token(x, prefill=True)
    d = layer.token(x)
    assert list(p["idx"]) == [0, 1] and list(d["idx"]) == [0, 1]
    assert np.allclose(p["y"], want_p, rtol=1e-12, atol=0)
    assert np.allclose(d["y"], want_d, rtol=1e-12, atol=0)
    assert abs(want_p - want_d) > 1e-4 * abs(want_d)  # the two definitions differ here


# --------------------------------------------------------------------------
# invariants on a random tiny layer
# --------------------------------------------------------------------------

def _tiny_layer(seed=1, bits=4, with_bias=False):
    w = synth.CONFIGS["tiny"]
    H, E, k, I = w.hidden, w.n_experts, w.top_k, w.inter
    experts = {e: synth.expert(seed, 0, e, H, I, bits) for e in range(E)}
    shared = synth.expert(seed, 0, synth.SHARED, H, w.shared_inter, bits)
    rw = synth.router_weights(seed, 0, E, H, 0.02)
    wsg = synth.shared_gate_weights(seed, 0, H)
    bias = synth.zipf_bias(synth.rank_permutation(seed, 0, E)) if with_bias else None
    return oracle.Layer(H, E, k, I, w.shared_inter, rw, wsg, experts, shared=shared, router_bias=bias)


@pytest.mark.parametrize("bits", [4, 8])
def test_store_invariance_blob_vs_arrays(bits):
    """The answer is the same whether experts come from the arrays or from the
    oracle's own packed blobs (bitwise)."""
    layer = _tiny_layer(bits=bits)
    H, I = layer.hidden, layer.inter
    x = synth.tokens(1, 0, 3, H)
    a = layer.tokens(x)
    unpacked = {e: oracle.unpack_blob(oracle.pack_blob(d, H, I, bits), H, I, bits) for e, d in layer.experts.items()}
    layer.set_experts(unpacked)
    b = layer.tokens(x)
    assert np.array_equal(a["y"], b["y"]) and np.array_equal(a["idx"], b["idx"])


def test_layer_linear_in_shared_and_routed_parts():
    """y = route/combine split: combine with the routing weights doubled and sigma
    doubled is exactly twice as large (fp64 linearity of the combine)."""
    layer = _tiny_layer()
    x = synth.tokens(2, 0, 1, layer.hidden)[0]
    _, idx, w, sig = layer.route(x)
    y1 = layer.combine(x, idx, w, sig)
    y2 = layer.combine(x, idx, 2 * w, 2 * sig)
    assert np.allclose(y2, 2 * y1, rtol=1e-14, atol=1e-18)


def test_missing_expert_is_an_error():
    layer = _tiny_layer()
    x = synth.tokens(2, 0, 1, layer.hidden)[0]
    _, idx, _, _ = layer.route(x)
    layer.set_experts({e: d for e, d in layer.experts.items() if e != int(idx[0])})
    with pytest.raises(ValueError):
        layer.token(x)


def test_prefill_mode_close_to_decode():
    """bf16 operand rounding moves the layer output by O(2^-8) relative, not more
    (and not zero: the emulation is active)."""
    layer = _tiny_layer()
    x = synth.tokens(4, 0, 4, layer.hidden)
    d = layer.tokens(x)
    p = layer.tokens(x, prefill=True)
    assert np.array_equal(d["idx"], p["idx"])
    rel = np.linalg.norm(p["y"] - d["y"]) / np.linalg.norm(d["y"])
    assert 0 < rel < 2 ** -6


def test_renorm_closed_form():
    y = np.full(64, -3.0, np.float32)
    x = oracle.renorm(y, eps=1e-6)
    assert np.allclose(x, -3.0 / math.sqrt(9 + 1e-6), rtol=1e-7)


# --------------------------------------------------------------------------
# slot pool simulator
# --------------------------------------------------------------------------

def _golden_traces():
    blocks, cur = [], None
    for line in open(os.path.join(GOLDEN, "pool_traces.txt")):
        line = line.split("#")[0].strip()
        if not line:
            continue
        tok = line.split()
        if tok[0] == "policy":
            cur = {"policy": tok[1], "slots": int(tok[3]), "experts": int(tok[5]),
                   "aging": int(tok[7]) if len(tok) > 7 and tok[6] == "aging" else 64, "calls": []}
        elif tok[0] == "call":
            cur["calls"].append(([int(t) for t in tok[2:]], []))
        elif tok[0] == "ev":
            cur["calls"][-1][1].append((int(tok[1]), oracle.HIT if tok[2] == "HIT" else oracle.MISS,
                                        int(tok[3]), int(tok[4])))
        elif tok[0] == "end":
            blocks.append(cur)
    return blocks


_POLICY = {"lfu": oracle.POLICY_LFU_RECENCY, "lru": oracle.POLICY_LRU, "persist": oracle.POLICY_LFU_PERSIST,
           "aged": oracle.POLICY_LFU_AGED}


@pytest.mark.parametrize("block", range(5))
def test_pool_sim_hand_traces(block):
    b = _golden_traces()[block]
    sim = oracle.PoolSim(b["slots"], b["experts"], _POLICY[b["policy"]], aging_period=b["aging"])
    for req, want in b["calls"]:
        assert sim.request(req) == want, req


def test_pool_golden_covers_every_policy():
    assert sorted(b["policy"] for b in _golden_traces()) == ["aged", "lfu", "lfu", "lru", "persist"]


def test_pool_persistent_lfu_equals_brute_force_perfect_lfu():
    """Single-expert requests: persistent-count LFU is 'perfect LFU' (all-time
    counts, kept across evictions) with least-recent use as the tie-break."""
    rng = np.random.default_rng(11)
    S, E = 4, 12
    sim = oracle.PoolSim(S, E, oracle.POLICY_LFU_PERSIST)
    count, last, slot_of = Counter(), {}, {}
    for t in range(800):
        e = int(min(rng.zipf(1.3), E) - 1)
        (ev,) = sim.request([e])
        count[e] += 1
        if e in slot_of:
            assert ev == (e, oracle.HIT, slot_of[e], -1)
        else:
            if len(slot_of) < S:
                evicted, slot = -1, min(set(range(S)) - set(slot_of.values()))
            else:
                evicted = min(slot_of, key=lambda r: (count[r], last[r]))
                slot = slot_of.pop(evicted)
            slot_of[e] = slot
            assert ev == (e, oracle.MISS, slot, evicted)
        last[e] = t


def test_pool_aged_lfu_without_an_aging_call_is_lfu_recency():
    rng = np.random.default_rng(12)
    a = oracle.PoolSim(6, 20, oracle.POLICY_LFU_AGED, aging_period=1000)
    b = oracle.PoolSim(6, 20, oracle.POLICY_LFU_RECENCY)
    for _ in range(400):
        req = rng.choice(20, size=int(rng.integers(1, 4)), replace=False)
        assert a.request(req) == b.request(req)


def _belady_hits(stream, S):
    """Belady's MIN (evict the resident expert whose next request is furthest
    away): the most hits any policy can reach on single-expert requests."""
    resident, hits = set(), 0
    for t, e in enumerate(stream):
        if e in resident:
            hits += 1
            continue
        if len(resident) == S:
            def next_use(r):
                for u in range(t + 1, len(stream)):
                    if stream[u] == r:
                        return u
                return len(stream)
            resident.remove(max(resident, key=next_use))
        resident.add(e)
    return hits


@pytest.mark.parametrize("policy", range(4))
def test_pool_hits_bounded_by_belady_and_compulsory_misses(policy):
    rng = np.random.default_rng(13 + policy)
    stream = [int(min(rng.zipf(1.2), 16) - 1) for _ in range(600)]
    sim = oracle.PoolSim(5, 16, policy, aging_period=8)
    hits = sum(sim.request([e])[0][1] == oracle.HIT for e in stream)
    assert hits <= _belady_hits(stream, 5)
    big = oracle.PoolSim(16, 16, policy, aging_period=8)  # room for every expert: only first requests miss
    misses = sum(big.request([e])[0][1] == oracle.MISS for e in stream)
    assert misses == len(set(stream))


def test_pool_lru_equals_textbook_lru():
    """Single-expert requests: the LRU policy is textbook LRU (OrderedDict)."""
    rng = np.random.default_rng(9)
    S, E = 4, 10
    sim = oracle.PoolSim(S, E, oracle.POLICY_LRU)
    lru = OrderedDict()
    for _ in range(500):
        e = int(rng.integers(0, E))
        (ev,) = sim.request([e])
        if e in lru:
            lru.move_to_end(e)
            assert ev[1] == oracle.HIT
        else:
            evicted = -1
            if len(lru) == S:
                evicted, _ = lru.popitem(last=False)
            lru[e] = True
            assert ev[1] == oracle.MISS and ev[3] == evicted


def test_pool_request_larger_than_pool_is_error_and_preload_hits():
    sim = oracle.PoolSim(2, 6)
    with pytest.raises(ValueError):
        sim.request([0, 1, 2])
    pre = oracle.PoolSim(6, 6, preload=True)
    evs = pre.request([5, 1, 3])
    assert evs == [(1, oracle.HIT, 1, -1), (3, oracle.HIT, 3, -1), (5, oracle.HIT, 5, -1)]
