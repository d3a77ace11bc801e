"""CPU oracle for the routed sparse-MoE layer -- TEST INFRASTRUCTURE.

Only ``tests/``, ``__graft_entry__.smoke()`` and the CPU-baseline leg of
``bench.py`` may import this package.  The product path (the
``int4_expert_streaming_gb300`` package and its CUDA library) never does.

The arithmetic lives in ``moe_oracle.c`` (plain C, fp64, built with
``-ffp-contract=off``); this module only marshals numpy arrays into it.  It
shares no code with the CUDA library.
"""
from __future__ import annotations

import concurrent.futures as _cf
import ctypes
import os
import subprocess
import threading

import numpy as np

_HERE = os.path.dirname(os.path.abspath(__file__))
_SO = os.path.join(_HERE, "liboracle.so")
_lock = threading.Lock()
_lib = None

OK, EINVAL, EMISSING, EPOOL = 0, -1, -2, -3
POLICY_LFU_RECENCY, POLICY_LRU, POLICY_LFU_PERSIST, POLICY_LFU_AGED = 0, 1, 2, 3
HIT, MISS = 0, 1


def build(force: bool = False) -> str:
    src = os.path.join(_HERE, "moe_oracle.c")
    if not force and os.path.exists(_SO) and os.path.getmtime(_SO) >= os.path.getmtime(src):
        return _SO
    tmp = _SO + f".tmp{os.getpid()}"
    subprocess.check_call(["gcc", "-O2", "-std=c11", "-ffp-contract=off", "-fPIC", "-shared", "-o", tmp, src, "-lm"])
    os.replace(tmp, _SO)
    return _SO


class _Expert(ctypes.Structure):
    _fields_ = [
        ("q_gate", ctypes.c_void_p), ("sb_gate", ctypes.c_void_p),
        ("q_up", ctypes.c_void_p), ("sb_up", ctypes.c_void_p),
        ("q_down", ctypes.c_void_p), ("sb_down", ctypes.c_void_p),
    ]


class _Layer(ctypes.Structure):
    _fields_ = [
        ("hidden", ctypes.c_int32), ("n_experts", ctypes.c_int32), ("top_k", ctypes.c_int32),
        ("inter", ctypes.c_int32), ("shared_inter", ctypes.c_int32), ("norm_topk", ctypes.c_int32),
        ("router_w", ctypes.c_void_p), ("router_bias", ctypes.c_void_p), ("shared_gate_w", ctypes.c_void_p),
        ("experts", ctypes.POINTER(_Expert)), ("shared", ctypes.POINTER(_Expert)),
    ]


def _p(a):
    return None if a is None else a.ctypes.data_as(ctypes.c_void_p)


def _load():
    global _lib
    with _lock:
        if _lib is not None:
            return _lib
        lib = ctypes.CDLL(build())
        c = ctypes
        vp = c.c_void_p
        lib.orc_half_to_double.argtypes = [c.c_uint16]
        lib.orc_half_to_double.restype = c.c_double
        lib.orc_bf16_to_float.argtypes = [c.c_uint16]
        lib.orc_bf16_to_float.restype = c.c_float
        lib.orc_float_to_bf16.argtypes = [c.c_float]
        lib.orc_float_to_bf16.restype = c.c_uint16
        lib.orc_dequant.argtypes = [vp, vp, c.c_int, c.c_int, vp]
        lib.orc_router_logit.argtypes = [vp, vp, c.c_int, c.c_float]
        lib.orc_router_logit.restype = c.c_float
        lib.orc_router_logits.argtypes = [vp, vp, vp, c.c_int, c.c_int, vp]
        lib.orc_topk.argtypes = [vp, c.c_int, c.c_int, vp]
        lib.orc_topk_weights.argtypes = [vp, c.c_int, c.c_int, vp, c.c_int, vp]
        lib.orc_shared_gate.argtypes = [vp, vp, c.c_int]
        lib.orc_shared_gate.restype = c.c_double
        lib.orc_route_token.argtypes = [c.POINTER(_Layer), vp, vp, vp, vp, vp]
        lib.orc_route_token.restype = c.c_int
        lib.orc_combine_token.argtypes = [c.POINTER(_Layer), vp, vp, vp, c.c_double, c.c_int, vp]
        lib.orc_combine_token.restype = c.c_int
        lib.orc_layer_token.argtypes = [c.POINTER(_Layer), vp, c.c_int, vp, vp, vp, vp, vp]
        lib.orc_layer_token.restype = c.c_int
        lib.orc_renorm.argtypes = [vp, c.c_int, c.c_double, vp]
        lib.orc_blob_bytes.argtypes = [c.c_int, c.c_int, c.c_int]
        lib.orc_blob_bytes.restype = c.c_size_t
        lib.orc_blob_stride.argtypes = [c.c_int, c.c_int, c.c_int]
        lib.orc_blob_stride.restype = c.c_size_t
        lib.orc_pack_blob.argtypes = [c.c_int, c.c_int, c.c_int, c.POINTER(_Expert), vp, c.c_size_t]
        lib.orc_pack_blob.restype = c.c_int
        lib.orc_unpack_blob.argtypes = [c.c_int, c.c_int, c.c_int, vp, vp, vp, vp, vp, vp, vp]
        lib.orc_unpack_blob.restype = c.c_int
        lib.orc_pool_request.argtypes = [c.c_int, c.c_int, c.c_int, c.c_int, vp, vp, vp, vp, vp, c.c_int64, vp,
                                          c.c_int, vp]
        lib.orc_pool_request.restype = c.c_int
        _lib = lib
        return lib


# --------------------------------------------------------------------------
# scalar helpers
# --------------------------------------------------------------------------

def half_to_double(h: int) -> float:
    return float(_load().orc_half_to_double(h))


def float_to_bf16(v: float) -> int:
    return int(_load().orc_float_to_bf16(v))


def dequant(q: np.ndarray, sb: np.ndarray) -> np.ndarray:
    q = np.ascontiguousarray(q, np.uint8)
    sb = np.ascontiguousarray(sb, np.uint16)
    rows, cols = q.shape
    w = np.empty((rows, cols), np.float64)
    _load().orc_dequant(_p(q), _p(sb), rows, cols, _p(w))
    return w


def router_logits(w_bf16: np.ndarray, x: np.ndarray, bias=None) -> np.ndarray:
    w_bf16 = np.ascontiguousarray(w_bf16, np.uint16)
    x = np.ascontiguousarray(x, np.float32)
    e, h = w_bf16.shape
    b = None if bias is None else np.ascontiguousarray(bias, np.float32)
    out = np.empty(e, np.float32)
    _load().orc_router_logits(_p(w_bf16), _p(b), _p(x), h, e, _p(out))
    return out


def topk(logits: np.ndarray, k: int) -> np.ndarray:
    logits = np.ascontiguousarray(logits, np.float32)
    idx = np.empty(k, np.int32)
    _load().orc_topk(_p(logits), logits.shape[0], k, _p(idx))
    return idx


def topk_weights(logits: np.ndarray, idx: np.ndarray, norm_topk: bool = True) -> np.ndarray:
    logits = np.ascontiguousarray(logits, np.float32)
    idx = np.ascontiguousarray(idx, np.int32)
    w = np.empty(idx.shape[0], np.float64)
    _load().orc_topk_weights(_p(logits), logits.shape[0], idx.shape[0], _p(idx), int(norm_topk), _p(w))
    return w


def shared_gate(w_sg: np.ndarray, x: np.ndarray) -> float:
    w_sg = np.ascontiguousarray(w_sg, np.uint16)
    x = np.ascontiguousarray(x, np.float32)
    return float(_load().orc_shared_gate(_p(w_sg), _p(x), x.shape[0]))


def renorm(y: np.ndarray, eps: float = 1e-6) -> np.ndarray:
    """Row-wise (last axis) x = y / sqrt(mean(y^2) + eps)."""
    y = np.ascontiguousarray(y, np.float32)
    x = np.empty_like(y)
    rows_y, rows_x = y.reshape(-1, y.shape[-1]), x.reshape(-1, y.shape[-1])
    for r in range(rows_y.shape[0]):
        _load().orc_renorm(_p(rows_y[r]), y.shape[-1], eps, _p(rows_x[r]))
    return x


# --------------------------------------------------------------------------
# blobs
# --------------------------------------------------------------------------

def blob_bytes(hidden: int, inter: int, bits: int) -> int:
    return int(_load().orc_blob_bytes(hidden, inter, bits))


def blob_stride(hidden: int, inter: int, bits: int) -> int:
    return int(_load().orc_blob_stride(hidden, inter, bits))


def _expert_struct(d) -> _Expert:
    return _Expert(_p(d["q_gate"]), _p(d["sb_gate"]), _p(d["q_up"]), _p(d["sb_up"]),
                   _p(d["q_down"]), _p(d["sb_down"]))


def pack_blob(expert: dict, hidden: int, inter: int, bits: int) -> np.ndarray:
    """The oracle's own packer: one expert -> its fixed-stride blob (uint8)."""
    e = {k: np.ascontiguousarray(v) for k, v in expert.items()}
    out = np.empty(blob_stride(hidden, inter, bits), np.uint8)
    rc = _load().orc_pack_blob(hidden, inter, bits, ctypes.byref(_expert_struct(e)), _p(out), out.nbytes)
    if rc != OK:
        raise ValueError(f"orc_pack_blob failed ({rc})")
    return out


def unpack_blob(blob: np.ndarray, hidden: int, inter: int, bits: int) -> dict:
    blob = np.ascontiguousarray(blob, np.uint8)
    d = {
        "q_gate": np.empty((inter, hidden), np.uint8), "sb_gate": np.empty((inter, hidden // 64, 2), np.uint16),
        "q_up": np.empty((inter, hidden), np.uint8), "sb_up": np.empty((inter, hidden // 64, 2), np.uint16),
        "q_down": np.empty((hidden, inter), np.uint8), "sb_down": np.empty((hidden, inter // 64, 2), np.uint16),
    }
    rc = _load().orc_unpack_blob(hidden, inter, bits, _p(blob), _p(d["q_gate"]), _p(d["sb_gate"]),
                                 _p(d["q_up"]), _p(d["sb_up"]), _p(d["q_down"]), _p(d["sb_down"]))
    if rc != OK:
        raise ValueError(f"orc_unpack_blob failed ({rc})")
    return d


# --------------------------------------------------------------------------
# layers
# --------------------------------------------------------------------------

class Layer:
    """One MoE layer's inputs as numpy arrays.

    experts: dict expert_id -> expert dict (missing ids are "not supplied";
    routing to one is an error).  shared: expert dict or None.
    router_w: bf16 bits (E, H); shared_gate_w: bf16 bits (H,); router_bias: fp32 (E,) or None.
    """

    def __init__(self, hidden, n_experts, top_k, inter, shared_inter, router_w, shared_gate_w, experts,
                 shared=None, router_bias=None, norm_topk=True):
        self.hidden, self.n_experts, self.top_k = hidden, n_experts, top_k
        self.inter, self.shared_inter = inter, shared_inter
        self.router_w = np.ascontiguousarray(router_w, np.uint16)
        self.shared_gate_w = np.ascontiguousarray(shared_gate_w, np.uint16)
        self.router_bias = None if router_bias is None else np.ascontiguousarray(router_bias, np.float32)
        self.experts = {int(k): {n: np.ascontiguousarray(a) for n, a in v.items()} for k, v in experts.items()}
        self.shared = None if shared is None else {n: np.ascontiguousarray(a) for n, a in shared.items()}
        self.norm_topk = bool(norm_topk)
        self._rebuild()

    def _rebuild(self):
        arr = (_Expert * self.n_experts)()
        for e, d in self.experts.items():
            arr[e] = _expert_struct(d)
        self._arr = arr
        self._shared = _expert_struct(self.shared) if self.shared is not None else None
        self._struct = _Layer(
            self.hidden, self.n_experts, self.top_k, self.inter,
            self.shared_inter if self.shared is not None else 0, int(self.norm_topk),
            _p(self.router_w), _p(self.router_bias), _p(self.shared_gate_w),
            ctypes.cast(arr, ctypes.POINTER(_Expert)),
            ctypes.pointer(self._shared) if self._shared is not None else None,
        )

    def set_experts(self, experts: dict):
        self.experts = {int(k): {n: np.ascontiguousarray(a) for n, a in v.items()} for k, v in experts.items()}
        self._rebuild()

    # -- routing only -----------------------------------------------------
    def route(self, x: np.ndarray):
        """-> (logits fp32 (E,), idx int32 (k,), w fp64 (k,), sigma float)"""
        x = np.ascontiguousarray(x, np.float32)
        logits = np.empty(self.n_experts, np.float32)
        idx = np.empty(self.top_k, np.int32)
        w = np.empty(self.top_k, np.float64)
        sig = ctypes.c_double()
        rc = _load().orc_route_token(ctypes.byref(self._struct), _p(x), _p(logits), _p(idx), _p(w),
                                     ctypes.byref(sig))
        if rc != OK:
            raise ValueError(f"orc_route_token failed ({rc})")
        return logits, idx, w, sig.value

    def combine(self, x, idx, w, sigma, prefill=False) -> np.ndarray:
        """fp64 (H,) output of the experts given the routing."""
        x = np.ascontiguousarray(x, np.float32)
        idx = np.ascontiguousarray(idx, np.int32)
        w = np.ascontiguousarray(w, np.float64)
        y = np.empty(self.hidden, np.float64)
        rc = _load().orc_combine_token(ctypes.byref(self._struct), _p(x), _p(idx), _p(w), float(sigma),
                                       int(prefill), _p(y))
        if rc != OK:
            raise ValueError(f"orc_combine_token failed ({rc})")
        return y

    def token(self, x: np.ndarray, prefill=False):
        """-> dict(y fp32 (H,), idx, w, sigma, logits)"""
        x = np.ascontiguousarray(x, np.float32)
        y = np.empty(self.hidden, np.float32)
        logits = np.empty(self.n_experts, np.float32)
        idx = np.empty(self.top_k, np.int32)
        w = np.empty(self.top_k, np.float64)
        sig = ctypes.c_double()
        rc = _load().orc_layer_token(ctypes.byref(self._struct), _p(x), int(prefill), _p(y), _p(idx), _p(w),
                                     ctypes.byref(sig), _p(logits))
        if rc != OK:
            raise ValueError(f"orc_layer_token failed ({rc})")
        return {"y": y, "idx": idx, "w": w, "sigma": sig.value, "logits": logits}

    def tokens(self, X: np.ndarray, prefill=False, threads: int = 1):
        """All rows of X, optionally split over host threads (per-token work unchanged)."""
        X = np.ascontiguousarray(X, np.float32)
        if threads <= 1 or X.shape[0] == 1:
            outs = [self.token(X[t], prefill) for t in range(X.shape[0])]
        else:
            with _cf.ThreadPoolExecutor(threads) as ex:
                outs = list(ex.map(lambda t: self.token(X[t], prefill), range(X.shape[0])))
        return {
            "y": np.stack([o["y"] for o in outs]),
            "idx": np.stack([o["idx"] for o in outs]),
            "w": np.stack([o["w"] for o in outs]),
            "sigma": np.array([o["sigma"] for o in outs]),
            "logits": np.stack([o["logits"] for o in outs]),
        }


# --------------------------------------------------------------------------
# slot pool simulator
# --------------------------------------------------------------------------

class PoolSim:
    """Per-layer slot pool: LFU + recency, LRU, persistent-count LFU or aged LFU
    (halving every `aging_period` calls); see orc_pool_request."""

    def __init__(self, slots: int, n_experts: int, policy: int = POLICY_LFU_RECENCY, preload: bool = False,
                 aging_period: int = 64):
        self.slots, self.n_experts, self.policy, self.aging_period = slots, n_experts, policy, aging_period
        self.slot_expert = np.full(slots, -1, np.int32)
        self.slot_freq = np.zeros(slots, np.int64)
        self.slot_last = np.full(slots, -1, np.int64)
        self.expert_slot = np.full(n_experts, -1, np.int32)
        self.expert_count = np.zeros(n_experts, np.int64)
        self.clock = 0
        if preload:
            if slots < n_experts:
                raise ValueError("preload needs one slot per expert")
            for e in range(n_experts):
                self.slot_expert[e] = e
                self.expert_slot[e] = e

    def request(self, experts) -> list:
        """Request the set of experts (any order, duplicates allowed); advances the
        clock; returns events [(expert, kind, slot, evicted)]."""
        req = np.array(sorted(set(int(e) for e in experts)), np.int32)
        ev = np.empty((max(len(req), 1), 4), np.int32)
        n = _load().orc_pool_request(self.slots, self.n_experts, self.policy, self.aging_period,
                                     _p(self.slot_expert), _p(self.slot_freq), _p(self.slot_last),
                                     _p(self.expert_slot), _p(self.expert_count), self.clock, _p(req), len(req),
                                     _p(ev))
        if n < 0:
            raise ValueError(f"orc_pool_request failed ({n})")
        self.clock += 1
        return [tuple(int(v) for v in ev[i]) for i in range(n)]
