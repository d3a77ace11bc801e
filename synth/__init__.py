"""Seeded synthetic inputs for the routed sparse-MoE layer (shared by the CUDA
path's tests/bench and by the CPU oracle).

This package holds none of the layer's arithmetic.  It draws Gaussian weights
and activations from Philox4x32-10 streams, quantises weight matrices with an
MLX-style affine group quantiser into (q, scale, bias) arrays, draws bf16
router weights and a Zipf expert-popularity bias, and applies popularity
drift.  See ``synth.c`` for the stream addressing.
"""
from __future__ import annotations

import ctypes
import os
import subprocess
import threading

import numpy as np

from .configs import CONFIGS, Workload  # noqa: F401

_HERE = os.path.dirname(os.path.abspath(__file__))
_SO = os.path.join(_HERE, "libsynth.so")
_lock = threading.Lock()
_lib = None

SHARED = 0xFFFFF  # expert id that addresses the shared expert's streams

_u8p = np.ctypeslib.ndpointer(dtype=np.uint8, flags="C_CONTIGUOUS")
_u16p = np.ctypeslib.ndpointer(dtype=np.uint16, flags="C_CONTIGUOUS")
_i32p = np.ctypeslib.ndpointer(dtype=np.int32, flags="C_CONTIGUOUS")
_u32p = np.ctypeslib.ndpointer(dtype=np.uint32, flags="C_CONTIGUOUS")
_f32p = np.ctypeslib.ndpointer(dtype=np.float32, flags="C_CONTIGUOUS")


def build(force: bool = False) -> str:
    """Compile libsynth.so with gcc (plain C, no fast-math, no contraction)."""
    src = os.path.join(_HERE, "synth.c")
    if not force and os.path.exists(_SO) and os.path.getmtime(_SO) >= os.path.getmtime(src):
        return _SO
    tmp = _SO + f".tmp{os.getpid()}"
    subprocess.check_call(
        ["gcc", "-O2", "-std=gnu11", "-ffp-contract=off", "-fPIC", "-shared", "-o", tmp, src, "-lm"]
    )
    os.replace(tmp, _SO)
    return _SO


def _load():
    global _lib
    with _lock:
        if _lib is not None:
            return _lib
        lib = ctypes.CDLL(build())
        c = ctypes
        lib.synth_philox4x32_10.argtypes = [_u32p, _u32p, _u32p]
        lib.synth_normal_row.argtypes = [c.c_uint64, c.c_uint32, c.c_uint32, c.c_uint32, c.c_uint32,
                                         c.c_uint32, c.c_float, _f32p]
        lib.synth_normal_matrix.argtypes = [c.c_uint64, c.c_uint32, c.c_uint32, c.c_uint32, c.c_uint32,
                                            c.c_uint32, c.c_uint32, c.c_float, _f32p]
        lib.synth_f32_to_f16.argtypes = [c.c_float]
        lib.synth_f32_to_f16.restype = c.c_uint16
        lib.synth_f16_to_f32.argtypes = [c.c_uint16]
        lib.synth_f16_to_f32.restype = c.c_float
        lib.synth_f32_to_bf16.argtypes = [c.c_float]
        lib.synth_f32_to_bf16.restype = c.c_uint16
        lib.synth_quantize_affine.argtypes = [_f32p, c.c_uint32, c.c_uint32, c.c_uint32, c.c_int, _u8p, _u16p]
        lib.synth_expert.argtypes = [c.c_uint64, c.c_uint32, c.c_uint32, c.c_uint32, c.c_uint32, c.c_int,
                                     c.c_float, _u8p, _u16p, _u8p, _u16p, _u8p, _u16p, _f32p]
        lib.synth_expert.restype = c.c_int
        lib.synth_router_weights.argtypes = [c.c_uint64, c.c_uint32, c.c_uint32, c.c_uint32, c.c_float,
                                             _u16p, _f32p]
        lib.synth_shared_gate_weights.argtypes = [c.c_uint64, c.c_uint32, c.c_uint32, c.c_float, _u16p, _f32p]
        lib.synth_tokens.argtypes = [c.c_uint64, c.c_uint32, c.c_uint32, c.c_uint32, _f32p]
        lib.synth_rank_permutation.argtypes = [c.c_uint64, c.c_uint32, c.c_uint32, _i32p]
        lib.synth_zipf_bias.argtypes = [c.c_uint32, c.c_double, _i32p, _f32p]
        lib.synth_drift_step.argtypes = [c.c_uint64, c.c_uint32, c.c_uint32, c.c_uint32, c.c_uint32, _i32p]
        _lib = lib
        return lib


def philox4x32_10(ctr, key) -> np.ndarray:
    out = np.zeros(4, np.uint32)
    _load().synth_philox4x32_10(np.asarray(ctr, np.uint32), np.asarray(key, np.uint32), out)
    return out


def normal_matrix(seed, layer, kind, expert, rows, cols, sigma, row0=0) -> np.ndarray:
    out = np.empty((rows, cols), np.float32)
    _load().synth_normal_matrix(seed, layer, kind, expert, row0, rows, cols, sigma, out)
    return out


def f32_to_f16(v: float) -> int:
    return int(_load().synth_f32_to_f16(v))


def f16_to_f32(h: int) -> float:
    return float(_load().synth_f16_to_f32(h))


def f32_to_bf16(v: float) -> int:
    return int(_load().synth_f32_to_bf16(v))


def quantize_affine(w: np.ndarray, bits: int, group: int = 64):
    """(rows, cols) fp32 -> q uint8 (rows, cols), sb uint16 (rows, cols/group, 2)."""
    w = np.ascontiguousarray(w, np.float32)
    rows, cols = w.shape
    q = np.empty((rows, cols), np.uint8)
    sb = np.empty((rows, cols // group, 2), np.uint16)
    _load().synth_quantize_affine(w, rows, cols, group, bits, q, sb.reshape(-1))
    return q, sb


def expert(seed: int, layer: int, expert_id: int, hidden: int, inter: int, bits: int, sigma: float = 0.02):
    """Quantised arrays of one expert (expert_id = SHARED for the shared expert).

    Returns dict with q_gate/q_up (inter, hidden) uint8, q_down (hidden, inter)
    uint8 and sb_* uint16 (rows, cols/64, 2) holding fp16 (scale, bias).
    """
    lib = _load()
    d = {
        "q_gate": np.empty((inter, hidden), np.uint8),
        "sb_gate": np.empty((inter, hidden // 64, 2), np.uint16),
        "q_up": np.empty((inter, hidden), np.uint8),
        "sb_up": np.empty((inter, hidden // 64, 2), np.uint16),
        "q_down": np.empty((hidden, inter), np.uint8),
        "sb_down": np.empty((hidden, inter // 64, 2), np.uint16),
    }
    scratch = np.empty(inter * hidden, np.float32)
    rc = lib.synth_expert(seed, layer, expert_id, hidden, inter, bits, sigma,
                          d["q_gate"].reshape(-1), d["sb_gate"].reshape(-1),
                          d["q_up"].reshape(-1), d["sb_up"].reshape(-1),
                          d["q_down"].reshape(-1), d["sb_down"].reshape(-1), scratch)
    if rc != 0:
        raise ValueError("synth_expert: bad shape or bits")
    return d


def router_weights(seed: int, layer: int, n_experts: int, hidden: int, sigma: float) -> np.ndarray:
    """bf16 bit patterns (n_experts, hidden)."""
    out = np.empty((n_experts, hidden), np.uint16)
    _load().synth_router_weights(seed, layer, n_experts, hidden, sigma, out.reshape(-1),
                                 np.empty(hidden, np.float32))
    return out


def shared_gate_weights(seed: int, layer: int, hidden: int, sigma: float = 0.02) -> np.ndarray:
    out = np.empty(hidden, np.uint16)
    _load().synth_shared_gate_weights(seed, layer, hidden, sigma, out, np.empty(hidden, np.float32))
    return out


def tokens(seed: int, step: int, n_tokens: int, hidden: int) -> np.ndarray:
    out = np.empty((n_tokens, hidden), np.float32)
    _load().synth_tokens(seed, step, n_tokens, hidden, out.reshape(-1))
    return out


def rank_permutation(seed: int, layer: int, n_experts: int) -> np.ndarray:
    out = np.empty(n_experts, np.int32)
    _load().synth_rank_permutation(seed, layer, n_experts, out)
    return out


def zipf_bias(expert_at: np.ndarray, s: float = 1.1) -> np.ndarray:
    expert_at = np.ascontiguousarray(expert_at, np.int32)
    out = np.empty(expert_at.shape[0], np.float32)
    _load().synth_zipf_bias(expert_at.shape[0], s, expert_at, out)
    return out


def drift_step(seed: int, layer: int, step: int, expert_at: np.ndarray, n_swaps: int = 4) -> None:
    """In-place adjacent-rank swaps of expert_at (int32, contiguous)."""
    assert expert_at.dtype == np.int32 and expert_at.flags["C_CONTIGUOUS"]
    _load().synth_drift_step(seed, layer, step, expert_at.shape[0], n_swaps, expert_at)


def bf16_to_f32(bits: np.ndarray) -> np.ndarray:
    """Exact widening of bf16 bit patterns (a bit shift; no rounding involved)."""
    return (np.asarray(bits, np.uint32) << 16).view(np.float32)


def layer_inputs(w: "Workload", layer: int):
    """Router weights (bf16 bits), shared-gate weights (bf16 bits) and router
    bias (fp32 or None) of one layer of a workload."""
    wr = router_weights(w.seed, layer, w.n_experts, w.hidden, w.router_sigma)
    wsg = shared_gate_weights(w.seed, layer, w.hidden, w.sigma)
    beta = None
    if w.zipf_s:
        beta = zipf_bias(rank_permutation(w.seed, layer, w.n_experts), w.zipf_s)
    return wr, wsg, beta
