"""Python binding of libmoe.so -- the routed sparse-MoE layer with expert
streaming on one GB300 (sm_103a).

Argument marshalling only: every step of the layer runs in the library's CUDA
kernels.  The names mirror the C ABI in ``include/moe.h``.  Device buffers are
passed as CUDA torch tensors (fp32 / int32, contiguous) or raw integer device
addresses; streams as ``torch.cuda.Stream`` or raw ``cudaStream_t`` integers.

Importing the package does not need a GPU; loading the library does need the
built ``libmoe.so`` and raises if it is missing -- there is no fallback.
"""
from __future__ import annotations

import ctypes
import os
import threading

import numpy as np

from ._build import LIB as _LIB_PATH, build  # noqa: F401

MOE_OK, MOE_EINVAL, MOE_ENOMEM, MOE_ECUDA, MOE_EPOOL, MOE_ETIMEOUT, MOE_ESTATE, MOE_EIO = 0, -1, -2, -3, -4, -5, -6, -7
MOE_STORE_DIRECT = 0x1
MOE_EVICT_LFU_RECENCY, MOE_EVICT_LRU, MOE_EVICT_LFU_PERSIST, MOE_EVICT_LFU_AGED = 0, 1, 2, 3
MOE_FAULT_PINNED_ALLOC, MOE_FAULT_MISS_COPY, MOE_FAULT_WAIT_TIMEOUT, MOE_FAULT_DEVICE_WAIT = 0x1, 0x2, 0x4, 0x8
_ERRNAMES = {MOE_EINVAL: "MOE_EINVAL", MOE_ENOMEM: "MOE_ENOMEM", MOE_ECUDA: "MOE_ECUDA", MOE_EPOOL: "MOE_EPOOL",
             MOE_ETIMEOUT: "MOE_ETIMEOUT", MOE_ESTATE: "MOE_ESTATE", MOE_EIO: "MOE_EIO"}

# every symbol include/moe.h declares
EXPORTS = (
    "moe_blob_bytes", "moe_blob_stride", "moe_pack_expert", "moe_create", "moe_destroy", "moe_load_experts",
    "moe_set_router_bias", "moe_set_router_bias_all", "moe_forward_decode", "moe_forward_decode_stack", "moe_forward_prefill",
    "moe_pool_stats", "moe_pool_reset", "moe_pool_trace", "moe_launch_count", "moe_prefill_profile", "moe_prefill_kernel_ms", "moe_route_noalloc", "moe_last_error", "moe_slotpool_create", "moe_slotpool_destroy",
    "moe_slotpool_request", "moe_store_create", "moe_store_write_layer", "moe_store_info", "moe_store_read",
)


class MoeError(RuntimeError):
    def __init__(self, code: int, msg: str):
        super().__init__(f"{_ERRNAMES.get(code, code)}: {msg}")
        self.code = code


class moe_config(ctypes.Structure):
    _fields_ = [(n, ctypes.c_int32) for n in (
        "n_layers", "hidden", "n_experts", "top_k", "inter", "shared_inter", "bits", "group_size", "pool_slots",
        "norm_topk", "policy", "device", "max_batch", "max_tokens")] + [
        ("fault_flags", ctypes.c_uint32), ("fault_arg", ctypes.c_int32), ("timeout_ms", ctypes.c_int32),
        ("aging_period", ctypes.c_int32), ("store_flags", ctypes.c_uint32), ("store_path", ctypes.c_char_p),
        ("layer_bits", ctypes.POINTER(ctypes.c_int32))]


class moe_pool_stats_t(ctypes.Structure):
    _fields_ = [("hits", ctypes.c_uint64), ("misses", ctypes.c_uint64), ("evictions", ctypes.c_uint64),
                ("h2d_bytes", ctypes.c_uint64), ("h2d_ms", ctypes.c_double), ("resident", ctypes.c_int32),
                ("calls", ctypes.c_int32)]


_lock = threading.Lock()
_lib = None


def load_library(path: str | None = None):
    """Load libmoe.so (raises if it has not been built)."""
    global _lib
    with _lock:
        if _lib is not None:
            return _lib
        p = path or _LIB_PATH
        if not os.path.exists(p):
            raise RuntimeError(f"{p} is missing: build it with int4_expert_streaming_gb300.build() "
                               "(this package has no CPU fallback)")
        lib = ctypes.CDLL(p)
        c, vp, i32, sz = ctypes, ctypes.c_void_p, ctypes.c_int32, ctypes.c_size_t
        lib.moe_blob_bytes.argtypes = [i32, i32, i32]
        lib.moe_blob_bytes.restype = sz
        lib.moe_blob_stride.argtypes = [i32, i32, i32]
        lib.moe_blob_stride.restype = sz
        lib.moe_pack_expert.argtypes = [i32, i32, i32, vp, vp, vp, vp, vp, vp, vp, sz]
        lib.moe_create.argtypes = [c.POINTER(moe_config), c.POINTER(vp)]
        lib.moe_destroy.argtypes = [vp]
        lib.moe_destroy.restype = None
        lib.moe_load_experts.argtypes = [vp, i32, vp, sz, vp, vp, vp, vp]
        lib.moe_set_router_bias.argtypes = [vp, i32, vp, vp]
        lib.moe_set_router_bias_all.argtypes = [vp, vp, vp]
        lib.moe_forward_decode.argtypes = [vp, i32, vp, i32, vp, vp, vp, vp]
        lib.moe_forward_decode_stack.argtypes = [vp, i32, i32, vp, i32, vp, c.c_float, vp, vp, vp, vp]
        lib.moe_forward_prefill.argtypes = [vp, i32, vp, i32, vp, vp, vp, vp]
        lib.moe_pool_stats.argtypes = [vp, i32, c.POINTER(moe_pool_stats_t)]
        lib.moe_pool_reset.argtypes = [vp, i32, i32, i32, vp]
        lib.moe_pool_trace.argtypes = [vp, vp, sz, c.POINTER(sz)]
        lib.moe_launch_count.argtypes = [vp, c.POINTER(c.c_uint64)]
        lib.moe_prefill_profile.argtypes = [vp, i32]
        lib.moe_route_noalloc.argtypes = [vp, i32, vp, i32, vp, vp, vp]
        lib.moe_prefill_kernel_ms.argtypes = [vp, c.POINTER(c.c_double), c.POINTER(c.c_int64)]
        lib.moe_last_error.argtypes = [vp]
        lib.moe_last_error.restype = c.c_char_p
        lib.moe_slotpool_create.argtypes = [i32, i32, i32, i32, c.POINTER(vp)]
        lib.moe_slotpool_destroy.argtypes = [vp]
        lib.moe_slotpool_destroy.restype = None
        lib.moe_slotpool_request.argtypes = [vp, vp, i32, vp]
        lib.moe_store_create.argtypes = [c.c_char_p, i32, i32, i32, i32, i32]
        lib.moe_store_write_layer.argtypes = [c.c_char_p, i32, vp, sz]
        lib.moe_store_info.argtypes = [c.c_char_p, c.POINTER(c.c_int32), c.POINTER(c.c_uint64)]
        lib.moe_store_read.argtypes = [c.c_char_p, i32, i32, vp, sz]
        for name in EXPORTS:
            if name not in ("moe_destroy", "moe_slotpool_destroy", "moe_blob_bytes", "moe_blob_stride",
                            "moe_last_error"):
                getattr(lib, name).restype = c.c_int
        _lib = lib
        return lib


def _check(rc: int, ctx=None) -> int:
    if rc < 0:
        msg = load_library().moe_last_error(ctx)
        raise MoeError(rc, msg.decode() if msg else "")
    return rc


def _ptr(t):
    """Device/host address of a torch tensor, numpy array, int or None."""
    if t is None:
        return None
    if isinstance(t, int):
        return t
    if isinstance(t, np.ndarray):
        if not t.flags["C_CONTIGUOUS"]:
            raise ValueError("numpy array must be C-contiguous")
        return t.ctypes.data
    if hasattr(t, "data_ptr"):
        if not t.is_contiguous():
            raise ValueError("tensor must be contiguous")
        return t.data_ptr()
    raise TypeError(f"cannot take the address of {type(t)}")


def _dev(t, dtype_name: str):
    if t is None or isinstance(t, int):
        return _ptr(t)
    if not getattr(t, "is_cuda", False):
        raise ValueError("expected a CUDA tensor")
    if str(t.dtype) != "torch." + dtype_name:
        raise ValueError(f"expected torch.{dtype_name}, got {t.dtype}")
    return _ptr(t)


def _stream(s):
    if s is None:
        return None
    if isinstance(s, int):
        return s
    return s.cuda_stream


# --------------------------------------------------------------------------
# the C ABI, name for name
# --------------------------------------------------------------------------

def moe_blob_bytes(hidden: int, inter: int, bits: int) -> int:
    return int(load_library().moe_blob_bytes(hidden, inter, bits))


def moe_blob_stride(hidden: int, inter: int, bits: int) -> int:
    return int(load_library().moe_blob_stride(hidden, inter, bits))


def moe_pack_expert(hidden: int, inter: int, bits: int, expert: dict, out: np.ndarray | None = None) -> np.ndarray:
    """Pack one expert's quantised arrays (dict q_gate, sb_gate, q_up, sb_up,
    q_down, sb_down as produced by the input generator) into its blob."""
    stride = moe_blob_stride(hidden, inter, bits)
    if out is None:
        out = np.empty(stride, np.uint8)
    arrs = [np.ascontiguousarray(expert[k]) for k in ("q_gate", "sb_gate", "q_up", "sb_up", "q_down", "sb_down")]
    _check(load_library().moe_pack_expert(hidden, inter, bits, *[a.ctypes.data for a in arrs], _ptr(out),
                                          out.nbytes))
    return out


def moe_create(cfg: moe_config):
    h = ctypes.c_void_p()
    _check(load_library().moe_create(ctypes.byref(cfg), ctypes.byref(h)))
    return h.value


def moe_destroy(ctx) -> None:
    if ctx:
        load_library().moe_destroy(ctx)


def moe_load_experts(ctx, layer: int, blobs, stride: int, shared_blob, router_w, shared_gate_w, router_bias=None):
    """blobs: host uint8 [n_experts * stride]; shared_blob: host uint8; router_w,
    shared_gate_w: host uint16 bf16 bits; router_bias: host fp32 or None."""
    _check(load_library().moe_load_experts(ctx, layer, _ptr(blobs), stride, _ptr(shared_blob), _ptr(router_w),
                                           _ptr(shared_gate_w), _ptr(router_bias)), ctx)


def moe_set_router_bias(ctx, layer: int, bias_host, stream=None):
    _check(load_library().moe_set_router_bias(ctx, layer, _ptr(bias_host), _stream(stream)), ctx)


def moe_set_router_bias_all(ctx, bias_host, stream=None):
    """bias_host: contiguous fp32 host array [n_layers, n_experts]."""
    _check(load_library().moe_set_router_bias_all(ctx, _ptr(bias_host), _stream(stream)), ctx)


def moe_forward_decode(ctx, layer: int, x, B: int, y, topk_idx=None, topk_w=None, stream=None):
    _check(load_library().moe_forward_decode(ctx, layer, _dev(x, "float32"), B, _dev(y, "float32"),
                                             _dev(topk_idx, "int32"), _dev(topk_w, "float32"), _stream(stream)), ctx)


def moe_forward_decode_stack(ctx, layer0: int, n_layers: int, x, B: int, y, renorm_eps: float = 1e-6,
                             x_trace=None, idx_trace=None, y_trace=None, stream=None):
    _check(load_library().moe_forward_decode_stack(ctx, layer0, n_layers, _dev(x, "float32"), B,
                                                   _dev(y, "float32"), renorm_eps, _dev(x_trace, "float32"),
                                                   _dev(idx_trace, "int32"), _dev(y_trace, "float32"),
                                                   _stream(stream)), ctx)


def moe_forward_prefill(ctx, layer: int, x, T: int, y, topk_idx=None, topk_w=None, stream=None):
    _check(load_library().moe_forward_prefill(ctx, layer, _dev(x, "float32"), T, _dev(y, "float32"),
                                              _dev(topk_idx, "int32"), _dev(topk_w, "float32"), _stream(stream)),
           ctx)


def moe_route_noalloc(ctx, layer: int, x, B: int, topk_idx, topk_w, stream=None):
    _check(load_library().moe_route_noalloc(ctx, layer, _dev(x, "float32"), B, _dev(topk_idx, "int32"),
                                            _dev(topk_w, "float32"), _stream(stream)), ctx)


def moe_pool_reset(ctx, slots: int, policy: int = MOE_EVICT_LFU_RECENCY, aging_period: int = 0, stream=None) -> None:
    """Empty every layer's pool, use `slots` of the reserved slots and evict by `policy` (streaming contexts)."""
    _check(load_library().moe_pool_reset(ctx, slots, policy, aging_period, _stream(stream)), ctx)


def moe_pool_stats(ctx, layer: int = -1) -> dict:
    s = moe_pool_stats_t()
    _check(load_library().moe_pool_stats(ctx, layer, ctypes.byref(s)), ctx)
    return {f: getattr(s, f) for f, _ in s._fields_}


def moe_pool_trace(ctx) -> np.ndarray:
    n = ctypes.c_size_t()
    lib = load_library()
    _check(lib.moe_pool_trace(ctx, None, 0, ctypes.byref(n)), ctx)
    buf = np.empty((n.value, 6), np.int32)
    _check(lib.moe_pool_trace(ctx, _ptr(buf) if n.value else None, n.value, ctypes.byref(n)), ctx)
    return buf


PREFILL_KERNELS = ("router_logits", "select", "histogram", "scan", "scatter", "gather_x", "gateup_gemm", "down_gemm")


def moe_prefill_profile(ctx, enable: bool = True) -> None:
    _check(load_library().moe_prefill_profile(ctx, int(bool(enable))), ctx)


def moe_prefill_kernel_ms(ctx) -> tuple:
    """-> ({kernel name: accumulated device ms}, recorded calls)"""
    ms = (ctypes.c_double * len(PREFILL_KERNELS))()
    n = ctypes.c_int64()
    _check(load_library().moe_prefill_kernel_ms(ctx, ms, ctypes.byref(n)), ctx)
    return dict(zip(PREFILL_KERNELS, list(ms))), n.value


def moe_launch_count(ctx) -> int:
    n = ctypes.c_uint64()
    _check(load_library().moe_launch_count(ctx, ctypes.byref(n)), ctx)
    return int(n.value)


def moe_last_error(ctx=None) -> str:
    m = load_library().moe_last_error(ctx)
    return m.decode() if m else ""


def moe_slotpool_create(slots: int, n_experts: int, policy: int = MOE_EVICT_LFU_RECENCY, aging_period: int = 0):
    h = ctypes.c_void_p()
    _check(load_library().moe_slotpool_create(slots, n_experts, policy, aging_period, ctypes.byref(h)))
    return h.value


def moe_slotpool_destroy(pool) -> None:
    if pool:
        load_library().moe_slotpool_destroy(pool)


def moe_slotpool_request(pool, req) -> list:
    """req: distinct ascending expert ids -> [(expert, kind, slot, evicted)]."""
    r = np.ascontiguousarray(req, np.int32)
    ev = np.empty((max(len(r), 1), 4), np.int32)
    n = _check(load_library().moe_slotpool_request(pool, _ptr(r) if len(r) else None, len(r), _ptr(ev)))
    return [tuple(int(v) for v in ev[i]) for i in range(n)]


def make_config(n_layers, hidden, n_experts, top_k, inter, shared_inter, bits=4, pool_slots=None, norm_topk=True,
                policy=MOE_EVICT_LFU_RECENCY, device=0, max_batch=1, max_tokens=0, fault_flags=0, fault_arg=0,
                timeout_ms=0, aging_period=0, store_path=None, store_flags=0, layer_bits=None) -> moe_config:
    """store_path: an expert container (moe_store_create) for a streaming context;
    layer_bits: 4 or 8 per layer (a mixed store).  The library copies both at
    moe_create; until then the struct keeps the Python-side buffers alive."""
    lb = None
    if layer_bits is not None:
        lb = (ctypes.c_int32 * len(layer_bits))(*[int(b) for b in layer_bits])
    cfg = moe_config(n_layers, hidden, n_experts, top_k, inter, shared_inter, bits, 64,
                     n_experts if pool_slots is None else pool_slots, int(norm_topk), policy, device, max_batch,
                     max_tokens, fault_flags, fault_arg, timeout_ms, aging_period, store_flags,
                     os.fsencode(store_path) if store_path is not None else None,
                     ctypes.cast(lb, ctypes.POINTER(ctypes.c_int32)) if lb is not None else None)
    cfg._layer_bits = lb  # keeps the array alive with the struct
    return cfg


# --------------------------------------------------------------------------
# expert container (routed blobs on disk; host only)
# --------------------------------------------------------------------------

def moe_store_create(path, n_layers: int, n_experts: int, hidden: int, inter: int, bits: int) -> None:
    _check(load_library().moe_store_create(os.fsencode(path), n_layers, n_experts, hidden, inter, bits))


def moe_store_write_layer(path, layer: int, blobs, stride: int) -> None:
    """blobs: host uint8 [n_experts * stride] (the layer's packed routed blobs)."""
    b = np.ascontiguousarray(blobs, np.uint8)
    _check(load_library().moe_store_write_layer(os.fsencode(path), layer, _ptr(b), stride))


def moe_store_info(path) -> dict:
    shape = (ctypes.c_int32 * 5)()
    stride = ctypes.c_uint64()
    _check(load_library().moe_store_info(os.fsencode(path), shape, ctypes.byref(stride)))
    return dict(zip(("n_layers", "n_experts", "hidden", "inter", "bits"), list(shape)), stride=stride.value)


def moe_store_read(path, layer: int, expert: int, stride: int) -> np.ndarray:
    out = np.empty(stride, np.uint8)
    _check(load_library().moe_store_read(os.fsencode(path), layer, expert, _ptr(out), stride))
    return out
