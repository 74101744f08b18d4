"""B300 routed Mixture-of-Experts layer with a device-side LRU expert cache.

Thin ctypes binding of the C ABI in ``include/moe.h`` (``libmoe_b300.so``,
built in-tree for sm_103a by ``expert_offload_softmax_b300.build``). The
functions keep the C names and only marshal arguments; every step of the layer
runs in the library's CUDA kernels. Device buffers are passed as integer
addresses (e.g. ``tensor.data_ptr()``) and streams as ``cudaStream_t`` handles
(``torch.cuda.Stream.cuda_stream``); nothing here depends on torch.

If the library is missing this module raises on import of the library
(``load()``): there is no CPU fallback.
"""
from __future__ import annotations

import ctypes
import os

import numpy as np

_HERE = os.path.dirname(os.path.abspath(__file__))
LIB_PATH = os.path.join(_HERE, "libmoe_b300.so")

MOE_OK, MOE_ERR_INVALID, MOE_ERR_OOM, MOE_ERR_CUDA = 0, -1, -2, -3
MOE_ERR_CAPACITY, MOE_ERR_TIMEOUT, MOE_ERR_STATE = -4, -5, -6
MOE_FMT_FP32, MOE_FMT_BF16, MOE_FMT_NVFP4, MOE_FMT_MXFP4, MOE_FMT_FP8 = 0, 1, 2, 3, 4
MOE_ACT_FP32, MOE_ACT_BF16 = 0, 1
MOE_MODE_SWIGLU, MOE_MODE_LINEAR_TEST = 0, 1
MOE_DECODE_MAX_T = 8
MOE_CACHE_PREFETCH_NEXT_LAYER = 1
MOE_CACHE_LOG_EVENTS = 2
MOE_CACHE_SYNC_MISSES = 4
MOE_CACHE_HOST_MISSES = 8

# every symbol the header declares
EXPORTS = ["moe_init", "moe_expert_bytes", "moe_repack_expert", "moe_load_expert", "moe_cache_config",
           "moe_cache_resize", "moe_layer_forward", "moe_sync",
           "moe_stats", "moe_stats_reset", "moe_stats_events", "moe_debug_routing", "moe_debug_lru_table",
           "moe_last_error", "moe_destroy", "moe_timing_enable", "moe_timing", "moe_route_topk_noalloc"]
MOE_ROUTE_NOALLOC_MAX_LOGITS = 1 << 20


class moe_model_desc(ctypes.Structure):
    _fields_ = [(n, ctypes.c_int32) for n in (
        "num_layers", "num_experts", "num_shared", "top_k", "hidden", "inter", "weight_fmt",
        "act_dtype", "act_mode", "max_tokens", "device")]


class moe_tensor_host(ctypes.Structure):
    _fields_ = [("data", ctypes.c_void_p), ("scales", ctypes.c_void_p), ("global_scale", ctypes.c_float)]


class moe_expert_host(ctypes.Structure):
    _fields_ = [("gate", moe_tensor_host), ("up", moe_tensor_host), ("down", moe_tensor_host)]


class moe_stats_t(ctypes.Structure):
    _fields_ = [(n, ctypes.c_uint64) for n in (
        "calls", "decode_calls", "prefill_calls", "hits", "misses", "prefetch_hits", "prefetch_misses",
        "evictions", "copies_h2d", "bytes_h2d", "device_errors", "kernel_launches")]

    def as_dict(self):
        return {n: int(getattr(self, n)) for n, _ in self._fields_}


class moe_timing_t(ctypes.Structure):
    _fields_ = [("calls", ctypes.c_uint64)] + [(n, ctypes.c_double) for n in (
        "route_ms", "gate_up_ms", "down_ms", "combine_ms", "copy_ms")] + [(n, ctypes.c_uint64) for n in (
        "gate_up_bytes", "down_bytes", "combine_bytes", "copy_bytes", "resident_calls")]

    def as_dict(self):
        return {n: (float(getattr(self, n)) if t is ctypes.c_double else int(getattr(self, n)))
                for n, t in self._fields_}


class moe_event(ctypes.Structure):
    _fields_ = [(n, ctypes.c_int32) for n in ("layer", "expert", "hit", "slot", "evicted_key", "prefetch")]


class MoeError(RuntimeError):
    def __init__(self, code, msg):
        super().__init__(f"{msg} (status {code})")
        self.code = code


_lib = None


def load(path: str | None = None):
    """Loads libmoe_b300.so (raises if it has not been built)."""
    global _lib
    if _lib is not None:
        return _lib
    p = path or LIB_PATH
    if not os.path.exists(p):
        raise ImportError(f"{p} is missing: build it with `python -m expert_offload_softmax_b300.build`")
    lib = ctypes.CDLL(p)
    vp, i32, u32 = ctypes.c_void_p, ctypes.c_int, ctypes.c_uint
    P = ctypes.POINTER
    lib.moe_init.argtypes = [P(moe_model_desc), P(vp)]
    lib.moe_expert_bytes.argtypes = [P(moe_model_desc), P(ctypes.c_size_t)]
    lib.moe_repack_expert.argtypes = [P(moe_model_desc), P(moe_expert_host), ctypes.c_void_p, ctypes.c_size_t]
    lib.moe_load_expert.argtypes = [vp, i32, i32, P(moe_expert_host)]
    lib.moe_cache_config.argtypes = [vp, i32, u32, vp, ctypes.c_size_t]
    lib.moe_cache_resize.argtypes = [vp, i32, vp, ctypes.c_size_t]
    lib.moe_layer_forward.argtypes = [vp, vp, vp, i32, i32, vp, vp]
    lib.moe_sync.argtypes = [vp]
    lib.moe_stats.argtypes = [vp, P(moe_stats_t)]
    lib.moe_stats_reset.argtypes = [vp]
    lib.moe_timing_enable.argtypes = [vp, i32]
    lib.moe_timing.argtypes = [vp, P(moe_timing_t)]
    lib.moe_stats_events.argtypes = [vp, P(moe_event), i32, P(i32)]
    lib.moe_debug_routing.argtypes = [vp, vp, vp, vp, vp, vp, P(ctypes.c_int32)]
    lib.moe_debug_lru_table.argtypes = [vp, vp]
    lib.moe_route_topk_noalloc.argtypes = [vp, vp, i32, i32, i32, i32, i32, vp, vp, vp]
    lib.moe_last_error.argtypes = [vp]
    lib.moe_last_error.restype = ctypes.c_char_p
    lib.moe_destroy.argtypes = [vp]
    lib.moe_destroy.restype = None
    for name in EXPORTS:
        if name not in ("moe_last_error", "moe_destroy"):
            getattr(lib, name).restype = ctypes.c_int
    _lib = lib
    return lib


def _check(h, rc):
    if rc != MOE_OK:
        msg = load().moe_last_error(h).decode() if h else "moe call failed"
        raise MoeError(rc, msg)


def _np_ptr(a):
    return None if a is None else ctypes.c_void_p(a.ctypes.data)


# --------------------------------------------------------------------------- C names

def moe_init(desc: moe_model_desc) -> int:
    h = ctypes.c_void_p()
    rc = load().moe_init(ctypes.byref(desc), ctypes.byref(h))
    if rc != MOE_OK:
        raise MoeError(rc, "moe_init failed")
    return h.value


def moe_expert_bytes(desc: moe_model_desc) -> int:
    n = ctypes.c_size_t()
    rc = load().moe_expert_bytes(ctypes.byref(desc), ctypes.byref(n))
    if rc != MOE_OK:
        raise MoeError(rc, "moe_expert_bytes failed")
    return n.value


def _tensor(t: dict) -> moe_tensor_host:
    data = t["data"] if "data" in t else t["codes"]
    data = np.ascontiguousarray(data)
    sc = np.ascontiguousarray(t["scales"]) if "scales" in t else None
    th = moe_tensor_host(data.ctypes.data, None if sc is None else sc.ctypes.data, float(t.get("gscale", 1.0)))
    return th, (data, sc)


def moe_repack_expert(desc: moe_model_desc, w: dict) -> np.ndarray:
    """The device-layout blob (uint8, moe_expert_bytes long) of canonical weights w. Host only."""
    g, kg = _tensor(w["gate"])
    u, ku = _tensor(w["up"])
    d, kd = _tensor(w["down"])
    eh = moe_expert_host(g, u, d)
    blob = np.empty(moe_expert_bytes(desc), np.uint8)
    rc = load().moe_repack_expert(ctypes.byref(desc), ctypes.byref(eh), blob.ctypes.data, blob.size)
    del kg, ku, kd
    if rc != MOE_OK:
        raise MoeError(rc, "moe_repack_expert failed")
    return blob


def moe_load_expert(h: int, layer: int, expert: int, w: dict) -> None:
    """w: canonical weights {gate, up, down} -> {data | codes, scales, gscale} (numpy)."""
    g, kg = _tensor(w["gate"])
    u, ku = _tensor(w["up"])
    d, kd = _tensor(w["down"])
    eh = moe_expert_host(g, u, d)
    _check(h, load().moe_load_expert(h, layer, expert, ctypes.byref(eh)))
    del kg, ku, kd


def moe_cache_config(h: int, capacity_slots: int, flags: int = 0, pool_dev: int = 0, pool_bytes: int = 0) -> None:
    """Safe point: (re)build an empty cache of capacity_slots slots. pool_dev:
    optional caller-owned device buffer (address) of pool_bytes bytes."""
    _check(h, load().moe_cache_config(h, capacity_slots, flags, pool_dev or None, pool_bytes))


def moe_cache_resize(h: int, capacity_slots: int, pool_dev: int = 0, pool_bytes: int = 0) -> None:
    """Safe point: resize the cache, keeping the most recently used experts."""
    _check(h, load().moe_cache_resize(h, capacity_slots, pool_dev or None, pool_bytes))


def moe_layer_forward(h: int, hidden: int, router_w: int, layer_id: int, T: int, out: int,
                      stream: int | None = None) -> None:
    _check(h, load().moe_layer_forward(h, hidden, router_w, layer_id, T, out, stream))


def moe_sync(h: int) -> None:
    """Waits for every enqueued call; raises the first error found for any of them."""
    _check(h, load().moe_sync(h))


def moe_stats(h: int) -> dict:
    s = moe_stats_t()
    _check(h, load().moe_stats(h, ctypes.byref(s)))
    return s.as_dict()


def moe_timing_enable(h: int, enable: bool = True) -> None:
    _check(h, load().moe_timing_enable(h, 1 if enable else 0))


def moe_timing(h: int) -> dict:
    t = moe_timing_t()
    _check(h, load().moe_timing(h, ctypes.byref(t)))
    return t.as_dict()


def moe_stats_reset(h: int) -> None:
    _check(h, load().moe_stats_reset(h))


def moe_stats_events(h: int, cap: int = 8192) -> np.ndarray:
    """Drains the event log: int32 array [n, 6] (layer, expert, hit, slot, evicted_key, prefetch)."""
    buf = (moe_event * cap)()
    n = ctypes.c_int()
    _check(h, load().moe_stats_events(h, buf, cap, ctypes.byref(n)))
    arr = np.frombuffer(buf, dtype=np.int32, count=n.value * 6).reshape(n.value, 6)
    return arr.copy()


def moe_debug_routing(h: int, T: int, k: int, E: int) -> dict:
    topk = np.empty(T * k, np.int32)
    gates = np.empty(T * k, np.float32)
    perm = np.empty(T * k, np.int32)
    counts = np.empty(E, np.int32)
    uniq = np.empty(E, np.int32)
    nu = ctypes.c_int32()
    _check(h, load().moe_debug_routing(h, _np_ptr(topk), _np_ptr(gates), _np_ptr(perm), _np_ptr(counts),
                                       _np_ptr(uniq), ctypes.byref(nu)))
    return {"topk_idx": topk.reshape(T, k), "gates": gates.reshape(T, k), "perm": perm, "counts": counts,
            "uniq": uniq[:nu.value].copy()}


def moe_debug_lru_table(h: int, L: int, E: int) -> np.ndarray:
    t = np.empty(L * E, np.int32)
    _check(h, load().moe_debug_lru_table(h, _np_ptr(t)))
    return t


def moe_route_topk_noalloc(hidden: int, router_w: int, T: int, E: int, H: int, k: int, act_dtype: int,
                           topk_idx: int, gates: int, stream: int | None = None) -> None:
    """Router top-k into caller-provided device outputs; allocates nothing (for
    callers that cannot call cudaMalloc). Pointers are device addresses."""
    rc = load().moe_route_topk_noalloc(hidden, router_w, T, E, H, k, act_dtype, topk_idx, gates, stream)
    if rc != MOE_OK:
        raise MoeError(rc, "moe_route_topk_noalloc failed")


def moe_last_error(h: int) -> str:
    return load().moe_last_error(h).decode()


def moe_destroy(h: int) -> None:
    if h:
        load().moe_destroy(h)


def make_desc(L, E, k, H, I, fmt, act, shared=0, mode=0, max_tokens=0, device=0) -> moe_model_desc:
    return moe_model_desc(L, E, shared, k, H, I, fmt, act, mode, max_tokens, device)
