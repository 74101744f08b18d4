"""ORACLE — test infrastructure, not the product.

Python face of ``oracle.c``: a plain single-threaded fp32 CPU implementation of
the routed MoE layer (router softmax + top-k + renormalisation, permutation by
expert, SwiGLU experts over dequantised weights, gate-weighted combine) and of
the LRU expert cache that feeds it. Only ``tests/``, ``__graft_entry__.smoke()``
and ``bench.py``'s CPU-baseline leg may import it. It shares no code with the
CUDA library and never receives a value computed by it.

The sources each function follows are cited in ``oracle.c``.
"""
from __future__ import annotations

import ctypes
import os
import subprocess

import numpy as np

_HERE = os.path.dirname(os.path.abspath(__file__))
_SO = os.path.join(_HERE, "liboracle.so")
_lib = None

FP32, BF16, NVFP4, MXFP4, FP8 = 0, 1, 2, 3, 4
DECODE_MAX_T = 8


def build(force: bool = False) -> str:
    src = os.path.join(_HERE, "oracle.c")
    if force or not os.path.exists(_SO) or os.path.getmtime(_SO) < os.path.getmtime(src):
        subprocess.check_call(["gcc", "-O2", "-ffp-contract=off", "-fno-fast-math", "-fPIC",
                               "-shared", "-o", _SO, src, "-lm"])
    return _SO


def _L():
    global _lib
    if _lib is None:
        build()
        lib = ctypes.CDLL(_SO)
        vp, i32, f32, sz = ctypes.c_void_p, ctypes.c_int, ctypes.c_float, ctypes.c_size_t
        lib.orc_e2m1.restype = f32
        lib.orc_e2m1.argtypes = [ctypes.c_uint]
        lib.orc_e4m3fn.restype = f32
        lib.orc_e4m3fn.argtypes = [ctypes.c_uint]
        lib.orc_e8m0.restype = f32
        lib.orc_e8m0.argtypes = [ctypes.c_uint]
        lib.orc_bf16.restype = f32
        lib.orc_bf16.argtypes = [ctypes.c_uint16]
        lib.orc_bf16_rne.restype = ctypes.c_uint16
        lib.orc_bf16_rne.argtypes = [f32]
        lib.orc_bf16_to_f32.argtypes = [vp, sz, vp]
        lib.orc_f32_to_bf16.argtypes = [vp, sz, vp]
        lib.orc_dequant.argtypes = [i32, vp, vp, f32, i32, i32, vp]
        lib.orc_e4m3_rne.restype = f32
        lib.orc_e4m3_rne.argtypes = [f32]
        lib.orc_e2m1_rne.restype = f32
        lib.orc_e2m1_rne.argtypes = [f32]
        lib.orc_quant_act.argtypes = [i32, vp, i32, vp]
        lib.orc_expert_ffn_q.argtypes = [vp, vp, vp, vp, i32, i32, i32, i32, vp]
        lib.orc_router_logits.argtypes = [vp, vp, i32, i32, i32, vp]
        lib.orc_router_topk.argtypes = [vp, i32, i32, i32, vp, vp, vp]
        lib.orc_permute.restype = i32
        lib.orc_permute.argtypes = [vp, i32, i32, i32, vp, vp, vp, vp, vp]
        lib.orc_lru_batch.restype = i32
        lib.orc_lru_batch.argtypes = [i32, i32, i32, vp, vp, vp, vp, i32, vp, i32, vp, i32,
                                      vp, vp, vp, vp]
        lib.orc_expert_ffn.argtypes = [vp, vp, vp, vp, i32, i32, i32, vp, vp]
        lib.orc_layer_tokens.argtypes = [vp, i32, i32, i32, i32, i32, i32, vp, vp, vp, vp, vp,
                                         vp, i32, vp]
        lib.orc_combine.argtypes = [i32, i32, i32, vp, vp, vp]
        lib.orc_lru_resize.restype = i32
        lib.orc_lru_resize.argtypes = [i32, i32, i32, vp, vp, vp, i32, vp, vp, vp]
        _lib = lib
    return _lib


def _p(a):
    return None if a is None else ctypes.c_void_p(a.ctypes.data)


def _c(a, dt):
    return np.ascontiguousarray(a, dtype=dt)


# --------------------------------------------------------------------------- codecs

def e2m1(code: int) -> float:
    return float(_L().orc_e2m1(code))


def e4m3fn(b: int) -> float:
    return float(_L().orc_e4m3fn(b))


def e8m0(b: int) -> float:
    return float(_L().orc_e8m0(b))


def bf16_to_f32(bits) -> np.ndarray:
    bits = _c(bits, np.uint16)
    out = np.empty(bits.shape, dtype=np.float32)
    _L().orc_bf16_to_f32(_p(bits), bits.size, _p(out))
    return out


def f32_to_bf16(x) -> np.ndarray:
    x = _c(x, np.float32)
    out = np.empty(x.shape, dtype=np.uint16)
    _L().orc_f32_to_bf16(_p(x), x.size, _p(out))
    return out


def dequant(fmt: int, t: dict, N: int, K: int) -> np.ndarray:
    """Dequantise one canonical tensor dict (see ``synth``) to fp32 [N, K]."""
    out = np.empty((N, K), dtype=np.float32)
    if fmt == FP32:
        data, sc, g = _c(t["data"], np.float32), None, 1.0
    elif fmt == BF16:
        data, sc, g = _c(t["data"], np.uint16), None, 1.0
    elif fmt == FP8:
        data, sc, g = _c(t["codes"], np.uint8), None, t["gscale"]
    else:
        data, sc = _c(t["codes"], np.uint8), _c(t["scales"], np.uint8)
        g = t.get("gscale", 1.0)
    _L().orc_dequant(fmt, _p(data), _p(sc), ctypes.c_float(g), N, K, _p(out))
    return out


def dequant_expert(fmt: int, w: dict, H: int, I: int):
    return (dequant(fmt, w["gate"], I, H), dequant(fmt, w["up"], I, H),
            dequant(fmt, w["down"], H, I))


# --------------------------------------------------------------------------- router

def act_to_f32(x, act_bf16: bool) -> np.ndarray:
    return bf16_to_f32(x) if act_bf16 else _c(x, np.float32)


def router_logits(x: np.ndarray, w: np.ndarray) -> np.ndarray:
    x = _c(x, np.float32)
    w = _c(w, np.float32)
    T, H = x.shape
    E = w.shape[0]
    out = np.empty((T, E), dtype=np.float32)
    _L().orc_router_logits(_p(x), _p(w), T, E, H, _p(out))
    return out


def router_topk(logits: np.ndarray, k: int, want_probs: bool = False):
    logits = _c(logits, np.float32)
    T, E = logits.shape
    idx = np.empty((T, k), dtype=np.int32)
    gates = np.empty((T, k), dtype=np.float32)
    probs = np.empty((T, E), dtype=np.float32) if want_probs else None
    _L().orc_router_topk(_p(logits), T, E, k, _p(idx), _p(gates), _p(probs))
    return (idx, gates, probs) if want_probs else (idx, gates)


def permute(idx: np.ndarray, E: int) -> dict:
    idx = _c(idx, np.int32)
    T, k = idx.shape
    n = T * k
    counts = np.empty(E, np.int32)
    offsets = np.empty(E + 1, np.int32)
    perm = np.empty(n, np.int32)
    inv = np.empty(n, np.int32)
    uniq = np.empty(E, np.int32)
    nu = _L().orc_permute(_p(idx), T, E, k, _p(counts), _p(offsets), _p(perm), _p(inv), _p(uniq))
    return {"counts": counts, "offsets": offsets, "perm": perm, "inv_perm": inv,
            "uniq": uniq[:nu].copy()}


def route(x_f32: np.ndarray, router_w_f32: np.ndarray, k: int) -> dict:
    lg = router_logits(x_f32, router_w_f32)
    idx, gates = router_topk(lg, k)
    r = permute(idx, router_w_f32.shape[0])
    r.update(logits=lg, topk_idx=idx, gates=gates)
    return r


# --------------------------------------------------------------------------- LRU

class LRU:
    """The global LRU slot pool shared by all layers (see ``orc_lru_batch``).

    ``access(layer, uniq, T, prefetch)`` applies one forward call's batches:
    the layer's own access batch, then, for a prefill call (T > 8) with
    prefetch enabled and room for it (S >= |uniq| + E, layer + 1 < L), a batch
    over all E experts of the next layer that protects this layer's experts.
    Returns the events, or raises ``CapacityError``.
    """

    class CapacityError(RuntimeError):
        pass

    def __init__(self, L: int, E: int, S: int):
        self.L, self.E, self.S = L, E, S
        self.table = np.full(L * E, -1, np.int32)
        self.owner = np.full(S, -1, np.int32)
        self.stamp = np.zeros(S, np.uint64)
        self.clock = np.zeros(1, np.uint64)

    def batch(self, layer: int, members: np.ndarray, protect_keys: np.ndarray | None = None):
        m = _c(members, np.int32)
        n = m.size
        pk = _c(protect_keys if protect_keys is not None else np.empty(0), np.int32)
        ev = [np.empty(n, np.int32) for _ in range(4)]
        r = _L().orc_lru_batch(self.L, self.E, self.S, _p(self.table), _p(self.owner),
                               _p(self.stamp), _p(self.clock), layer, _p(m), n, _p(pk), pk.size,
                               *[_p(e) for e in ev])
        if r < 0:
            raise LRU.CapacityError(f"layer {layer}: {n} experts do not fit in {self.S} slots")
        return {"expert": ev[0], "hit": ev[1], "slot": ev[2], "evicted": ev[3],
                "layer": np.full(n, layer, np.int32)}

    def resize(self, S_new: int) -> np.ndarray:
        """Resize the pool at a safe point (see ``orc_lru_resize``): the most
        recently used experts that fit stay cached. Returns moved[old slot] =
        new slot (or -1)."""
        new_owner = np.empty(S_new, np.int32)
        new_stamp = np.empty(S_new, np.uint64)
        S_old = self.S
        moved = np.empty(max(1, S_old), np.int32)
        _L().orc_lru_resize(self.L, self.E, S_old, _p(self.table), _p(self.owner), _p(self.stamp), S_new,
                            _p(new_owner), _p(new_stamp), _p(moved))
        self.owner, self.stamp, self.S = new_owner, new_stamp, S_new
        return moved[:S_old]

    def access(self, layer: int, uniq: np.ndarray, T: int, prefetch: bool):
        evs = [self.batch(layer, uniq)]
        evs[0]["prefetch"] = np.zeros(len(uniq), np.int32)
        if (prefetch and T > DECODE_MAX_T and layer + 1 < self.L
                and self.S >= len(uniq) + self.E):
            keys = (layer * self.E + _c(uniq, np.int32)).astype(np.int32)
            e2 = self.batch(layer + 1, np.arange(self.E, dtype=np.int32), keys)
            e2["prefetch"] = np.ones(self.E, np.int32)
            evs.append(e2)
        return {k: np.concatenate([e[k] for e in evs]) for k in evs[0]}


# --------------------------------------------------------------------------- experts / layer

def expert_ffn(x: np.ndarray, Wg, Wu, Wd, mode: int = 0):
    x = _c(x, np.float32)
    H = x.size
    I = Wg.shape[0]
    y = np.empty(H, np.float32)
    h = np.empty(I, np.float32)
    _L().orc_expert_ffn(_p(x), _p(_c(Wg, np.float32)), _p(_c(Wu, np.float32)),
                        _p(_c(Wd, np.float32)), H, I, mode, _p(y), _p(h))
    return y, h


QUANT_MXFP8, QUANT_NVFP4 = 1, 2


def e4m3_rne(v: float) -> float:
    return float(_L().orc_e4m3_rne(ctypes.c_float(v)))


def e2m1_rne(v: float) -> float:
    return float(_L().orc_e2m1_rne(ctypes.c_float(v)))


def quant_act(kind: int, x: np.ndarray) -> np.ndarray:
    """Activation quantiser of a block-scaled MMA (see orc_quant_act)."""
    x = _c(x, np.float32)
    out = np.empty_like(x)
    _L().orc_quant_act(kind, _p(x), x.size, _p(out))
    return out


def expert_ffn_q(x: np.ndarray, Wg, Wu, Wd, kind: int, mode: int = 0) -> np.ndarray:
    """expert_ffn with x and h quantised by quant_act(kind)."""
    x = _c(x, np.float32)
    H = x.size
    I = Wg.shape[0]
    y = np.empty(H, np.float32)
    _L().orc_expert_ffn_q(_p(x), _p(_c(Wg, np.float32)), _p(_c(Wu, np.float32)),
                          _p(_c(Wd, np.float32)), H, I, mode, kind, _p(y))
    return y


def combine(gates_row: np.ndarray, ys) -> np.ndarray:
    """One token's layer output from its k routed expert outputs ``ys[:k]``
    (in selection order) and its shared expert outputs ``ys[k:]``."""
    g = _c(gates_row, np.float32)
    k = g.size
    rows = [_c(y, np.float32) for y in ys]
    H = rows[0].size
    arr = (ctypes.c_void_p * len(rows))(*[r.ctypes.data for r in rows])
    out = np.empty(H, np.float32)
    _L().orc_combine(H, k, len(rows) - k, _p(g), arr, _p(out))
    return out


def layer_tokens(x_f32: np.ndarray, idx: np.ndarray, gates: np.ndarray, weights: dict,
                 E: int, n_shared: int, mode: int, toks) -> np.ndarray:
    """fp32 layer output rows for tokens ``toks``. ``weights[e] = (Wg, Wu, Wd)``
    (dequantised fp32) for every routed expert those tokens use and every shared
    expert (ids E..E+n_shared-1)."""
    x = _c(x_f32, np.float32)
    T, H = x.shape
    k = idx.shape[1]
    any_w = next(iter(weights.values()))
    I = any_w[0].shape[0]
    n = E + n_shared
    keep = []
    arrs = [(ctypes.c_void_p * n)() for _ in range(3)]
    for e, ws in weights.items():
        for j in range(3):
            a = _c(ws[j], np.float32)
            keep.append(a)
            arrs[j][e] = a.ctypes.data
    toks = _c(np.asarray(toks), np.int32)
    out = np.empty((toks.size, H), np.float32)
    _L().orc_layer_tokens(_p(x), H, I, E, n_shared, k, mode, _p(_c(idx, np.int32)),
                          _p(_c(gates, np.float32)), arrs[0], arrs[1], arrs[2], _p(toks),
                          toks.size, _p(out))
    return out


def layer(shape, experts: dict, router_w, hidden, toks=None) -> dict:
    """One call of the layer on canonical inputs (``synth`` encodings).

    ``experts[e]`` is the canonical weight dict of expert e; only experts that
    the routed tokens select (and the shared ones) are dequantised. Returns the
    routing and ``out`` (fp32 rows for ``toks``, default all tokens).
    """
    act_bf16 = shape.act == 1
    x = act_to_f32(hidden, act_bf16)
    w = act_to_f32(router_w, act_bf16)
    r = route(x, w, shape.k)
    T = x.shape[0]
    toks = np.arange(T) if toks is None else np.asarray(toks)
    need = set(int(e) for e in np.unique(r["topk_idx"][toks]))
    need |= set(range(shape.E, shape.E + shape.shared))
    weights = {e: dequant_expert(shape.fmt, experts[e], shape.H, shape.I) for e in sorted(need)}
    r["out"] = layer_tokens(x, r["topk_idx"], r["gates"], weights, shape.E, shape.shared,
                            shape.act_mode, toks)
    r["toks"] = toks
    return r
