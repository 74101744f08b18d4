"""Seeded synthetic inputs for the routed MoE layer.

One module serves the oracle tests, the CUDA path's tests, ``smoke()`` and
``bench.py`` with byte-identical inputs. It holds none of the layer's
arithmetic: it draws counter-based random numbers (``synth.c``) and maps them
through value or code tables built here. Weight tensors are produced directly
in their storage encodings (packed 4-bit codes, scale bytes, a per-tensor fp32
scale) from fixed code histograms, so nothing here decodes a weight format.

Canonical host layout of one expert (what both the oracle and the library's
loader consume):

* ``gate`` and ``up``: ``[I, H]`` (row = output unit, K = H contiguous)
* ``down``: ``[H, I]`` (K = I contiguous)
* fp32: float32 rows; bf16: uint16 bit patterns
* NVFP4 / MXFP4: ``codes`` uint8 ``[N, K/2]`` with element 2i in the low nibble
  of byte i; ``scales`` uint8 ``[N, K/16]`` (E4M3 bytes, NVFP4) or
  ``[N, K/32]`` (E8M0 bytes, MXFP4); NVFP4 also has one fp32 ``gscale``.
* FP8: ``codes`` uint8 ``[N, K]``, one E4M3 (FN) byte per element, and one
  fp32 ``gscale`` per tensor.
"""
from __future__ import annotations

import ctypes
import math
import os
import subprocess
from dataclasses import dataclass, field

import numpy as np

_HERE = os.path.dirname(os.path.abspath(__file__))
_SO = os.path.join(_HERE, "libsynth.so")
_lib = None

FMT_FP32, FMT_BF16, FMT_NVFP4, FMT_MXFP4, FMT_FP8 = 0, 1, 2, 3, 4
FMT_NAMES = {"fp32": FMT_FP32, "bf16": FMT_BF16, "nvfp4": FMT_NVFP4, "mxfp4": FMT_MXFP4, "fp8": FMT_FP8}
ACT_FP32, ACT_BF16 = 0, 1

# tensor tags inside a (layer, expert) key
TAG_GATE, TAG_UP, TAG_DOWN = 0, 1, 2
PART_DATA, PART_SCALE, PART_GSCALE = 0, 1, 2
TAG_ROUTER, TAG_HIDDEN, TAG_RANK, TAG_REUSE = 100, 200, 300, 400


def build(force: bool = False) -> str:
    src = os.path.join(_HERE, "synth.c")
    if force or not os.path.exists(_SO) or os.path.getmtime(_SO) < os.path.getmtime(src):
        subprocess.check_call(["gcc", "-O2", "-fPIC", "-shared", "-o", _SO, src, "-lpthread"])
    return _SO


def _L():
    global _lib
    if _lib is None:
        build()
        lib = ctypes.CDLL(_SO)
        u64, sz, vp, i32 = ctypes.c_uint64, ctypes.c_size_t, ctypes.c_void_p, ctypes.c_int
        lib.synth_key.restype = u64
        lib.synth_key.argtypes = [u64, u64, u64, u64]
        lib.synth_word.restype = u64
        lib.synth_word.argtypes = [u64, u64]
        lib.synth_fill_tab16_u16.argtypes = [vp, sz, u64, vp, i32]
        lib.synth_fill_tab16_f32.argtypes = [vp, sz, u64, vp, i32]
        lib.synth_fill_nibbles.argtypes = [vp, sz, u64, vp, i32]
        lib.synth_fill_bytes.argtypes = [vp, sz, u64, ctypes.c_uint, ctypes.c_uint, i32]
        lib.synth_fill_tab8.argtypes = [vp, sz, u64, vp, i32]
        lib.synth_fill_uniform.argtypes = [vp, sz, u64]
        _lib = lib
    return _lib


def _nthreads() -> int:
    return max(1, min(32, os.cpu_count() or 1))


def key(seed: int, a: int, b: int = 0, c: int = 0) -> int:
    m = (1 << 64) - 1
    return int(_L().synth_key(seed & m, a & m, b & m, c & m))


def word(k: int, i: int) -> int:
    return int(_L().synth_word(k, i))


def _ptr(a: np.ndarray):
    return ctypes.c_void_p(a.ctypes.data)


# ---------------------------------------------------------------------------
# value and code tables
# ---------------------------------------------------------------------------

_NORMAL_F32 = None


def _normal_table() -> np.ndarray:
    """65536 quantiles of N(0, 1) at (j + 0.5) / 65536 (a 16-bit inverse-CDF table)."""
    global _NORMAL_F32
    if _NORMAL_F32 is None:
        from scipy.special import ndtri
        j = np.arange(65536, dtype=np.float64)
        _NORMAL_F32 = ndtri((j + 0.5) / 65536.0)
    return _NORMAL_F32


def f32_to_bf16_bits(x: np.ndarray) -> np.ndarray:
    """Round-to-nearest-even fp32 -> bf16 bit patterns (input preparation only)."""
    u = np.ascontiguousarray(x, dtype=np.float32).view(np.uint32).astype(np.uint64)
    r = ((u >> 16) & 1) + 0x7FFF
    return ((u + r) >> 16).astype(np.uint16)


_TABS = {}


def _tab_f32(std: float) -> np.ndarray:
    k = ("f32", std)
    if k not in _TABS:
        _TABS[k] = (_normal_table() * std).astype(np.float32)
    return _TABS[k]


def _tab_bf16(std: float) -> np.ndarray:
    k = ("bf16", std)
    if k not in _TABS:
        _TABS[k] = f32_to_bf16_bits((_normal_table() * std).astype(np.float32))
    return _TABS[k]


# Histogram of 4-bit code *indices* over 256 byte slots. The magnitude-index
# counts [22, 42, 38, 34, 44, 40, 26, 10] approximate the code frequencies of
# N(0, 1) data quantised with a per-block amax scale; non-zero indices are split
# evenly between the sign bit clear (idx) and set (idx | 8); index 0 keeps two
# slots with the sign bit set.
_MAG_COUNTS = [22, 42, 38, 34, 44, 40, 26, 10]


def _code_table() -> np.ndarray:
    if "codes" not in _TABS:
        t = []
        t += [0] * 20 + [8] * 2
        for m in range(1, 8):
            t += [m] * (_MAG_COUNTS[m] // 2) + [m | 8] * (_MAG_COUNTS[m] // 2)
        a = np.array(t, dtype=np.uint8)
        assert a.size == 256
        _TABS["codes"] = a
    return _TABS["codes"]


# Scale-byte ranges and per-tensor scale, chosen so that weights come out with a
# standard deviation of about 0.02 for the code histogram above:
# NVFP4 E4M3 bytes 0x50..0x6F, per-tensor fp32 scale ~1.56e-4 (x U[0.9, 1.1]);
# MXFP4 E8M0 bytes 118..121.
NVFP4_SCALE_BYTES = (0x50, 0x6F)
NVFP4_GSCALE = 1.561e-4
MXFP4_SCALE_BYTES = (118, 121)


def e4m3_encode_rne(v: np.ndarray) -> np.ndarray:
    """Harness quantiser for FP8 weights: non-negative values -> E4M3 (FN)
    bytes, rounded to nearest (ties to even) and saturated at 448. Exponent e
    (bias 7) and 3 mantissa bits; below 2^-6 the code is subnormal, m * 2^-9.
    Used only to build the FP8 code table below."""
    v = np.asarray(v, np.float64)
    assert np.all(v >= 0)
    out = np.zeros(v.shape, np.int64)
    sub = v < 2.0 ** -6
    out[sub] = np.rint(v[sub] / 2.0 ** -9).astype(np.int64)  # 8 carries into exponent 1
    e = np.floor(np.log2(np.where(sub, 1.0, v))).astype(np.int64)
    m = np.rint((np.where(sub, 1.0, v) / 2.0 ** e - 1.0) * 8).astype(np.int64)
    out[~sub] = ((e + 7) * 8 + m)[~sub]  # m = 8 carries into the next exponent
    return np.minimum(out, 0x7E).astype(np.uint8)


# FP8 weights: each byte is a draw from 256 E4M3 codes, the RNE encodings of the
# N(0, 1) quantiles at (j + 0.5) / 256 scaled so that the largest is 448 (the
# E4M3 maximum); the sign bit of the lower half set. With the per-tensor scale
# below the weights come out with a standard deviation of about 0.02.
FP8_QMAX = 448.0


def _fp8_table() -> np.ndarray:
    if "fp8" not in _TABS:
        q = _normal_table()[128::256].astype(np.float64)  # 256 quantiles, ascending
        mag = e4m3_encode_rne(np.abs(q) * (FP8_QMAX / np.abs(q).max()))
        _TABS["fp8"] = np.where(q < 0, mag | 0x80, mag).astype(np.uint8)
    return _TABS["fp8"]


def fp8_gscale(std: float) -> float:
    """Per-tensor scale that maps the FP8 code table to weights of std ~ ``std``."""
    q = _normal_table()[128::256].astype(np.float64)
    return std * np.abs(q).max() / FP8_QMAX


# Test-only block-scale tables: every finite E4M3 byte (all but the two NaN
# codes 0x7F, 0xFF: subnormals, zeros and negative scales included), and E8M0
# exponent bytes 100..154 (2^-27 .. 2^27).
E4M3_FINITE_BYTES = tuple(b for b in range(256) if b & 0x7F != 0x7F)
E8M0_WIDE_BYTES = tuple(range(100, 155))


# ---------------------------------------------------------------------------
# fills
# ---------------------------------------------------------------------------

def normal_f32(k: int, n: int, std: float) -> np.ndarray:
    out = np.empty(n, dtype=np.float32)
    _L().synth_fill_tab16_f32(_ptr(out), n, k, _ptr(_tab_f32(std)), _nthreads())
    return out


def normal_bf16(k: int, n: int, std: float, out: np.ndarray | None = None) -> np.ndarray:
    if out is None:
        out = np.empty(n, dtype=np.uint16)
    _L().synth_fill_tab16_u16(_ptr(out), n, k, _ptr(_tab_bf16(std)), _nthreads())
    return out


def code_bytes(k: int, n: int, out: np.ndarray | None = None) -> np.ndarray:
    if out is None:
        out = np.empty(n, dtype=np.uint8)
    _L().synth_fill_nibbles(_ptr(out), n, k, _ptr(_code_table()), _nthreads())
    return out


def fp8_bytes(k: int, n: int) -> np.ndarray:
    out = np.empty(n, dtype=np.uint8)
    _L().synth_fill_tab8(_ptr(out), n, k, _ptr(_fp8_table()), _nthreads())
    return out


def range_bytes(k: int, n: int, lo: int, hi: int) -> np.ndarray:
    out = np.empty(n, dtype=np.uint8)
    _L().synth_fill_bytes(_ptr(out), n, k, lo, hi, _nthreads())
    return out


def uniform(k: int, n: int) -> np.ndarray:
    out = np.empty(n, dtype=np.float64)
    _L().synth_fill_uniform(_ptr(out), n, k)
    return out


# ---------------------------------------------------------------------------
# model shapes and workloads
# ---------------------------------------------------------------------------

@dataclass
class Shape:
    """Shape and storage of one MoE layer stack."""
    name: str
    L: int          # MoE layers
    E: int          # routed experts per layer
    k: int          # experts per token
    H: int          # hidden size
    I: int          # SwiGLU intermediate size
    fmt: int        # expert weight format (FMT_*)
    act: int        # activation dtype (ACT_*)
    shared: int = 0  # always-on shared experts per layer
    w_std: float = 0.02
    router_std: float = 0.02
    zipf_s: float = 0.0  # router skew exponent (0 = none)
    act_mode: int = 0    # 0 = SwiGLU, 1 = linear stand-in (closed-form tests)
    scale_table: tuple = ()  # FP4 block-scale bytes to draw from (uniformly), instead of the default range
    code_table: tuple = ()   # FP8 code bytes to draw from (uniformly), instead of the default table

    def elems_per_expert(self) -> int:
        return 3 * self.H * self.I

    def expert_bytes(self) -> int:
        """Bytes of one expert in its storage format (codes + scales)."""
        n = self.elems_per_expert()
        if self.fmt == FMT_FP32:
            return 4 * n
        if self.fmt == FMT_BF16:
            return 2 * n
        if self.fmt == FMT_NVFP4:
            return n // 2 + n // 16 + 3 * 4
        if self.fmt == FMT_FP8:
            return n + 3 * 4
        return n // 2 + n // 32


# The five workloads (sizes as stated by the method's evaluation recipe).
TINY_FP32 = Shape("tiny-1L-H64-E8-k2-I32-fp32", L=1, E=8, k=2, H=64, I=32, fmt=FMT_FP32, act=ACT_FP32)
DECODE_NVFP4 = Shape("decode-40L-H2048-E256-k8-I512-nvfp4", L=40, E=256, k=8, H=2048, I=512,
                     fmt=FMT_NVFP4, act=ACT_BF16, zipf_s=1.0)
PREFILL_BF16 = Shape("prefill-40L-H2048-E256-k8-I512-bf16", L=40, E=256, k=8, H=2048, I=512,
                     fmt=FMT_BF16, act=ACT_BF16)
LARGE_MXFP4 = Shape("large-24L-H4096-E256+1-k8-I2048-mxfp4", L=24, E=256, k=8, H=4096, I=2048,
                    fmt=FMT_MXFP4, act=ACT_BF16, shared=1)
STRESS_NVFP4 = Shape("stress-16L-H6144-E160-k8-I2048-nvfp4", L=16, E=160, k=8, H=6144, I=2048,
                     fmt=FMT_NVFP4, act=ACT_BF16, zipf_s=1.1)

# The decode and prefill stacks' shape with FP8 experts (the fourth weight format).
DECODE_FP8 = Shape("decode-40L-H2048-E256-k8-I512-fp8", L=40, E=256, k=8, H=2048, I=512,
                   fmt=FMT_FP8, act=ACT_BF16, zipf_s=1.0)
PREFILL_FP8 = Shape("prefill-40L-H2048-E256-k8-I512-fp8", L=40, E=256, k=8, H=2048, I=512,
                    fmt=FMT_FP8, act=ACT_BF16)

SHAPES = {s.name: s for s in (TINY_FP32, DECODE_NVFP4, PREFILL_BF16, LARGE_MXFP4, STRESS_NVFP4,
                              DECODE_FP8, PREFILL_FP8)}


def _tensor(shape: Shape, seed: int, layer: int, expert: int, tag: int, N: int, K: int) -> dict:
    kd = key(seed, layer, expert, tag * 4 + PART_DATA)
    if shape.fmt == FMT_FP32:
        return {"data": normal_f32(kd, N * K, shape.w_std).reshape(N, K)}
    if shape.fmt == FMT_BF16:
        return {"data": normal_bf16(kd, N * K, shape.w_std).reshape(N, K)}
    if shape.fmt == FMT_FP8:
        u = uniform(key(seed, layer, expert, tag * 4 + PART_GSCALE), 1)[0]
        g = np.float32(fp8_gscale(shape.w_std) * (0.9 + 0.2 * u))
        if shape.code_table:
            tab = np.asarray(shape.code_table, dtype=np.uint8)
            codes = tab[range_bytes(kd, N * K, 0, len(tab) - 1)].reshape(N, K)
        else:
            codes = fp8_bytes(kd, N * K).reshape(N, K)
        return {"codes": codes, "gscale": float(g)}
    codes = code_bytes(kd, N * K // 2).reshape(N, K // 2)
    ks = key(seed, layer, expert, tag * 4 + PART_SCALE)
    nblk = N * K // (16 if shape.fmt == FMT_NVFP4 else 32)
    if shape.scale_table:
        tab = np.asarray(shape.scale_table, dtype=np.uint8)
        sc = tab[range_bytes(ks, nblk, 0, len(tab) - 1)].reshape(N, -1)
    elif shape.fmt == FMT_NVFP4:
        sc = range_bytes(ks, nblk, *NVFP4_SCALE_BYTES).reshape(N, K // 16)
    else:
        sc = range_bytes(ks, nblk, *MXFP4_SCALE_BYTES).reshape(N, K // 32)
    if shape.fmt == FMT_NVFP4:
        u = uniform(key(seed, layer, expert, tag * 4 + PART_GSCALE), 1)[0]
        g = np.float32(NVFP4_GSCALE * (0.9 + 0.2 * u))
        return {"codes": codes, "scales": sc, "gscale": float(g)}
    return {"codes": codes, "scales": sc}


def expert_weights(shape: Shape, seed: int, layer: int, expert: int) -> dict:
    """Canonical weights of expert ``expert`` of ``layer`` (expert >= E: shared)."""
    H, I = shape.H, shape.I
    return {
        "gate": _tensor(shape, seed, layer, expert, TAG_GATE, I, H),
        "up": _tensor(shape, seed, layer, expert, TAG_UP, I, H),
        "down": _tensor(shape, seed, layer, expert, TAG_DOWN, H, I),
    }


def expert_ranks(shape: Shape, seed: int, layer: int) -> np.ndarray:
    """Seeded popularity rank r_e in 1..E of each routed expert of ``layer``."""
    u = uniform(key(seed, layer, TAG_RANK), shape.E)
    order = np.argsort(u, kind="stable")
    r = np.empty(shape.E, dtype=np.int64)
    r[order] = np.arange(1, shape.E + 1)
    return r


def router_weights(shape: Shape, seed: int, layer: int) -> np.ndarray:
    """Router matrix [E, H] (float32 or bf16 bits). With a Zipf exponent s > 0,
    column 0 carries -s*ln(r_e) so that, with hidden[:, 0] = 1, the routing
    prior is proportional to r_e^-s."""
    E, H = shape.E, shape.H
    kd = key(seed, layer, TAG_ROUTER)
    w = normal_f32(kd, E * H, shape.router_std).reshape(E, H)
    if shape.zipf_s > 0:
        r = expert_ranks(shape, seed, layer)
        w[:, 0] += (-shape.zipf_s * np.log(r.astype(np.float64))).astype(np.float32)
    if shape.act == ACT_BF16:
        return f32_to_bf16_bits(w)
    return w


def hidden_states(shape: Shape, seed: int, layer: int, T: int, step: int = 0) -> np.ndarray:
    """Hidden states [T, H] ~ N(0, 1) (float32 or bf16 bits)."""
    kd = key(seed, layer, TAG_HIDDEN, step)
    if shape.act == ACT_BF16:
        x = normal_bf16(kd, T * shape.H, 1.0).reshape(T, shape.H)
        if shape.zipf_s > 0:
            x[:, 0] = 0x3F80  # 1.0
        return x
    x = normal_f32(kd, T * shape.H, 1.0).reshape(T, shape.H)
    if shape.zipf_s > 0:
        x[:, 0] = 1.0
    return x


def reuse_flags(seed: int, steps: int, p: float) -> np.ndarray:
    """One Bernoulli(p) per decode step: True = every layer reuses the previous
    step's hidden states (step 0 never reuses)."""
    u = uniform(key(seed, TAG_REUSE), steps)
    f = u < p
    f[0] = False
    return f


def capacity_slots(shape: Shape, frac: float) -> int:
    """Global slot pool size for "frac of the experts of every layer"."""
    return int(math.floor(frac * shape.E * shape.L + 1e-9))
