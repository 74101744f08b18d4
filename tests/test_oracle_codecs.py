"""Pins for the oracle's weight codecs against sources other than itself:
the OCP MX specification's E2M1 table (golden file), PyTorch's float8 dtypes
(E4M3FN, E8M0) and bfloat16 conversion, and a hand-written packing example."""
import os

import numpy as np
import pytest
import torch

import oracle

GOLDEN = os.path.join(os.path.dirname(__file__), "golden")


def _golden_e2m1():
    vals = {}
    for line in open(os.path.join(GOLDEN, "e2m1_values.txt")):
        line = line.strip()
        if not line or line.startswith("#"):
            continue
        c, v = line.split()
        vals[int(c)] = float(v)
    return vals


def test_e2m1_all_codes_match_spec_table():
    g = _golden_e2m1()
    assert len(g) == 16
    for c in range(16):
        v = oracle.e2m1(c)
        assert v == g[c]
        assert np.signbit(v) == np.signbit(g[c])


def test_e4m3fn_all_bytes_match_torch():
    t = torch.arange(256, dtype=torch.uint8).view(torch.float8_e4m3fn).to(torch.float32).numpy()
    for b in range(256):
        v = oracle.e4m3fn(b)
        if np.isnan(t[b]):
            assert np.isnan(v), b
        else:
            assert v == t[b], (b, v, t[b])
    assert oracle.e4m3fn(0x7E) == 448.0
    assert oracle.e4m3fn(0x01) == 2.0 ** -9
    assert np.isnan(oracle.e4m3fn(0x7F)) and np.isnan(oracle.e4m3fn(0xFF))


def test_e8m0_all_bytes_match_torch():
    t = torch.arange(256, dtype=torch.uint8).view(torch.float8_e8m0fnu).to(torch.float32).numpy()
    for b in range(256):
        v = oracle.e8m0(b)
        if b == 255:
            assert np.isnan(v) and np.isnan(t[b])
        else:
            assert v == 2.0 ** (b - 127)
            assert v == t[b], (b, v, t[b])


def test_bf16_roundtrip_and_rne_match_torch():
    rng = np.random.default_rng(1)
    x = np.concatenate([
        rng.standard_normal(20000).astype(np.float32) * 10.0 ** rng.integers(-30, 30, 20000),
        np.array([0.0, -0.0, 1.0, 1.00390625, 1.01171875, 3.0e38, -3.4e38, 1e-40], np.float32),
    ]).astype(np.float32)
    # add exact ties: values halfway between two bf16 numbers
    ties = (np.arange(1, 200, dtype=np.uint32) << 16 | 0x8000).view(np.float32)
    x = np.concatenate([x, ties, -ties])
    ours = oracle.f32_to_bf16(x)
    ref = torch.from_numpy(x).to(torch.bfloat16).view(torch.int16).numpy().view(np.uint16)
    assert np.array_equal(ours, ref)
    back = oracle.bf16_to_f32(ours)
    ref_back = torch.from_numpy(ref.view(np.int16)).view(torch.bfloat16).to(torch.float32).numpy()
    assert np.array_equal(back.view(np.uint32), ref_back.view(np.uint32))


def test_products_exact_in_bf16_and_fp16():
    """Premise of exact in-register dequantisation: every E2M1 x E4M3 product and
    every E2M1 x E8M0 product within bf16's range is a bf16 (and, for E4M3, an
    fp16) number."""
    codes = [oracle.e2m1(c) for c in range(16)]
    for b in range(256):
        s = oracle.e4m3fn(b)
        if np.isnan(s):
            continue
        for c in codes:
            p = np.float32(c) * np.float32(s)
            assert float(torch.tensor(p).to(torch.bfloat16).float()) == float(p)
            assert float(torch.tensor(p).to(torch.float16).float()) == float(p)
    for b in range(1, 255):
        s = oracle.e8m0(b)
        for c in codes:
            p = np.float64(c) * np.float64(s)
            if (p != 0 and abs(p) < 2.0 ** -126) or abs(p) > 3.0e38:
                continue
            p = np.float32(p)
            assert float(torch.tensor(p).to(torch.bfloat16).float()) == float(p)


def test_packing_order_golden():
    line = [l for l in open(os.path.join(GOLDEN, "packing.txt")) if not l.startswith("#")][0]
    lhs, rhs = line.split("->")
    data = np.array([int(b, 16) for b in lhs.split()], np.uint8).reshape(1, -1)
    codes = [int(c) for c in rhs.split()]
    g = _golden_e2m1()
    # MXFP4 with scale byte 127 (= 1.0) decodes codes to their plain values
    w = oracle.dequant(oracle.MXFP4, {"codes": data, "scales": np.full((1, 1), 127, np.uint8)},
                       1, 8)
    assert list(w[0]) == [g[c] for c in codes]


def _torch_decode(fmt, t, N, K):
    """Independent decode: codes via the spec table, scales via torch dtypes."""
    g = _golden_e2m1()
    tab = np.array([g[c] for c in range(16)], np.float32)
    b = t["codes"].reshape(N, K // 2)
    c = np.empty((N, K), np.float32)
    c[:, 0::2] = tab[b & 0xF]
    c[:, 1::2] = tab[b >> 4]
    if fmt == oracle.NVFP4:
        s = torch.from_numpy(t["scales"]).view(torch.float8_e4m3fn).float().numpy()
        return (c * np.repeat(s, 16, axis=1)) * np.float32(t["gscale"])
    s = torch.from_numpy(t["scales"]).view(torch.float8_e8m0fnu).float().numpy()
    return c * np.repeat(s, 32, axis=1)


@pytest.mark.parametrize("fmt", [oracle.NVFP4, oracle.MXFP4])
def test_dequant_fp4_matches_independent_decode(fmt):
    import synth
    shape = synth.Shape("t", L=1, E=1, k=1, H=256, I=64, fmt=fmt, act=1)
    w = synth.expert_weights(shape, 7, 0, 0)
    for name, (N, K) in (("gate", (64, 256)), ("down", (256, 64))):
        ours = oracle.dequant(fmt, w[name], N, K)
        ref = _torch_decode(fmt, w[name], N, K)
        assert np.array_equal(ours, ref.astype(np.float32))


def test_e4m3_golden_values_and_fp8_dequant():
    """Hand-worked E4M3 values (tests/golden/e4m3_values.txt, from the OFP8
    definition): the oracle's decode, and FP8 dequantisation with a per-tensor
    scale of 0.25, reproduce them."""
    pairs = []
    for line in open(os.path.join(GOLDEN, "e4m3_values.txt")):
        line = line.strip()
        if not line or line.startswith("#"):
            continue
        b, v = line.split()
        pairs.append((int(b, 16), float(v)))
    for b, v in pairs:
        got = oracle.e4m3fn(b)
        assert got == v and np.signbit(got) == np.signbit(v), (hex(b), got, v)
    codes = np.array([[b for b, _ in pairs] + [0x38] * (128 - len(pairs))], np.uint8)
    w = oracle.dequant(oracle.FP8, {"codes": codes, "gscale": 0.25}, 1, 128)
    assert list(w[0, :len(pairs)]) == [np.float32(v) * np.float32(0.25) for _, v in pairs]


def test_dequant_fp8_matches_independent_decode():
    """FP8 weights: every E4M3 byte decoded by torch's float8_e4m3fn dtype,
    times the per-tensor scale, equals the oracle's dequantisation."""
    import synth
    shape = synth.Shape("t", L=1, E=1, k=1, H=256, I=64, fmt=oracle.FP8, act=1)
    w = synth.expert_weights(shape, 7, 0, 0)
    for name, (N, K) in (("gate", (64, 256)), ("down", (256, 64))):
        t = w[name]
        ours = oracle.dequant(oracle.FP8, t, N, K)
        ref = torch.from_numpy(t["codes"]).view(torch.float8_e4m3fn).float().numpy() * np.float32(t["gscale"])
        assert np.array_equal(ours, ref)
    # all finite bytes (subnormals, zeros, negatives, +-448) in one row, scale 2^-3
    b = np.array([x for x in range(256) if x & 0x7F != 0x7F], np.uint8).reshape(1, -1)
    ours = oracle.dequant(oracle.FP8, {"codes": b, "gscale": 0.125}, 1, b.shape[1])
    ref = torch.from_numpy(b).view(torch.float8_e4m3fn).float().numpy() * np.float32(0.125)
    assert np.array_equal(ours, ref)


def test_dequant_bf16_fp32_identity():
    import synth
    for fmt in (oracle.FP32, oracle.BF16):
        shape = synth.Shape("t", L=1, E=1, k=1, H=64, I=32, fmt=fmt, act=1)
        w = synth.expert_weights(shape, 3, 0, 0)["up"]
        ours = oracle.dequant(fmt, w, 32, 64)
        if fmt == oracle.FP32:
            ref = w["data"]
        else:
            ref = torch.from_numpy(w["data"].view(np.int16)).view(torch.bfloat16).float().numpy()
        assert np.array_equal(ours, ref)
