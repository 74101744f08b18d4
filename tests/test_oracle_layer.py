"""Pins for the oracle's expert FFN and layer combine: closed forms with
identity-like experts in every weight format, and a dense fp64 numpy (einsum)
re-computation on the tiny fp32 workload."""
import os

import numpy as np
import pytest

import oracle
import synth

ROOT = os.path.dirname(os.path.dirname(os.path.abspath(__file__)))

FORMATS = [synth.FMT_FP32, synth.FMT_BF16, synth.FMT_NVFP4, synth.FMT_MXFP4, synth.FMT_FP8]


def _eye_tensor(fmt, N, K, alpha_log2):
    """[N, K] tensor equal to 2^alpha_log2 * (identity on the leading min(N, K)
    block), written directly in the storage encoding of ``fmt``."""
    m = min(N, K)
    alpha = 2.0 ** alpha_log2
    if fmt == synth.FMT_FP32:
        d = np.zeros((N, K), np.float32)
        d[np.arange(m), np.arange(m)] = alpha
        return {"data": d}
    if fmt == synth.FMT_BF16:
        d = np.zeros((N, K), np.uint16)
        d[np.arange(m), np.arange(m)] = synth.f32_to_bf16_bits(np.array([alpha], np.float32))[0]
        return {"data": d}
    if fmt == synth.FMT_FP8:
        codes = np.zeros((N, K), np.uint8)
        codes[np.arange(m), np.arange(m)] = 0x38  # E4M3 1.0
        return {"codes": codes, "gscale": alpha}
    codes = np.zeros((N, K // 2), np.uint8)
    for i in range(m):
        # E2M1 code 2 is 1.0 (golden table); low nibble = even element
        codes[i, i // 2] |= (2 << 4) if (i & 1) else 2
    if fmt == synth.FMT_NVFP4:
        return {"codes": codes, "scales": np.full((N, K // 16), 0x38, np.uint8),  # E4M3 1.0
                "gscale": alpha}
    return {"codes": codes, "scales": np.full((N, K // 32), 127 + alpha_log2, np.uint8)}


def _eye_experts(fmt, E, n_shared, H, I, alog):
    return {e: {"gate": _eye_tensor(fmt, I, H, 0), "up": _eye_tensor(fmt, I, H, 0),
                "down": _eye_tensor(fmt, H, I, alog[e])} for e in range(E + n_shared)}


@pytest.mark.parametrize("fmt", FORMATS)
@pytest.mark.parametrize("mode", [1, 0])
def test_closed_form_identity_experts(fmt, mode):
    H, I, E, k, T, n_sh = 128, 64, 8, 3, 5, 1
    shape = synth.Shape("cf", L=1, E=E, k=k, H=H, I=I, fmt=fmt, act=synth.ACT_FP32,
                        shared=n_sh, act_mode=mode)
    rng = np.random.default_rng(fmt * 10 + mode)
    alog = [int(a) for a in rng.integers(-1, 2, E + n_sh)]
    experts = _eye_experts(fmt, E, n_sh, H, I, alog)
    x = rng.standard_normal((T, H)).astype(np.float32)
    w = (rng.standard_normal((E, H)) * 0.5).astype(np.float32)
    r = oracle.layer(shape, experts, w, x)
    assert np.all(np.abs(r["gates"].astype(np.float64).sum(1) - 1) <= 1e-6)
    alpha = np.array([2.0 ** a for a in alog])
    x64 = x.astype(np.float64)[:, :I]
    act = x64 if mode == 1 else x64 / (1 + np.exp(-x64))
    coef = (r["gates"].astype(np.float64) * alpha[r["topk_idx"]]).sum(1) + alpha[E]
    ref = np.zeros((T, H))
    ref[:, :I] = coef[:, None] * act * x64
    err = np.abs(r["out"] - ref).max() / np.abs(ref).max()
    assert err <= 2e-6, err
    assert np.all(r["out"][:, I:] == 0)


def test_closed_form_all_alpha_one_gives_square():
    H, I, E, k, T = 64, 64, 8, 2, 4
    shape = synth.Shape("cf", L=1, E=E, k=k, H=H, I=I, fmt=synth.FMT_BF16, act=synth.ACT_FP32,
                        act_mode=1)
    experts = _eye_experts(synth.FMT_BF16, E, 0, H, I, [0] * E)
    rng = np.random.default_rng(9)
    x = rng.standard_normal((T, H)).astype(np.float32)
    w = rng.standard_normal((E, H)).astype(np.float32)
    r = oracle.layer(shape, experts, w, x)
    assert np.max(np.abs(r["out"] - x.astype(np.float64) ** 2)) <= 4e-6 * np.max(x ** 2)


def test_dense_einsum_cross_check_tiny_fp32():
    shape = synth.TINY_FP32
    seed = 0
    x = synth.hidden_states(shape, seed, 0, 4)
    w = synth.router_weights(shape, seed, 0)
    experts = {e: synth.expert_weights(shape, seed, 0, e) for e in range(shape.E)}
    r = oracle.layer(shape, experts, w, x)
    Wg = np.stack([experts[e]["gate"]["data"] for e in range(shape.E)]).astype(np.float64)
    Wu = np.stack([experts[e]["up"]["data"] for e in range(shape.E)]).astype(np.float64)
    Wd = np.stack([experts[e]["down"]["data"] for e in range(shape.E)]).astype(np.float64)
    x64 = x.astype(np.float64)
    g = np.einsum("eih,th->tei", Wg, x64)
    u = np.einsum("eih,th->tei", Wu, x64)
    h = g / (1 + np.exp(-g)) * u
    y = np.einsum("ehi,tei->teh", Wd, h)                          # every expert, every token
    sel = y[np.arange(4)[:, None], r["topk_idx"]]                 # [T, k, H]
    ref = (r["gates"].astype(np.float64)[:, :, None] * sel).sum(1)
    err = np.abs(r["out"] - ref).max() / np.abs(ref).max()
    assert err <= 1e-5, err
    # routing from fp64 logits agrees with the oracle's (no near-ties here)
    lg = x64 @ w.astype(np.float64).T
    top = np.argsort(-lg, axis=1, kind="stable")[:, :shape.k]
    assert np.array_equal(top, r["topk_idx"])


def test_layer_token_subset_matches_full():
    shape = synth.Shape("s", L=1, E=16, k=4, H=128, I=64, fmt=synth.FMT_NVFP4,
                        act=synth.ACT_BF16)
    x = synth.hidden_states(shape, 1, 0, 10)
    w = synth.router_weights(shape, 1, 0)
    experts = {e: synth.expert_weights(shape, 1, 0, e) for e in range(shape.E)}
    full = oracle.layer(shape, experts, w, x)
    part = oracle.layer(shape, experts, w, x, toks=[7, 2])
    assert np.array_equal(part["out"], full["out"][[7, 2]])


def test_expert_major_evaluation_matches_layer_tokens():
    """The test harness's expert-at-a-time evaluation (expert outputs in worker
    processes, then the oracle's combine per token) gives the same bits as
    the oracle's token-at-a-time layer output, shared expert included."""
    import sys
    sys.path.insert(0, os.path.join(ROOT, "tests"))
    from moe_harness import OracleStack, cover_tokens
    s = synth.Shape("em", L=1, E=16, k=4, H=256, I=128, fmt=synth.FMT_MXFP4, act=synth.ACT_BF16, shared=1)
    x = synth.hidden_states(s, 3, 0, 24, 0)
    a = OracleStack(s, 3, 1, 32, False).forward(0, x, np.arange(24))
    b = OracleStack(s, 3, 1, 32, False, workers=2).forward(0, x, np.arange(24))
    assert np.array_equal(a["out"], b["out"])
    t = cover_tokens(a["topk_idx"], 5)
    assert set(a["topk_idx"][t].ravel()) == set(a["topk_idx"].ravel()) and len(t) >= 5
