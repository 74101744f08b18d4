"""Pins for the oracle's activation quantisers (the tolerance study of a
block-scaled MMA; the layer itself never quantises activations): the element
roundings against torch's float8 conversion and the E2M1 grid with its tie
rule, exactness on representable inputs, the error bound, sign symmetry and
power-of-two scaling."""
import numpy as np
import pytest
import torch

import oracle


def test_e4m3_rne_matches_torch_on_codes_midpoints_and_neighbours():
    grid = torch.arange(0, 0x7F, dtype=torch.uint8).view(torch.float8_e4m3fn).double().numpy()
    mids = (grid[1:] + grid[:-1]) / 2
    v = np.concatenate([grid, mids, mids * (1 + 1e-5), mids * (1 - 1e-5)])
    v = np.concatenate([v, -v]).astype(np.float32)
    ours = np.array([oracle.e4m3_rne(float(a)) for a in v], np.float32)
    ref = torch.from_numpy(v).to(torch.float8_e4m3fn).float().numpy()
    assert np.array_equal(ours, ref)
    assert oracle.e4m3_rne(500.0) == 448.0 and oracle.e4m3_rne(-1e9) == -448.0


def test_e2m1_rne_grid_ties_and_saturation():
    # ties go to the even code: codes 0 (0), 2 (1.0), 4 (2.0), 6 (4.0)
    cases = {0.0: 0.0, 0.25: 0.0, 0.26: 0.5, 0.75: 1.0, 1.25: 1.0, 1.75: 2.0, 2.5: 2.0, 3.5: 4.0,
             5.0: 4.0, 5.01: 6.0, 6.0: 6.0, 100.0: 6.0, 0.5: 0.5, 3.0: 3.0, 1.5: 1.5}
    for v, want in cases.items():
        assert oracle.e2m1_rne(v) == want, v
        assert oracle.e2m1_rne(-v) == -want, v


@pytest.mark.parametrize("kind", [oracle.QUANT_MXFP8, oracle.QUANT_NVFP4])
def test_quantisers_symmetry_scaling_and_idempotence(kind):
    rng = np.random.default_rng(kind)
    x = rng.standard_normal(4096).astype(np.float32)
    q = oracle.quant_act(kind, x)
    assert np.array_equal(oracle.quant_act(kind, -x), -q)
    for k in (-20, -3, 5, 17):
        assert np.array_equal(oracle.quant_act(kind, x * np.float32(2.0 ** k)), q * np.float32(2.0 ** k))
    assert np.array_equal(oracle.quant_act(kind, np.zeros(64, np.float32)), np.zeros(64, np.float32))
    if kind == oracle.QUANT_MXFP8:
        # quantised blocks are fixed points (their amax keeps its binade, every element is on the grid)
        assert np.array_equal(oracle.quant_act(kind, q), q)


def test_mxfp8_exact_on_representable_blocks_and_error_bound():
    rng = np.random.default_rng(7)
    codes = torch.arange(0, 0x7F, dtype=torch.uint8).view(torch.float8_e4m3fn).float().numpy()
    for p in (-9, 0, 6):
        X = np.float32(2.0 ** (p - 8))
        blk = rng.choice(codes[codes <= 448], 32).astype(np.float32)
        blk[rng.integers(32)] = 256.0 + 0.0  # amax = 2^p: X = 2^(p - 8)
        blk[rng.integers(32)] *= -1
        x = blk * X
        assert np.array_equal(oracle.quant_act(oracle.QUANT_MXFP8, x), x)
    # below saturation each element is within half a step (2^-4 of its binade)
    x = rng.standard_normal(32 * 64).astype(np.float32)
    q = oracle.quant_act(oracle.QUANT_MXFP8, x)
    xb, qb = x.reshape(-1, 32), q.reshape(-1, 32)
    for a, b in zip(xb, qb):
        e = np.floor(np.log2(np.abs(a).max()))
        X = 2.0 ** (e - 8)
        ok = np.abs(a) / X <= 448
        step = np.maximum(2.0 ** (np.floor(np.log2(np.maximum(np.abs(a[ok]) / X, 2.0 ** -6))) - 3), 2.0 ** -9) * X
        assert np.all(np.abs(a[ok] - b[ok]) <= step / 2 * (1 + 1e-6))
        assert np.all(np.abs(b[~ok]) == np.float32(448 * X))


def test_nvfp4_exact_on_representable_vectors():
    # amax = 6 * 448 * g with g = 1: every block whose amax / 6 is an E4M3 value and whose
    # elements are E2M1 values times that block scale comes back unchanged
    rng = np.random.default_rng(11)
    grid = np.array([0, 0.5, 1, 1.5, 2, 3, 4, 6], np.float32)
    scales = np.array([448.0, 1.0, 0.5, 3.0, 40.0, 2.0 ** -6, 0.875, 96.0], np.float32)
    blocks = []
    for s in scales:
        b = rng.choice(grid, 16) * np.sign(rng.standard_normal(16))
        b[rng.integers(16)] = 6.0
        blocks.append(b.astype(np.float32) * s)
    x = np.concatenate(blocks).astype(np.float32)
    assert np.array_equal(oracle.quant_act(oracle.QUANT_NVFP4, x), x)


def test_tolerance_study_runs_and_quantised_layer_moves():
    from oracle.tolerance_study import study
    import synth
    s = synth.Shape("tiny-q", L=1, E=8, k=2, H=128, I=64, fmt=synth.FMT_NVFP4, act=synth.ACT_BF16, shared=1)
    res = study(s, 4)
    for kind in (oracle.QUANT_MXFP8, oracle.QUANT_NVFP4):
        tensor_err, row_err = res[kind]
        assert 0 < tensor_err <= row_err < 1
    assert res[oracle.QUANT_MXFP8][0] < res[oracle.QUANT_NVFP4][0]
