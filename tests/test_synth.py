"""The seeded input generator: deterministic, independent of thread count, and
with the value distributions the workloads ask for."""
import numpy as np

import synth


def test_streams_are_deterministic_and_thread_independent():
    k = synth.key(0, 1, 2, 3)
    a = synth.normal_bf16(k, 5_000_001, 0.02)
    b = synth.normal_bf16(k, 5_000_001, 0.02)
    assert np.array_equal(a, b)
    lib = synth._L()
    c = np.empty_like(a)
    lib.synth_fill_tab16_u16(synth._ptr(c), c.size, k, synth._ptr(synth._tab_bf16(0.02)), 1)
    assert np.array_equal(a, c)
    assert synth.key(0, 1, 2, 3) != synth.key(0, 1, 2, 4)


def test_normal_moments():
    x = synth.normal_f32(synth.key(5, 0), 1 << 20, 0.02).astype(np.float64)
    assert abs(x.mean()) < 1e-4 and abs(x.std() - 0.02) < 2e-4


def test_code_table_and_scale_ranges():
    t = synth._code_table()
    assert t.size == 256 and t.max() < 16
    s = synth.range_bytes(synth.key(1, 1), 10000, *synth.NVFP4_SCALE_BYTES)
    assert s.min() == synth.NVFP4_SCALE_BYTES[0] and s.max() == synth.NVFP4_SCALE_BYTES[1]


def test_zipf_bias_and_reuse_flags():
    shape = synth.DECODE_NVFP4
    r = synth.expert_ranks(shape, 0, 3)
    assert sorted(r) == list(range(1, shape.E + 1))
    f = synth.reuse_flags(0, 4096, 0.7)
    assert not f[0] and 0.66 < f.mean() < 0.74
    x = synth.hidden_states(shape, 0, 0, 8)
    assert np.all(x[:, 0] == 0x3F80)
    assert synth.capacity_slots(shape, 0.25) == 2560
    assert synth.capacity_slots(synth.STRESS_NVFP4, 0.05) == 128


def test_fp8_encoder_matches_torch_rne_and_weights_have_the_asked_spread():
    import torch
    # every representable magnitude, the midpoints between neighbours (ties go
    # to the even code) and points just off them
    grid = torch.arange(0, 0x7F, dtype=torch.uint8).view(torch.float8_e4m3fn).double().numpy()
    mids = (grid[1:] + grid[:-1]) / 2
    v = np.concatenate([grid, mids, mids * (1 + 1e-6), mids * (1 - 1e-6), [448.0, 500.0, 1e4]])
    ours = synth.e4m3_encode_rne(v)
    ref = torch.from_numpy(np.minimum(v, 448.0)).to(torch.float8_e4m3fn).view(torch.uint8).numpy()
    assert np.array_equal(ours, ref)
    t = synth._fp8_table()
    assert t.size == 256 and not np.any((t & 0x7F) == 0x7F)
    s = synth.Shape("t", L=1, E=1, k=1, H=512, I=256, fmt=synth.FMT_FP8, act=1)
    w = synth.expert_weights(s, 0, 0, 0)
    assert w["gate"]["codes"].shape == (256, 512) and w["down"]["codes"].shape == (512, 256)
    vals = torch.from_numpy(w["up"]["codes"]).view(torch.float8_e4m3fn).double().numpy() * w["up"]["gscale"]
    assert abs(vals.std() - 0.02) < 0.003 and abs(vals.mean()) < 1e-3
    assert np.array_equal(w["up"]["codes"], synth.expert_weights(s, 0, 0, 0)["up"]["codes"])
