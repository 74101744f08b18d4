"""CUDA path vs oracle on the same seeded inputs, through the C ABI.

Bit-exact: top-k indices, permutation, counts, unique-expert list and the LRU
hit/miss/slot/eviction event sequence. Outputs: max |y - y_ref| / max |y_ref|
<= 2e-2 (bf16 I/O, fp32 accumulation). Small shapes span several 128-wide
K groups, 16-row tiles and 8-column tiles with ragged tails; the workload
shapes run on a subset of their layers with sampled output rows."""
import numpy as np
import pytest

import synth

pytestmark = pytest.mark.gpu

try:
    import torch
    HAVE_GPU = torch.cuda.is_available()
except Exception:  # pragma: no cover
    HAVE_GPU = False


@pytest.fixture(scope="module", autouse=True)
def _need_gpu():
    if not HAVE_GPU:
        pytest.skip("no CUDA device")
    from expert_offload_softmax_b300 import build
    build.build()


def _run(shape, seed, L, capacity, calls, flags=0, sample=None, max_tokens=0, cover=None):
    """calls: list of (layer, T, step). sample: check outputs on that many evenly
    spaced tokens; cover: on at least that many tokens that together select
    every expert the call routes to. Returns the measured errors."""
    from moe_harness import GpuStack, OracleStack, compare, oracle_workers
    g = GpuStack(shape, seed, L, capacity, flags, max_tokens=max_tokens)
    o = OracleStack(shape, seed, L, capacity, prefetch=bool(flags & 1), workers=oracle_workers() if cover else 0)
    errs = []
    try:
        for (layer, T, step) in calls:
            x = synth.hidden_states(shape, seed, layer, T, step)
            toks = None if sample is None or T <= sample else np.linspace(0, T - 1, sample).astype(int)
            if cover and T > cover:
                toks = f"cover:{cover}"
            gr = g.forward(layer, x)
            orr = o.forward(layer, x, toks)
            errs.append(compare(gr, orr))
    finally:
        g.close()
    return errs


def test_tiny_fp32_workload():
    s = synth.TINY_FP32
    errs = _run(s, 0, 1, 8, [(0, 4, 0), (0, 4, 1), (0, 1, 2)])
    assert max(e["out_err"] for e in errs) < 1e-5


@pytest.mark.parametrize("fmt", [synth.FMT_BF16, synth.FMT_NVFP4, synth.FMT_MXFP4, synth.FMT_FP8])
@pytest.mark.parametrize("T", [1, 3, 8])
def test_small_decode_all_formats(fmt, T):
    s = synth.Shape("small", L=3, E=16, k=4, H=384, I=256, fmt=fmt, act=synth.ACT_BF16)
    calls = [(l % 3, T, l) for l in range(7)]
    _run(s, 11, 3, 10 if T < 8 else 20, calls)


@pytest.mark.parametrize("fmt", [synth.FMT_BF16, synth.FMT_NVFP4, synth.FMT_MXFP4, synth.FMT_FP8])
@pytest.mark.parametrize("T", [9, 37, 200])
def test_small_prefill_all_formats(fmt, T):
    s = synth.Shape("small", L=3, E=16, k=4, H=384, I=256, fmt=fmt, act=synth.ACT_BF16)
    calls = [(l % 3, T, l) for l in range(5)]
    _run(s, 12, 3, 20, calls, flags=0)


def test_prefill_bf16_tensor_core_multi_tile():
    """BF16 prefill takes the tcgen05 path: 8 experts x top-2 over 1000 tokens
    puts ~250 tokens on each expert (two 128-token tiles, ragged second tile),
    H=640 gives 10 K-blocks of 64 and 5 down-projection row tiles, I=384 gives
    three 128-unit gate/up tiles."""
    s = synth.Shape("umma", L=2, E=8, k=2, H=640, I=384, fmt=synth.FMT_BF16, act=synth.ACT_BF16)
    _run(s, 22, 2, 16, [(0, 1000, 0), (1, 130, 1), (0, 17, 2)], max_tokens=1000)


def test_prefill_bf16_tensor_core_shared_expert_fp32_act():
    """tcgen05 prefill with an always-on shared expert (its weights resident
    outside the pool) and fp32 activations converted to bf16 in the gather."""
    s = synth.Shape("umma-shared", L=2, E=16, k=4, H=256, I=256, fmt=synth.FMT_BF16, act=synth.ACT_FP32, shared=1)
    _run(s, 23, 2, 32, [(0, 300, 0), (1, 41, 0), (1, 2, 1)], max_tokens=512)


def test_fp8_prefill_tensor_core_multi_tile_ragged_chunks():
    """FP8 prefill: 8 experts x top-2 over 1000 tokens (two 128-token tiles per
    expert, the second ragged); H = 1152 gives a full 8-group chunk and a
    1-group chunk per gate/up row and I = 384 one 3-group down chunk."""
    s = synth.Shape("fp8-umma", L=2, E=8, k=2, H=1152, I=384, fmt=synth.FMT_FP8, act=synth.ACT_BF16)
    _run(s, 24, 2, 16, [(0, 1000, 0), (1, 130, 1), (0, 17, 2), (1, 1, 3), (0, 8, 4)], max_tokens=1000)


def test_fp8_shared_expert_fp32_activations_and_host_copied_misses():
    """FP8 decode and prefill with an always-on shared expert and fp32
    activations; then the same with the host's copy engines serving the
    decode misses."""
    s = synth.Shape("fp8-shared", L=2, E=16, k=4, H=256, I=256, fmt=synth.FMT_FP8, act=synth.ACT_FP32, shared=1)
    calls = [(0, 1, 0), (1, 8, 0), (0, 300, 1), (1, 5, 2), (0, 1, 3)]
    _run(s, 25, 2, 16, calls, max_tokens=512)  # 16 slots: one layer's experts, so every layer switch misses
    _run(s, 25, 2, 16, calls, flags=8, max_tokens=512)


def test_fp8_linear_mode():
    s = synth.Shape("lin8", L=1, E=8, k=3, H=256, I=128, fmt=synth.FMT_FP8, act=synth.ACT_BF16, act_mode=1)
    _run(s, 26, 1, 8, [(0, 6, 0), (0, 40, 1), (0, 1, 2)])


def test_prefill_more_than_512_routing_blocks():
    """T = 4200: 525 routing CTAs of 8 tokens, so the permutation kernel sums
    count columns past the first 512 (its tail loop); routing and permutation
    bit-exact, outputs on 64 tokens."""
    s = synth.Shape("long", L=1, E=16, k=2, H=256, I=128, fmt=synth.FMT_BF16, act=synth.ACT_BF16)
    _run(s, 27, 1, 16, [(0, 4200, 0)], sample=64, max_tokens=4200)


def test_prefill_prefetch_next_layer():
    s = synth.Shape("small", L=4, E=16, k=4, H=256, I=128, fmt=synth.FMT_NVFP4, act=synth.ACT_BF16)
    calls = [(l, 64, 0) for l in range(4)] + [(l, 64, 1) for l in range(4)]
    _run(s, 13, 4, 40, calls, flags=1)  # 40 >= 16 + 16: prefetch runs


def test_shared_expert_and_fp32_activations():
    s = synth.Shape("shared", L=2, E=8, k=2, H=256, I=128, fmt=synth.FMT_MXFP4, act=synth.ACT_FP32, shared=1)
    _run(s, 14, 2, 10, [(0, 5, 0), (1, 5, 0), (0, 20, 1), (1, 1, 2)])


def test_linear_mode_closed_form_path():
    s = synth.Shape("lin", L=1, E=8, k=3, H=256, I=128, fmt=synth.FMT_NVFP4, act=synth.ACT_BF16, act_mode=1)
    _run(s, 15, 1, 8, [(0, 6, 0), (0, 40, 1)])


def test_zipf_skewed_decode_many_steps():
    s = synth.Shape("zipf", L=4, E=64, k=8, H=256, I=128, fmt=synth.FMT_NVFP4, act=synth.ACT_BF16, zipf_s=1.0)
    calls = [(l, 1 + (st % 8), st) for st in range(12) for l in range(4)]
    _run(s, 16, 4, 64, calls)


def test_host_copied_decode_misses_match_oracle():
    """MOE_CACHE_HOST_MISSES: the host copies each decode call's misses with
    cudaMemcpyAsync and the decode kernel waits for its release; routing, the
    cache sequence and the outputs are those of the oracle (as for the default,
    where the kernel copies them itself)."""
    s = synth.Shape("zipf", L=4, E=64, k=8, H=256, I=128, fmt=synth.FMT_NVFP4, act=synth.ACT_BF16, zipf_s=1.0)
    _run(s, 16, 4, 64, [(l, 1 + (st % 8), st) for st in range(6) for l in range(4)], flags=8)
    s = synth.Shape("small", L=2, E=16, k=4, H=384, I=256, fmt=synth.FMT_MXFP4, act=synth.ACT_BF16, shared=1)
    _run(s, 13, 2, 20, [(l % 2, 1 + l % 8, l) for l in range(10)], flags=8)


def test_sync_misses_mode_matches_oracle():
    """MOE_CACHE_SYNC_MISSES moves the miss copies before the expert launches;
    the cache sequence and the outputs are those of the asynchronous path."""
    s = synth.Shape("zipf", L=4, E=64, k=8, H=256, I=128, fmt=synth.FMT_NVFP4, act=synth.ACT_BF16, zipf_s=1.0)
    _run(s, 16, 4, 64, [(l, 1 + (st % 8), st) for st in range(3) for l in range(4)], flags=4)
    s = synth.Shape("small", L=4, E=16, k=4, H=256, I=128, fmt=synth.FMT_MXFP4, act=synth.ACT_BF16)
    _run(s, 13, 4, 40, [(l, 64, 0) for l in range(4)] + [(0, 3, 1)], flags=4 | 1)


def test_unknown_cache_flag_is_rejected():
    import expert_offload_softmax_b300 as moe
    from moe_harness import GpuStack
    s = synth.Shape("small", L=1, E=8, k=2, H=256, I=128, fmt=synth.FMT_NVFP4, act=synth.ACT_BF16)
    g = GpuStack(s, 3, 1, 8)
    try:
        with pytest.raises(moe.MoeError) as ei:
            moe.moe_cache_config(g.h, 8, 64)
        assert ei.value.code == moe.MOE_ERR_INVALID
    finally:
        g.close()


def test_capacity_error_leaves_cache_unchanged():
    import expert_offload_softmax_b300 as moe
    from moe_harness import GpuStack
    s = synth.Shape("cap", L=1, E=16, k=4, H=256, I=128, fmt=synth.FMT_BF16, act=synth.ACT_BF16)
    g = GpuStack(s, 17, 1, 4)
    try:
        g.forward(0, synth.hidden_states(s, 17, 0, 1, 0))
        before = moe.moe_debug_lru_table(g.h, 1, 16).copy()
        x = synth.hidden_states(s, 17, 0, 8, 1)   # 8 tokens x 4 experts: more than 4 distinct
        with pytest.raises(moe.MoeError) as ei:
            g.forward(0, x)
        assert ei.value.code == moe.MOE_ERR_CAPACITY
        assert np.array_equal(before, moe.moe_debug_lru_table(g.h, 1, 16))
    finally:
        g.close()


def test_empty_call_and_bad_arguments():
    import expert_offload_softmax_b300 as moe
    from moe_harness import GpuStack
    s = synth.Shape("e", L=2, E=8, k=2, H=128, I=128, fmt=synth.FMT_NVFP4, act=synth.ACT_BF16)
    g = GpuStack(s, 18, 2, 8)
    try:
        x = g.to_dev(synth.hidden_states(s, 18, 0, 2, 0))
        out = g.out_buf(2)
        moe.moe_layer_forward(g.h, x.data_ptr(), g.router[0].data_ptr(), 0, 0, out.data_ptr())
        for layer, T in ((2, 2), (-1, 2), (0, 100000)):
            with pytest.raises(moe.MoeError) as ei:
                moe.moe_layer_forward(g.h, x.data_ptr(), g.router[0].data_ptr(), layer, T, out.data_ptr())
            assert ei.value.code == moe.MOE_ERR_INVALID
    finally:
        g.close()


def test_two_runs_bitwise_identical():
    from moe_harness import GpuStack
    s = synth.Shape("det", L=2, E=32, k=4, H=512, I=256, fmt=synth.FMT_NVFP4, act=synth.ACT_BF16)
    outs = []
    for _ in range(2):
        g = GpuStack(s, 19, 2, 64)
        try:
            outs.append([g.forward(l, synth.hidden_states(s, 19, l, T, 0))["out"] for l, T in ((0, 3), (1, 77))])
        finally:
            g.close()
    for a, b in zip(*outs):
        assert np.array_equal(a, b)


# --------------------------------------------------------------------------- workload shapes

def test_workload_decode_nvfp4_layer_subset():
    """decode-40L-H2048-E256-k8-I512-nvfp4 on 4 of its layers (same per-layer
    shape, Zipf s=1.0), pool = 25% of the experts of those layers."""
    s = synth.DECODE_NVFP4
    L = 4
    cap = synth.capacity_slots(synth.Shape("x", L=L, E=s.E, k=s.k, H=s.H, I=s.I, fmt=s.fmt, act=s.act), 0.25)
    calls = [(l, T, st) for st, T in enumerate((1, 8, 1, 8, 1)) for l in range(L)]
    _run(s, 0, L, cap, calls)


def test_workload_decode_shape_fp8_layer_subset():
    """The decode workload's shape (H2048, E256, k8, I512, Zipf s=1.0) with FP8
    experts on 3 of its layers, pool of 300 slots; decode
    T=1 and T=8, then one T=512 prefill call with outputs on 64 tokens."""
    d = synth.DECODE_NVFP4
    s = synth.Shape("decode-40L-H2048-E256-k8-I512-fp8", L=40, E=d.E, k=d.k, H=d.H, I=d.I, fmt=synth.FMT_FP8,
                    act=synth.ACT_BF16, zipf_s=1.0)
    L = 3
    cap = 300  # 39% of those layers' experts: room for one prefill call's unique experts
    calls = [(l, T, st) for st, T in enumerate((1, 8, 1)) for l in range(L)] + [(0, 512, 9)]
    _run(s, 0, L, cap, calls, sample=64, max_tokens=512)


def test_workload_prefill_bf16_layer_subset():
    """prefill-40L-H2048-E256-k8-I512-bf16 at T=4096 on 2 layers with prefetch,
    routing in full, outputs on at least 256 tokens that together select every
    expert the call routes to."""
    s = synth.PREFILL_BF16
    _run(s, 0, 2, 256 + 256 + 8, [(0, 4096, 0), (1, 4096, 0)], flags=1, cover=256, max_tokens=4096)


def test_workload_large_mxfp4_shared_layer_subset():
    """large-24L-H4096-E256+1-k8-I2048-mxfp4: decode T=1 and prefill T=2048 on
    2 layers; prefill outputs on at least 256 tokens that together select every
    expert the call routes to (and the shared expert on each of them)."""
    s = synth.LARGE_MXFP4
    _run(s, 0, 2, 300, [(0, 1, 0), (1, 1, 0), (0, 2048, 1)], cover=256, max_tokens=2048)


@pytest.mark.parametrize("frac", [0.05, 0.10, 0.25])
def test_workload_stress_nvfp4_pool_sweep(frac):
    """stress-16L-H6144-E160-k8-I2048-nvfp4: 24 decode steps of T=1 with Zipf
    s=1.1 and step reuse (p=0.7) on 3 layers, pool of 5%, 10% or 25% of those
    layers' experts (24, 48, 120 slots). Routing and the LRU sequence on every
    call; outputs on every call of the first 8 steps."""
    from moe_harness import GpuStack, OracleStack, compare
    s = synth.STRESS_NVFP4
    L = 3
    cap = max(s.k, int(frac * s.E * L + 1e-9))
    reuse = synth.reuse_flags(0, 24, 0.7)
    g = GpuStack(s, 0, L, cap)
    o = OracleStack(s, 0, L, cap, prefetch=False, max_cached_experts=96)
    try:
        src = 0
        for st in range(24):
            src = src if reuse[st] else st
            for l in range(L):
                x = synth.hidden_states(s, 0, l, 1, src)
                compare(g.forward(l, x), o.forward(l, x, None if st < 8 else []))
        st_ = g.stats()
        assert st_["misses"] > 0 and st_["hits"] > 0
    finally:
        g.close()
