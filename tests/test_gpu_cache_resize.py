"""The cache at its safe points, through the C ABI: a caller-owned pool buffer
(moe_cache_config with a device buffer the caller allocated, here by torch),
and live resizes between forward calls (moe_cache_resize), growing and
shrinking, into a new buffer or in place. After each resize the LRU event
sequence (hit, slot, evicted key) stays bit-exact with the oracle's, resized at
the same points by its own rule, and the outputs of later calls (which read the
kept experts from their new slots) stay within the tolerance."""
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


def _blob(moe, s):
    return moe.moe_expert_bytes(moe.make_desc(1, s.E, s.k, s.H, s.I, s.fmt, s.act, shared=s.shared))


def _calls(g, o, s, seed, steps, T_of, layers):
    from moe_harness import compare
    for st in steps:
        for l in layers:
            x = synth.hidden_states(s, seed, l, T_of(st), st)
            compare(g.forward(l, x), o.forward(l, x))


@pytest.mark.parametrize("fmt", [synth.FMT_NVFP4, synth.FMT_BF16])
def test_caller_owned_pool(fmt):
    import expert_offload_softmax_b300 as moe
    from moe_harness import GpuStack, OracleStack
    s = synth.Shape("pool", L=3, E=16, k=4, H=256, I=128, fmt=fmt, act=synth.ACT_BF16, zipf_s=1.0)
    g = GpuStack(s, 51, 3, 8, max_tokens=64)
    try:
        cap = 20
        buf = torch.empty(cap * _blob(moe, s), dtype=torch.uint8, device=g.dev)
        for bad in ((buf[1:].data_ptr(), buf.numel() - 1), (buf.data_ptr(), buf.numel() - 1)):
            with pytest.raises(moe.MoeError) as ei:
                moe.moe_cache_config(g.h, cap, moe.MOE_CACHE_LOG_EVENTS, *bad)
            assert ei.value.code == moe.MOE_ERR_INVALID
        g.reconfigure(cap, pool=buf)
        o = OracleStack(s, 51, 3, cap, prefetch=False)
        _calls(g, o, s, 51, range(4), lambda st: (1, 5, 40, 8)[st], range(3))
    finally:
        g.close()
    assert buf.numel() == cap * _blob(moe, s)  # still the caller's: nothing freed it


@pytest.mark.parametrize("fmt", [synth.FMT_NVFP4, synth.FMT_MXFP4, synth.FMT_FP8])
def test_resize_between_calls_matches_oracle(fmt):
    import expert_offload_softmax_b300 as moe
    from moe_harness import GpuStack, OracleStack
    s = synth.Shape("resize", L=4, E=32, k=4, H=256, I=128, fmt=fmt, act=synth.ACT_BF16, zipf_s=1.0)
    g = GpuStack(s, 53, 4, 24, max_tokens=64)
    o = OracleStack(s, 53, 4, 24, prefetch=False)
    T_of = lambda st: (1, 3, 8, 1, 20)[st % 5]
    try:
        _calls(g, o, s, 53, range(0, 5), T_of, range(4))
        for cap in (40, 12, 16, 8):          # grow, shrink, grow, shrink to the minimum of two tokens' experts
            g.resize(cap)
            o.resize(cap)
            np.testing.assert_array_equal(moe.moe_debug_lru_table(g.h, 4, 32), o.lru.table)
            _calls(g, o, s, 53, range(5 * cap, 5 * cap + 5), T_of, range(4))
        # in place, in a caller-owned buffer: shrink, then grow back within it
        buf = torch.empty(30 * _blob(moe, s), dtype=torch.uint8, device=g.dev)
        g.reconfigure(30, pool=buf)
        o = OracleStack(s, 53, 4, 30, prefetch=False)
        _calls(g, o, s, 53, range(100, 104), T_of, range(4))
        for cap in (14, 30):
            g.resize(cap, pool=buf)
            o.resize(cap)
            np.testing.assert_array_equal(moe.moe_debug_lru_table(g.h, 4, 32), o.lru.table)
            _calls(g, o, s, 53, range(200 + cap, 204 + cap), T_of, range(4))
    finally:
        g.close()
