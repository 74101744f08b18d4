"""Failure detection of the miss pipeline, with the failure made on the host.

The cache is configured so that the host copies decode misses
(MOE_CACHE_HOST_MISSES), and the service thread is told (MOE_FAULT=drop_release)
to skip the release of the first call that has cache misses, as if it had
died. The call's kernel then waits on a word that nothing sets; their wait is bounded (MOE_WAIT_MS), so
they give up, record a device error and return, and the context stays usable.
The error is reported (MOE_ERR_TIMEOUT) and stays until moe_cache_config,
after which the layer matches the oracle again. No GPU fault, trap or endless
loop is involved."""
import numpy as np
import pytest

import synth

pytestmark = pytest.mark.gpu


def test_dropped_release_times_out_reports_and_recovers(monkeypatch):
    import torch
    if not torch.cuda.is_available():
        pytest.skip("no CUDA device")
    from expert_offload_softmax_b300 import build
    build.build()
    import expert_offload_softmax_b300 as moe
    from moe_harness import GpuStack, OracleStack, compare

    monkeypatch.setenv("MOE_WAIT_MS", "200")
    monkeypatch.setenv("MOE_FAULT", "drop_release")
    shape = synth.Shape("fault-2L-H256-E16-k4-I128-nvfp4", L=2, E=16, k=4, H=256, I=128,
                        fmt=synth.FMT_NVFP4, act=synth.ACT_BF16)
    g = GpuStack(shape, 31, 2, 12, flags=moe.MOE_CACHE_HOST_MISSES)
    try:
        x = synth.hidden_states(shape, 31, 0, 3, 0)
        # cold cache: the call misses, its release is dropped, the kernels give up
        with pytest.raises(moe.MoeError) as ei:
            g.forward(0, x)
        assert ei.value.code == moe.MOE_ERR_TIMEOUT
        assert moe.moe_stats(g.h)["calls"] >= 1
        # sticky: the next call is refused before anything is enqueued
        xd = g.to_dev(x)
        out = g.out_buf(3)
        with pytest.raises(moe.MoeError) as ei:
            moe.moe_layer_forward(g.h, xd.data_ptr(), g.router[0].data_ptr(), 0, 3, out.data_ptr())
        assert ei.value.code == moe.MOE_ERR_TIMEOUT
        # the safe point resets the cache; the layer is correct again
        moe.moe_cache_config(g.h, 12, moe.MOE_CACHE_LOG_EVENTS | moe.MOE_CACHE_HOST_MISSES)
        o = OracleStack(shape, 31, 2, 12, prefetch=False)
        for layer, T, step in ((0, 3, 1), (1, 5, 1), (0, 3, 2)):
            xs = synth.hidden_states(shape, 31, layer, T, step)
            compare(g.forward(layer, xs), o.forward(layer, xs))
    finally:
        g.close()
