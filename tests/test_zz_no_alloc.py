"""moe_route_topk_noalloc: the allocation-free router entry point, for callers
that cannot call cudaMalloc (a plugin whose host framework's pool owns the
device memory, or a path that must not allocate). On two calls in a row (the
second reuses the shared scratch array the first one left behind) its top-k
indices must equal, bit for bit, and its gates must match within 1e-5, both the
oracle's routing of the same inputs and the routing that moe_layer_forward
computes for them.

This file sorts last so that a run stopping at its first failure has already
run every other test."""
import numpy as np
import pytest

import synth

pytestmark = pytest.mark.gpu


def test_noalloc_router_matches_oracle_and_layer_forward_twice():
    import torch
    if not torch.cuda.is_available():
        pytest.skip("no CUDA device")
    from expert_offload_softmax_b300 import build
    build.build()
    import expert_offload_softmax_b300 as moe
    import oracle
    from moe_harness import GpuStack, act_to_f32

    shape = synth.Shape("noalloc-1L-H512-E64-k8-I128-nvfp4", L=1, E=64, k=8, H=512, I=128,
                        fmt=synth.FMT_NVFP4, act=synth.ACT_BF16, zipf_s=1.0)
    g = GpuStack(shape, 21, 1, 64)
    router_f32 = act_to_f32(synth.router_weights(shape, 21, 0), shape)
    try:
        for call, T in enumerate((37, 5)):
            hidden = synth.hidden_states(shape, 21, 0, T, step=call)
            ref = g.forward(0, hidden)                       # existing entry point
            orc = oracle.route(act_to_f32(hidden, shape), router_f32, shape.k)
            x = g.to_dev(hidden)
            idx = torch.full((T * shape.k,), -1, dtype=torch.int32, device=g.dev)
            gates = torch.zeros((T * shape.k,), dtype=torch.float32, device=g.dev)
            moe.moe_route_topk_noalloc(x.data_ptr(), g.router[0].data_ptr(), T, shape.E, shape.H, shape.k,
                                       moe.MOE_ACT_BF16, idx.data_ptr(), gates.data_ptr(),
                                       g.stream.cuda_stream)
            g.stream.synchronize()
            got_idx = idx.cpu().numpy().reshape(T, shape.k)
            got_gates = gates.cpu().numpy().reshape(T, shape.k).astype(np.float64)
            np.testing.assert_array_equal(got_idx, orc["topk_idx"])
            assert np.abs(got_gates - orc["gates"]).max() <= 1e-5
            np.testing.assert_array_equal(got_idx, ref["topk_idx"])
            assert np.abs(got_gates - ref["gates"]).max() <= 1e-5
        # sizes beyond the scratch array, and token counts beyond the logits
        # grid, are rejected with nothing launched
        for T, E, k in ((moe.MOE_ROUTE_NOALLOC_MAX_LOGITS, shape.E, shape.k), (8 * 65535 + 1, 1, 1)):
            with pytest.raises(moe.MoeError) as ei:
                moe.moe_route_topk_noalloc(x.data_ptr(), g.router[0].data_ptr(), T, E, shape.H, k,
                                           moe.MOE_ACT_BF16, idx.data_ptr(), gates.data_ptr(),
                                           g.stream.cuda_stream)
            assert ei.value.code == moe.MOE_ERR_INVALID
    finally:
        g.close()
