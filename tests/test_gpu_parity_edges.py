"""Edge cases of the CUDA path against the oracle, through the C ABI.

Same bar as the other parity tests: top-k, permutation, counts, unique experts
and the LRU event sequence bit-exact; gates within 1e-5; outputs within 2e-2
of max |y_ref| (here per token row where rows differ in magnitude).

 * exact logit ties: duplicated router rows give bit-identical logits; the
   lower expert index must win, in order, on lanes of one warp and across the
   32-expert lane stride, in decode (T = 1, 8) and prefill (T = 300);
 * activation range: token rows with |x| up to 1e5 and down to 1e-6, decode and
   prefill, NVFP4 and MXFP4 weights;
 * block-scale bytes: every finite E4M3 byte (subnormals, zeros and negative
   scales included) and E8M0 bytes 100..154, decode and prefill."""
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


# groups of experts whose router rows are made identical: adjacent lanes, the
# same lane one 32-expert stride apart, and a three-way tie across both
TIE_GROUPS = ((4, 5), (3, 35), (10, 42, 43))


def tied_routers(shape, seed, L):
    """Seeded router matrices with the rows of each tie group made identical
    and lifted (column 0, which meets hidden[:, 0] = 1) so that they are selected."""
    out = []
    for l in range(L):
        w = synth.router_weights(shape, seed, l)
        lift = synth.f32_to_bf16_bits(np.array([3.0], np.float32))[0] if shape.act == synth.ACT_BF16 else 3.0
        for grp in TIE_GROUPS:
            w[grp[0], 0] = lift
            for e in grp[1:]:
                w[e] = w[grp[0]]
        out.append(w)
    return out


def _hidden_col0_one(shape, seed, layer, T, step):
    x = synth.hidden_states(shape, seed, layer, T, step)
    x[:, 0] = 0x3F80 if shape.act == synth.ACT_BF16 else 1.0
    return x


@pytest.mark.parametrize("fmt,T", [(synth.FMT_NVFP4, 1), (synth.FMT_NVFP4, 8), (synth.FMT_BF16, 8),
                                   (synth.FMT_MXFP4, 300)])
def test_exact_logit_ties_pick_lower_index(fmt, T):
    from moe_harness import GpuStack, OracleStack, compare
    s = synth.Shape("ties", L=2, E=64, k=8, H=256, I=128, fmt=fmt, act=synth.ACT_BF16)
    routers = tied_routers(s, 41, 2)
    g = GpuStack(s, 41, 2, 128, max_tokens=max(T, 8), routers=routers)
    o = OracleStack(s, 41, 2, 128, prefetch=False, routers=routers)
    try:
        for step in range(3):
            for layer in range(2):
                x = _hidden_col0_one(s, 41, layer, T, step)
                gr, orr = g.forward(layer, x), o.forward(layer, x, None if T <= 8 else np.arange(0, T, 7))
                compare(gr, orr)
                # the ties really were ties, and both members of a group were selected together
                idx = orr["topk_idx"]
                for grp in TIE_GROUPS:
                    lg = orr["logits"][:, list(grp)]
                    assert (lg == lg[:, :1]).all()
                    sel = np.isin(idx, grp)
                    assert sel.any()
                    for t in range(T):
                        pos = [int(np.where(idx[t] == e)[0][0]) for e in grp if e in idx[t]]
                        assert pos == sorted(pos)  # lower index first among equal logits
    finally:
        g.close()


def _scaled_rows(shape, seed, layer, T, step):
    """Hidden rows N(0,1) with row 0 scaled to max |x| ~ 1e5, row 1 to ~1e-6 and
    row 2 mixing both ranges (half its elements tiny); rows beyond stay N(0,1)."""
    from moe_harness import act_to_f32
    x = act_to_f32(synth.hidden_states(shape, seed, layer, T, step), shape).astype(np.float32)
    x[0] *= np.float32(1e5) / np.abs(x[0]).max()
    if T > 1:
        x[1] *= np.float32(1e-6) / np.abs(x[1]).max()
    if T > 2:
        x[2, ::2] *= np.float32(1e-6)
    return synth.f32_to_bf16_bits(x)


@pytest.mark.parametrize("fmt", [synth.FMT_NVFP4, synth.FMT_MXFP4, synth.FMT_FP8])
@pytest.mark.parametrize("T", [3, 8, 40])
def test_activation_range(fmt, T):
    from moe_harness import GpuStack, OracleStack, compare, rel_err_rows, TOL
    s = synth.Shape("range", L=2, E=16, k=4, H=512, I=256, fmt=fmt, act=synth.ACT_BF16)
    g = GpuStack(s, 43, 2, 32, max_tokens=64)
    o = OracleStack(s, 43, 2, 32, prefetch=False)
    try:
        for layer, step in ((0, 0), (1, 0), (0, 1)):
            x = _scaled_rows(s, 43, layer, T, step)
            gr, orr = g.forward(layer, x), o.forward(layer, x)
            compare(gr, orr)
            assert np.isfinite(gr["out"]).all()
            assert rel_err_rows(gr["out"], orr["out"]) <= TOL
    finally:
        g.close()


@pytest.mark.parametrize("fmt,table", [(synth.FMT_NVFP4, synth.E4M3_FINITE_BYTES),
                                       (synth.FMT_MXFP4, synth.E8M0_WIDE_BYTES)])
@pytest.mark.parametrize("T", [1, 8, 37])
def test_every_block_scale_byte(fmt, table, T):
    from moe_harness import GpuStack, OracleStack, compare
    s = synth.Shape("scales", L=1, E=16, k=4, H=512, I=256, fmt=fmt, act=synth.ACT_BF16, scale_table=table)
    w = synth.expert_weights(s, 47, 0, 0)
    drawn = set(np.unique(np.concatenate([w[p]["scales"].ravel() for p in ("gate", "up", "down")])).tolist())
    assert drawn == set(table)
    g = GpuStack(s, 47, 1, 16, max_tokens=64)
    o = OracleStack(s, 47, 1, 16, prefetch=False)
    try:
        for step in range(3):
            x = synth.hidden_states(s, 47, 0, T, step)
            compare(g.forward(0, x), o.forward(0, x))
    finally:
        g.close()


@pytest.mark.parametrize("T", [1, 8, 37])
def test_every_fp8_code_byte(T):
    """FP8 weights drawn from every finite E4M3 byte (zeros of both signs,
    subnormals down to 2^-9, +-448): each widens to f16 / bf16 exactly."""
    from moe_harness import GpuStack, OracleStack, compare
    s = synth.Shape("codes8", L=1, E=16, k=4, H=512, I=256, fmt=synth.FMT_FP8, act=synth.ACT_BF16,
                    code_table=synth.E4M3_FINITE_BYTES)
    w = synth.expert_weights(s, 48, 0, 0)
    drawn = set(np.unique(np.concatenate([w[p]["codes"].ravel() for p in ("gate", "up", "down")])).tolist())
    assert drawn == set(synth.E4M3_FINITE_BYTES)
    g = GpuStack(s, 48, 1, 16, max_tokens=64)
    o = OracleStack(s, 48, 1, 16, prefetch=False)
    try:
        for step in range(3):
            x = synth.hidden_states(s, 48, 0, T, step)
            compare(g.forward(0, x), o.forward(0, x))
    finally:
        g.close()
