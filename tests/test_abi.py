"""The C-ABI library builds, loads and exports every symbol the header declares
(no GPU needed); host-side validation answers with status codes."""
import ctypes
import os
import re

import pytest

import expert_offload_softmax_b300 as moe
from expert_offload_softmax_b300 import build

ROOT = os.path.dirname(os.path.dirname(os.path.abspath(__file__)))


def _declared():
    src = open(os.path.join(ROOT, "include", "moe.h")).read()
    src = re.sub(r"/\*.*?\*/", "", src, flags=re.S)
    return sorted(set(re.findall(r"\b(moe_[a-z_]+)\s*\(", src)))


def test_library_builds_and_exports_every_declared_symbol():
    build.build()
    lib = ctypes.CDLL(moe.LIB_PATH)
    names = _declared()
    assert "moe_layer_forward" in names and len(names) >= 10
    for n in names:
        assert hasattr(lib, n), n
    assert sorted(moe.EXPORTS) == names


def test_expert_bytes_layout():
    # NVFP4, H=2048, I=512: 3*H*I/2 code bytes + 3*H*I/16 scale bytes + 16, each part 256-aligned
    d = moe.make_desc(40, 256, 8, 2048, 512, moe.MOE_FMT_NVFP4, moe.MOE_ACT_BF16)
    n = moe.moe_expert_bytes(d)
    assert 1769488 <= n < 1769488 + 2048
    d = moe.make_desc(40, 256, 8, 2048, 512, moe.MOE_FMT_BF16, moe.MOE_ACT_BF16)
    assert 6291456 <= moe.moe_expert_bytes(d) < 6291456 + 2048


@pytest.mark.parametrize("bad", [
    dict(L=0), dict(E=0), dict(E=2000), dict(k=0), dict(k=9, E=8), dict(H=100), dict(I=100),
    dict(fmt=7), dict(shared=2),
])
def test_invalid_shapes_rejected(bad):
    p = dict(L=1, E=8, k=2, H=256, I=128, fmt=moe.MOE_FMT_NVFP4, act=moe.MOE_ACT_BF16, shared=0)
    p.update(bad)
    d = moe.make_desc(p["L"], p["E"], p["k"], p["H"], p["I"], p["fmt"], p["act"], shared=p["shared"])
    with pytest.raises(moe.MoeError) as ei:
        moe.moe_expert_bytes(d)
    assert ei.value.code == moe.MOE_ERR_INVALID


def test_init_without_gpu_reports_error_code():
    import torch
    if torch.cuda.is_available():
        pytest.skip("a GPU is present")
    d = moe.make_desc(1, 8, 2, 64, 32, moe.MOE_FMT_FP32, moe.MOE_ACT_FP32)
    with pytest.raises(moe.MoeError) as ei:
        moe.moe_init(d)
    assert ei.value.code == moe.MOE_ERR_CUDA
