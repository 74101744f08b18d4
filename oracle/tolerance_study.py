"""ORACLE — test infrastructure, not the product.

Tolerance study for a block-scaled tensor-core MMA in the prefill experts: how
far the layer output moves from the layer as specified when the activations
(x before gate/up, h before down) are quantised the way such an MMA needs
(oracle.quant_act: MXFP8 with E4M3 elements for kind::mxf8f6f4, NVFP4 for
kind::mxf4nvf4). Uses only the oracle and the seeded generator.

    python -m oracle.tolerance_study [--tokens N]

Prints, per workload shape and quantiser, the layer's error metric
max|y - y_exact| / max|y_exact| over the sampled tokens' output rows, and the
same per row (the worst row)."""
from __future__ import annotations

import argparse
import os
import sys

import numpy as np

sys.path.insert(0, os.path.dirname(os.path.dirname(os.path.abspath(__file__))))

import oracle  # noqa: E402
import synth  # noqa: E402


def study(shape, T: int, seed: int = 0, layer: int = 0):
    act_bf16 = shape.act == synth.ACT_BF16
    x = oracle.act_to_f32(synth.hidden_states(shape, seed, layer, T, 0), act_bf16)
    w = oracle.act_to_f32(synth.router_weights(shape, seed, layer), act_bf16)
    r = oracle.route(x, w, shape.k)
    idx, gates = r["topk_idx"], r["gates"]
    need = sorted(set(int(e) for e in np.unique(idx)) | set(range(shape.E, shape.E + shape.shared)))
    W = {e: oracle.dequant_expert(shape.fmt, synth.expert_weights(shape, seed, layer, e), shape.H, shape.I)
         for e in need}
    outs = {0: [], oracle.QUANT_MXFP8: [], oracle.QUANT_NVFP4: []}
    for t in range(T):
        experts = [int(e) for e in idx[t]] + list(range(shape.E, shape.E + shape.shared))
        for kind in outs:
            ys = [oracle.expert_ffn(x[t], *W[e], mode=shape.act_mode)[0] if kind == 0 else
                  oracle.expert_ffn_q(x[t], *W[e], kind, mode=shape.act_mode) for e in experts]
            outs[kind].append(oracle.combine(gates[t], ys))
    ref = np.array(outs[0], np.float64)
    res = {}
    for kind in (oracle.QUANT_MXFP8, oracle.QUANT_NVFP4):
        y = np.array(outs[kind], np.float64)
        d = np.abs(y - ref)
        res[kind] = (d.max() / np.abs(ref).max(), max(d[i].max() / np.abs(ref[i]).max() for i in range(T)))
    return res


def main():
    ap = argparse.ArgumentParser()
    ap.add_argument("--tokens", type=int, default=16)
    args = ap.parse_args()
    print("| workload | weights | activations quantised to | max err / max out (tensor) | worst row |")
    print("|---|---|---|---|---|")
    for shape in (synth.DECODE_NVFP4, synth.LARGE_MXFP4, synth.DECODE_FP8):
        res = study(shape, args.tokens)
        wname = {synth.FMT_NVFP4: "NVFP4", synth.FMT_MXFP4: "MXFP4", synth.FMT_FP8: "FP8"}[shape.fmt]
        for kind, name in ((oracle.QUANT_MXFP8, "MXFP8 (E4M3, E8M0 per 32)"),
                           (oracle.QUANT_NVFP4, "NVFP4 (E2M1, E4M3 per 16)")):
            a, b = res[kind]
            print(f"| {shape.name}, {args.tokens} tokens | {wname} | {name} | {a:.4f} | {b:.4f} |")
        sys.stdout.flush()


if __name__ == "__main__":
    main()
