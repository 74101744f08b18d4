"""Test and benchmark harness: drives the CUDA library through its C ABI on
seeded synthetic inputs, and the oracle on the same inputs, and compares them.
Only tests/, bench.py and __graft_entry__ use it."""
from __future__ import annotations

import numpy as np

import expert_offload_softmax_b300 as moe
import synth

TOL = 2e-2  # max |y - y_ref| / max |y_ref| per output tensor (bf16 I/O, fp32 accumulate)


def rel_err(y, ref) -> float:
    y = np.asarray(y, np.float64)
    ref = np.asarray(ref, np.float64)
    m = np.abs(ref).max()
    return float(np.abs(y - ref).max() / (m if m > 0 else 1.0))


def act_to_f32(x, shape):
    import oracle
    return oracle.bf16_to_f32(x) if shape.act == synth.ACT_BF16 else np.asarray(x, np.float32)


class GpuStack:
    """One library handle for ``L`` layers of ``shape`` with seeded weights.
    ``routers`` optionally replaces the seeded router matrices (one per layer,
    in the activation encoding)."""

    def __init__(self, shape: synth.Shape, seed: int, L: int, capacity: int, flags: int = 0,
                 max_tokens: int = 0, device: int = 0, routers=None):
        import torch
        self.torch = torch
        self.shape, self.seed, self.L = shape, seed, L
        self.dev = torch.device("cuda", device)
        desc = moe.make_desc(L, shape.E, shape.k, shape.H, shape.I, shape.fmt, shape.act,
                             shared=shape.shared, mode=shape.act_mode, max_tokens=max_tokens, device=device)
        self.h = moe.moe_init(desc)
        for l in range(L):
            for e in range(shape.E + shape.shared):
                moe.moe_load_expert(self.h, l, e, synth.expert_weights(shape, seed, l, e))
        moe.moe_cache_config(self.h, capacity, flags | moe.MOE_CACHE_LOG_EVENTS)
        self.router = [self.to_dev(routers[l] if routers is not None else synth.router_weights(shape, seed, l))
                       for l in range(L)]
        self.stream = torch.cuda.Stream(device=self.dev)

    def reconfigure(self, capacity: int, flags: int = 0, pool=None):
        """A safe point: empty the cache and rebuild the pool with ``capacity``
        slots (``pool``: optional caller-owned torch uint8 device tensor)."""
        moe.moe_cache_config(self.h, capacity, flags | moe.MOE_CACHE_LOG_EVENTS,
                             pool.data_ptr() if pool is not None else 0, pool.numel() if pool is not None else 0)

    def resize(self, capacity: int, pool=None):
        moe.moe_cache_resize(self.h, capacity, pool.data_ptr() if pool is not None else 0,
                             pool.numel() if pool is not None else 0)

    def to_dev(self, a: np.ndarray):
        t = self.torch
        if a.dtype == np.uint16:
            return t.from_numpy(a.view(np.int16)).to(self.dev).view(t.bfloat16)
        return t.from_numpy(np.ascontiguousarray(a)).to(self.dev)

    def out_buf(self, T):
        t = self.torch
        dt = t.bfloat16 if self.shape.act == synth.ACT_BF16 else t.float32
        return t.empty((T, self.shape.H), dtype=dt, device=self.dev)

    def forward_dev(self, layer: int, x_dev, out_dev, T: int):
        moe.moe_layer_forward(self.h, x_dev.data_ptr(), self.router[layer].data_ptr(), layer, T,
                              out_dev.data_ptr(), self.stream.cuda_stream)

    def forward(self, layer: int, hidden: np.ndarray):
        T = hidden.shape[0]
        x = self.to_dev(hidden)
        out = self.out_buf(T)
        self.torch.cuda.synchronize(self.dev)
        self.forward_dev(layer, x, out, T)
        moe.moe_sync(self.h)
        self.stream.synchronize()
        o = out.float().cpu().numpy()
        r = moe.moe_debug_routing(self.h, T, self.shape.k, self.shape.E)
        r["out"] = o
        r["events"] = moe.moe_stats_events(self.h)
        return r

    def stats(self):
        return moe.moe_stats(self.h)

    def close(self):
        if self.h:
            moe.moe_destroy(self.h)
            self.h = None


class OracleStack:
    """The oracle's view of the same stack: routing, LRU and sampled outputs.
    Output rows of many tokens are computed one expert at a time in worker
    processes (``workers`` > 1): each expert's output for every sampled token
    routed to it, then each token's combine in selection order; the same
    oracle functions as the single-process path, in the same order."""

    def __init__(self, shape: synth.Shape, seed: int, L: int, capacity: int, prefetch: bool,
                 max_cached_experts: int = 64, routers=None, workers: int = 0):
        import oracle
        self.o = oracle
        self.shape, self.seed, self.L = shape, seed, L
        self.lru = oracle.LRU(L, shape.E, capacity)
        self.prefetch = prefetch
        self.workers = workers
        self.router = [act_to_f32(routers[l] if routers is not None else synth.router_weights(shape, seed, l), shape)
                       for l in range(L)]
        self.cache = {}
        self.max_cached = max_cached_experts

    def resize(self, capacity: int):
        self.lru.resize(capacity)

    def weights(self, layer, e):
        key = (layer, e)
        if key not in self.cache:
            if len(self.cache) >= self.max_cached:
                self.cache.pop(next(iter(self.cache)))
            w = synth.expert_weights(self.shape, self.seed, layer, e)
            self.cache[key] = self.o.dequant_expert(self.shape.fmt, w, self.shape.H, self.shape.I)
        return self.cache[key]

    def forward(self, layer: int, hidden: np.ndarray, toks=None):
        s = self.shape
        x = act_to_f32(hidden, s)
        r = self.o.route(x, self.router[layer], s.k)
        T = x.shape[0]
        ev = self.lru.access(layer, r["uniq"], T, self.prefetch)
        r["events"] = np.stack([ev["layer"], ev["expert"], ev["hit"], ev["slot"], ev["evicted"],
                                ev["prefetch"]], axis=1)
        if isinstance(toks, str) and toks.startswith("cover:"):
            toks = cover_tokens(r["topk_idx"], int(toks.split(":")[1]))
        toks = np.arange(T) if toks is None else np.asarray(toks)
        if len(toks) and self.workers > 1:
            r["out"] = oracle_rows_parallel(s, self.seed, layer, x, r["topk_idx"], r["gates"], toks, self.workers)
        elif len(toks):
            need = sorted(set(int(e) for e in np.unique(r["topk_idx"][toks])) |
                          set(range(s.E, s.E + s.shared)))
            ws = {e: self.weights(layer, e) for e in need}
            r["out"] = self.o.layer_tokens(x, r["topk_idx"], r["gates"], ws, s.E, s.shared, s.act_mode, toks)
        r["toks"] = toks
        return r


def cover_tokens(topk: np.ndarray, n: int) -> np.ndarray:
    """At least ``n`` token indices (ascending) such that every expert the call
    routes to is selected by one of them: tokens that add a not yet covered
    expert, taken in token order, then evenly spaced tokens up to n."""
    T = topk.shape[0]
    seen, pick = set(), []
    for t in range(T):
        new = set(int(e) for e in topk[t]) - seen
        if new:
            seen |= new
            pick.append(t)
    rest = np.linspace(0, T - 1, min(T, n)).round().astype(int)
    return np.array(sorted(set(pick) | set(int(t) for t in rest)), dtype=np.int64)


def _expert_rows(job):
    """Worker: one expert's outputs (fp32 [n, H]) for the given token rows."""
    import oracle
    shape, seed, layer, e, xs = job
    w = synth.expert_weights(shape, seed, layer, e)
    Wg, Wu, Wd = oracle.dequant_expert(shape.fmt, w, shape.H, shape.I)
    return e, np.stack([oracle.expert_ffn(xr, Wg, Wu, Wd, shape.act_mode)[0] for xr in xs])


def oracle_rows_parallel(shape, seed, layer, x, topk, gates, toks, workers):
    """Oracle output rows for tokens ``toks``: expert outputs in ``workers``
    spawned processes (none touches a GPU), then the oracle's combine per token."""
    import multiprocessing as mp
    import oracle
    k = topk.shape[1]
    users = {}
    for t in toks:
        for e in topk[t]:
            users.setdefault(int(e), []).append(int(t))
    for e in range(shape.E, shape.E + shape.shared):
        users[e] = [int(t) for t in toks]
    jobs = [(shape, seed, layer, e, x[ts]) for e, ts in sorted(users.items())]
    with mp.get_context("spawn").Pool(min(workers, len(jobs))) as pool:
        done = dict(pool.imap_unordered(_expert_rows, jobs))
    pos = {e: {t: i for i, t in enumerate(ts)} for e, ts in users.items()}
    out = np.empty((len(toks), shape.H), np.float32)
    for i, t in enumerate(toks):
        t = int(t)
        ys = [done[int(e)][pos[int(e)][t]] for e in topk[t]]
        ys += [done[e][pos[e][t]] for e in range(shape.E, shape.E + shape.shared)]
        out[i] = oracle.combine(gates[t], ys)
    return out


def oracle_workers() -> int:
    import os
    return max(1, min(32, (os.cpu_count() or 2) - 1))


def rel_err_rows(y, ref) -> float:
    """Largest per-row error max_h |y - ref| / max_h |ref| (rows of very
    different magnitude are each held to the tolerance)."""
    y = np.asarray(y, np.float64)
    ref = np.asarray(ref, np.float64)
    m = np.abs(ref).max(axis=1)
    m[m == 0] = 1.0
    return float((np.abs(y - ref).max(axis=1) / m).max())


def compare(g: dict, o: dict, check_out: bool = True) -> dict:
    """Asserts bit-exact routing / permutation / cache events and the output
    tolerance; returns the measured errors."""
    np.testing.assert_array_equal(g["topk_idx"], o["topk_idx"])
    np.testing.assert_array_equal(g["perm"], o["perm"])
    np.testing.assert_array_equal(g["counts"], o["counts"])
    np.testing.assert_array_equal(g["uniq"], o["uniq"])
    np.testing.assert_array_equal(g["events"], o["events"])
    gerr = float(np.abs(g["gates"].astype(np.float64) - o["gates"]).max()) if g["gates"].size else 0.0
    assert gerr <= 1e-5, gerr
    res = {"gate_err": gerr}
    if check_out and len(o["toks"]):
        err = rel_err(g["out"][o["toks"]], o["out"])
        res["out_err"] = err
        assert err <= TOL, err
    return res
