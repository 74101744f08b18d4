"""Pins for the oracle's router (logits, softmax + top-k + renormalisation) and
permutation, against brute force, exact arithmetic and invariants."""
import itertools
import os

import numpy as np
import pytest

import oracle
import synth

GOLDEN = os.path.join(os.path.dirname(__file__), "golden")


def test_logit_order_golden():
    """Every hand-worked case of the fixture: the chunk -> partial mapping and
    the order in which the 32 partials are combined."""
    lines = [l for l in open(os.path.join(GOLDEN, "logit_order.txt")) if l.strip() and not l.startswith("#")]
    assert len(lines) >= 2
    for line in lines:
        lhs, rhs = line.split("->")
        parts = lhs.split()
        H = int(parts[0])
        w = np.zeros((1, H), np.float32)
        for p in parts[1:]:
            i, v = p.split(":")
            w[0, int(i)] = float(v)
        x = np.ones((1, H), np.float32)
        assert oracle.router_logits(x, w)[0, 0] == float(rhs), line


def test_logits_match_exact_sum_on_integers():
    # small integers: every partial sum is exact in fp32, so any order gives the
    # exact value; catches a transposed operand or a dropped chunk
    rng = np.random.default_rng(0)
    for (T, E, H) in ((3, 5, 64), (2, 7, 264), (4, 8, 1024)):
        x = rng.integers(-8, 9, (T, H)).astype(np.float32)
        w = rng.integers(-8, 9, (E, H)).astype(np.float32)
        exact = x.astype(np.float64) @ w.astype(np.float64).T
        assert np.array_equal(oracle.router_logits(x, w), exact.astype(np.float32))


def test_logits_close_to_fp64_on_gaussians():
    rng = np.random.default_rng(1)
    T, E, H = 6, 16, 2048
    x = rng.standard_normal((T, H)).astype(np.float32)
    w = (rng.standard_normal((E, H)) * 0.02).astype(np.float32)
    ref = x.astype(np.float64) @ w.astype(np.float64).T
    got = oracle.router_logits(x, w).astype(np.float64)
    bound = H * 2.0 ** -23 * (np.abs(x).astype(np.float64) @ np.abs(w).astype(np.float64).T)
    assert np.all(np.abs(got - ref) <= bound)


def _dominant(logits_row, k):
    """All k-subsets S such that every i in S beats every j outside S under
    (larger logit, then lower index)."""
    E = len(logits_row)
    out = []
    for S in itertools.combinations(range(E), k):
        ok = True
        for i in S:
            for j in range(E):
                if j in S:
                    continue
                li, lj = logits_row[i], logits_row[j]
                if not (li > lj or (li == lj and i < j)):
                    ok = False
        if ok:
            out.append(S)
    return out


@pytest.mark.parametrize("seed", range(6))
def test_topk_brute_force_with_ties(seed):
    rng = np.random.default_rng(seed)
    T, E, k = 16, 8, 2
    # integer logits in a small range force many exact ties
    logits = rng.integers(-2, 3, (T, E)).astype(np.float32)
    idx, gates = oracle.router_topk(logits, k)
    for t in range(T):
        subsets = _dominant(list(logits[t]), k)
        assert len(subsets) == 1
        assert set(idx[t]) == set(subsets[0])
        # order: logit descending, then index ascending
        keyed = sorted(subsets[0], key=lambda e: (-logits[t, e], e))
        assert list(idx[t]) == keyed


def test_topk_brute_force_tiny_config_inputs():
    shape = synth.TINY_FP32
    x = synth.hidden_states(shape, 0, 0, 4)
    w = synth.router_weights(shape, 0, 0)
    lg = oracle.router_logits(x, w)
    idx, _ = oracle.router_topk(lg, shape.k)
    for t in range(4):
        (S,) = _dominant(list(lg[t]), shape.k)
        assert set(idx[t]) == set(S)


def test_gates_renormalised_and_equal_softmax_over_selected():
    rng = np.random.default_rng(3)
    T, E, k = 64, 256, 8
    logits = (rng.standard_normal((T, E)) * 2.0).astype(np.float32)
    idx, gates, probs = oracle.router_topk(logits, k, want_probs=True)
    assert np.all(np.abs(gates.astype(np.float64).sum(1) - 1.0) <= 1e-6)
    assert np.all(np.abs(probs.astype(np.float64).sum(1) - 1.0) <= 1e-5)
    sel = np.take_along_axis(logits.astype(np.float64), idx.astype(np.int64), 1)
    ref = np.exp(sel - sel.max(1, keepdims=True))
    ref /= ref.sum(1, keepdims=True)
    assert np.max(np.abs(gates - ref)) <= 1e-6
    # the selected experts carry the k largest probabilities
    for t in range(T):
        assert probs[t, idx[t]].min() >= np.sort(probs[t])[-k]


def test_topk_k_equals_E_and_k_one():
    logits = np.array([[0.5, 2.0, 2.0, -1.0]], np.float32)
    idx, g = oracle.router_topk(logits, 1)
    assert idx[0, 0] == 1 and g[0, 0] == 1.0
    idx, g = oracle.router_topk(logits, 4)
    assert list(idx[0]) == [1, 2, 0, 3]
    assert abs(g.sum() - 1) < 1e-6


def _check_perm(idx, E, r):
    T, k = idx.shape
    n = T * k
    flat = idx.reshape(-1)
    assert np.array_equal(r["counts"], np.bincount(flat, minlength=E))
    assert r["offsets"][0] == 0 and r["offsets"][-1] == n
    assert np.array_equal(np.diff(r["offsets"]), r["counts"])
    assert np.array_equal(np.sort(r["perm"]), np.arange(n))          # bijection
    assert np.array_equal(r["inv_perm"][r["perm"]], np.arange(n))    # inverse
    for e in range(E):
        rows = r["perm"][r["offsets"][e]:r["offsets"][e + 1]]
        assert np.all(flat[rows] == e)
        assert np.all(np.diff(rows) > 0)                              # stable
    assert np.array_equal(r["uniq"], np.nonzero(r["counts"])[0])


@pytest.mark.parametrize("T,E,k", [(1, 8, 2), (4, 8, 2), (8, 256, 8), (300, 64, 6), (0, 8, 2)])
def test_permutation_invariants(T, E, k):
    rng = np.random.default_rng(T * 1000 + E)
    idx = np.stack([rng.permutation(E)[:k] for _ in range(T)]) if T else np.zeros((0, k), np.int32)
    r = oracle.permute(idx.astype(np.int32), E)
    _check_perm(idx.astype(np.int32), E, r)


def test_permutation_golden_small():
    # T=3, k=2: assignments a = t*k + j
    idx = np.array([[2, 0], [0, 3], [2, 3]], np.int32)
    r = oracle.permute(idx, 4)
    assert list(r["counts"]) == [2, 0, 2, 2]
    assert list(r["offsets"]) == [0, 2, 2, 4, 6]
    assert list(r["perm"]) == [1, 2, 0, 4, 3, 5]
    assert list(r["uniq"]) == [0, 2, 3]
