"""Pins of the oracle's router step (softmax over the router logits, then
top-k), the step before the route layout ("feat(pytorch): add CuTeDSL W4A16 MoE
backend" (LMDeploy), section Benchmark: routes come from a router score / top-k
computation; routing weights are FP32, renormalize=False).

Each check ties the oracle to something other than itself: closed forms,
invariants of softmax, and a brute-force pure-Python implementation over
every expert subset on tiny inputs."""
import itertools
import math

import numpy as np
import pytest

import oracle


def test_equal_logits_pick_the_lowest_indices_with_uniform_weights():
    G, k = 12, 5
    ids, w = oracle.route_topk(np.full((3, G), 0.25, np.float32), k)
    assert (ids == np.arange(k, dtype=np.int32)).all()
    assert np.allclose(w, 1.0 / G, rtol=0, atol=1e-15)


def test_one_dominant_logit():
    G, k, hot = 16, 4, 11
    lg = np.zeros((1, G), np.float32)
    lg[0, hot] = 40.0
    ids, w = oracle.route_topk(lg, k)
    assert ids[0, 0] == hot
    assert list(ids[0, 1:]) == [0, 1, 2]  # ties among the rest: lowest index first
    rest = math.exp(-40.0)
    denom = 1.0 + (G - 1) * rest
    assert w[0, 0] == pytest.approx(1.0 / denom, rel=1e-15)
    assert np.allclose(w[0, 1:], rest / denom, rtol=1e-12, atol=0)


def _brute_force(logits, k):
    """Every k-subset; the chosen one has no outside expert with a larger logit,
    nor an equal logit at a lower index; order: descending logit, then index."""
    G = len(logits)
    chosen = None
    for sub in itertools.combinations(range(G), k):
        inside = set(sub)
        ok = True
        for i in inside:
            for o in range(G):
                if o in inside:
                    continue
                if logits[o] > logits[i] or (logits[o] == logits[i] and o < i):
                    ok = False
        if ok:
            assert chosen is None, "two subsets qualify"
            chosen = sub
    order = sorted(chosen, key=lambda e: (-float(logits[e]), e))
    m = max(float(v) for v in logits)
    ex = [math.exp(float(v) - m) for v in logits]
    s = math.fsum(ex)
    return order, [ex[e] / s for e in order]


@pytest.mark.parametrize("seed", range(6))
def test_brute_force_tiny(seed):
    rng = np.random.default_rng(seed)
    T, G, k = 5, 7, 3
    lg = rng.standard_normal((T, G)).astype(np.float32)
    lg[1, 2] = lg[1, 5]  # an exact tie
    lg[3, :] = lg[3, 0]  # all equal
    ids, w = oracle.route_topk(lg, k)
    for t in range(T):
        order, ww = _brute_force(lg[t], k)
        assert list(ids[t]) == order
        assert np.allclose(w[t], ww, rtol=1e-13, atol=0)


def test_shift_invariance_and_full_selection_sums_to_one():
    rng = np.random.default_rng(7)
    lg = rng.standard_normal((4, 9)).astype(np.float32)
    ids_a, w_a = oracle.route_topk(lg, 9)
    ids_b, w_b = oracle.route_topk(lg + np.float32(3.0), 9)
    assert (ids_a == ids_b).all()
    assert np.allclose(w_a, w_b, rtol=1e-6, atol=0)  # the shift itself rounds in FP32
    assert np.allclose(w_a.sum(axis=1), 1.0, rtol=0, atol=1e-13)
    assert (np.diff(w_a, axis=1) <= 0).all()  # descending
