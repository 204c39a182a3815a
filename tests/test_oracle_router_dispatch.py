"""Pins of the oracle's router (top-k, weights) and pull schedule, on the CPU.

Top-k is pinned by brute-force enumeration of every k-subset; the router weights by closed-form
softmax identities; the pull schedule by the worked example of the page "Метод и эксперименты"
(tests/golden/pull_dispatch_example.txt) and by permutation/ordering properties.
"""

import itertools
import math
import os

import numpy as np
import pytest

import oracle

GOLDEN = os.path.join(os.path.dirname(__file__), "golden")


def _beats(l, a, b):
    """Expert a ranks before expert b: larger logit, or equal logit and lower index."""
    return l[a] > l[b] or (l[a] == l[b] and a < b)


@pytest.mark.parametrize("E,k", [(8, 2), (6, 3), (5, 1), (4, 4)])
def test_topk_matches_bruteforce_subsets(E, k):
    rng = np.random.default_rng(E * 10 + k)
    T = 40
    l = rng.standard_normal((T, E)).astype(np.float32)
    # plant exact ties, including ties straddling the k-th place
    l[0, :] = 1.0
    l[1, 1] = l[1, 3] = l[1, 0]
    l[2, :] = np.float32(0.5) * np.arange(E)[::-1].astype(np.float32)
    l[2, E - 1] = l[2, E - 2]
    got = oracle.topk_select(l, k)
    for t in range(T):
        valid = []
        for S in itertools.combinations(range(E), k):
            rest = [o for o in range(E) if o not in S]
            if all(_beats(l[t], s, o) for s in S for o in rest):
                valid.append(set(S))
        assert len(valid) == 1, "the tie rule makes the selected set unique"
        assert set(got[t].tolist()) == valid[0]
        # order inside the selection: descending logit, ascending index on ties
        for a, b in zip(got[t][:-1], got[t][1:]):
            assert _beats(l[t], a, b)


def test_router_weights_closed_forms():
    rng = np.random.default_rng(3)
    T, E, k = 30, 8, 3
    l = rng.standard_normal((T, E)) * 3.0
    idx = oracle.topk_select(l.astype(np.float32), k)
    w = oracle.weights_for_selection(l, idx)
    for t in range(T):
        # renormalised full softmax == softmax over the selected logits alone
        den = sum(math.exp(l[t, e]) for e in idx[t])
        for j in range(k):
            assert w[t, j] == pytest.approx(math.exp(l[t, idx[t, j]]) / den, rel=1e-13)
        assert sum(w[t]) == pytest.approx(1.0, abs=1e-14)
        # weights follow the selection order (descending logits)
        assert all(w[t, j] >= w[t, j + 1] for j in range(k - 1))
    # k = E: the weights are the plain softmax probabilities
    idx_all = oracle.topk_select(l.astype(np.float32), E)
    w_all = oracle.weights_for_selection(l, idx_all)
    for t in range(T):
        den = sum(math.exp(v) for v in l[t])
        for j in range(E):
            assert w_all[t, j] == pytest.approx(math.exp(l[t, idx_all[t, j]]) / den, rel=1e-13)


def test_router_bias_shifts_logits():
    rng = np.random.default_rng(5)
    x = rng.standard_normal((4, 6))
    Wr = rng.standard_normal((6, 3))
    b = np.array([10.0, -1.0, 0.25])
    l = oracle.router_logits(x, Wr, b)
    for t in range(4):
        for e in range(3):
            assert l[t, e] == pytest.approx(sum(x[t, i] * Wr[i, e] for i in range(6)) + b[e], rel=1e-13)
    # a large bias forces the selection
    idx = oracle.topk_select(l.astype(np.float32), 1)
    assert (idx[:, 0] == 0).all()


def test_topk_gap():
    l = np.array([[3.0, 1.0, 2.0, 2.0], [0.0, 0.5, 0.25, -1.0]], dtype=np.float32)
    g = oracle.topk_gap(l, 2)
    assert g[0] == 0.0          # tie between the 2nd and 3rd place
    assert g[1] == pytest.approx(0.25)
    assert np.isinf(oracle.topk_gap(l, 4)).all()


def _read_golden():
    routes, expect = {}, {}
    meta = {}
    with open(os.path.join(GOLDEN, "pull_dispatch_example.txt")) as f:
        for line in f:
            line = line.split("#")[0].strip()
            if not line:
                continue
            tok = line.split()
            if tok[0] == "route":
                routes[int(tok[1])] = int(tok[2])
            elif tok[0] == "expect":
                expect[int(tok[1])] = [int(v) for v in tok[2:]]
            else:
                meta[tok[0]] = int(tok[1])
    return meta, routes, expect


def test_dispatch_worked_example():
    meta, routes, expect = _read_golden()
    T, E, k = meta["T"], meta["E"], meta["k"]
    idx = np.array([[routes[t]] for t in range(T)], dtype=np.int32)
    counts, offsets, sorted_tok, inv_pos = oracle.dispatch(idx, E)
    for e in range(E):
        seg = sorted_tok[offsets[e]:offsets[e + 1]].tolist()
        assert seg == expect[e], f"expert {e}"
        assert counts[e] == len(expect[e])
    for t in range(T):
        assert sorted_tok[inv_pos[t, 0]] == t


@pytest.mark.parametrize("T,E,k,seed", [(37, 8, 2, 0), (100, 16, 4, 1), (5, 8, 8, 2), (1, 3, 1, 3)])
def test_dispatch_is_a_stable_permutation(T, E, k, seed):
    rng = np.random.default_rng(seed)
    # distinct experts per token, skewed towards low ids, some experts empty
    p = np.exp(-0.5 * np.arange(E))
    p /= p.sum()
    idx = np.stack([rng.choice(E, size=k, replace=False, p=p) for _ in range(T)]).astype(np.int32)
    counts, offsets, sorted_tok, inv_pos = oracle.dispatch(idx, E)
    assert offsets[0] == 0 and offsets[E] == T * k
    assert (np.diff(offsets) == counts).all()
    assert (counts == np.bincount(idx.ravel(), minlength=E)).all()
    seen = np.zeros(T * k, dtype=int)
    for t in range(T):
        for j in range(k):
            r = inv_pos[t, j]
            seen[r] += 1
            assert sorted_tok[r] == t
            assert offsets[idx[t, j]] <= r < offsets[idx[t, j] + 1]
    assert (seen == 1).all(), "every route lands in exactly one row"
    for e in range(E):
        seg = sorted_tok[offsets[e]:offsets[e + 1]]
        assert (np.diff(seg) > 0).all(), "tokens ascend inside an expert region"
