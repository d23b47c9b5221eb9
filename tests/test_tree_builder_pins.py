"""Pins of the oracle's best-first tree builder (BASTION page, Method §1-§3):
a hand-worked case with equal scores, brute force over every prefix on tiny
vocabularies, the input generator's own builder, tree invariants, and the
budget stop.  CPU only."""
import itertools

import numpy as np
import pytest

import oracle
import workloads


def test_hand_worked_equal_scores():
    # C = 2, all q = 1/2, depth cap 2: the frontier order decides every pop
    q = np.full((2, 2), 0.5)
    par, tok, rho = oracle.best_first(q, 6, 2)
    assert par.tolist() == [-1, -1, 0, 0, 1, 1]
    assert tok.tolist() == [0, 1, 0, 1, 0, 1]
    assert rho.tolist() == [0.5, 0.5, 0.25, 0.25, 0.25, 0.25]


def test_stops_when_frontier_is_empty():
    q = np.array([[0.7, 0.3]])
    par, tok, rho = oracle.best_first(q, 10, 1)
    assert len(par) == 2 and tok.tolist() == [0, 1]


def _paths(par, tok):
    out = []
    for i in range(len(par)):
        p, path = i, []
        while p >= 0:
            path.append(int(tok[p]))
            p = int(par[p])
        out.append(tuple(reversed(path)))
    return out


@pytest.mark.parametrize("C,cap,n,seed", [(2, 4, 9, 0), (3, 3, 20, 1), (3, 4, 40, 2), (2, 5, 31, 3)])
def test_brute_force_top_n_prefixes(C, cap, n, seed):
    """Scores shrink along a path (q <= 1), so best-first adds exactly the n
    highest-scoring prefixes; with continuous random marginals there are no ties."""
    q = np.random.default_rng(seed).dirichlet(np.ones(C), size=cap)
    scored = []
    for d in range(1, cap + 1):
        for xs in itertools.product(range(C), repeat=d):
            scored.append((float(np.prod([q[k, x] for k, x in enumerate(xs)])), xs))
    scored.sort(key=lambda t: -t[0])
    par, tok, rho = oracle.best_first(q, n, cap)
    got = _paths(par, tok)
    assert set(got) == {xs for _, xs in scored[:n]}
    assert np.all(np.diff(rho) <= 0)
    for (r, xs) in zip(rho, got):
        assert r == pytest.approx(np.prod([q[k, x] for k, x in enumerate(xs)]), rel=1e-12)


@pytest.mark.parametrize("C,cap,n,alpha", [(8, 8, 64, 0.3), (8, 16, 256, 0.2), (5, 3, 30, 1.0),
                                           (32, 4, 100, 0.5), (1, 6, 10, 1.0)])
def test_matches_generator_builder(C, cap, n, alpha):
    for seed in range(3):
        q = np.random.default_rng(seed).dirichlet(alpha * np.ones(C), size=cap)
        a = oracle.best_first(q, n, cap)
        b = workloads.tree_best_first(q, n, cap)
        for x, y in zip(a, b):
            assert np.array_equal(x, y)


def test_tree_invariants():
    q = np.random.default_rng(7).dirichlet(0.3 * np.ones(8), size=10)
    par, tok, rho = oracle.best_first(q, 200, 10)
    dep = workloads.depths_from_parents(par)
    assert np.all(par < np.arange(len(par)))
    assert dep.max() <= 10
    for i in range(len(par)):
        up = 1.0 if par[i] < 0 else rho[par[i]]
        assert rho[i] == up * q[dep[i] - 1, tok[i]]


def test_budget_stop_is_first_drop_of_the_speedup_estimate():
    q = np.random.default_rng(9).dirichlet(0.4 * np.ones(8), size=8)
    n = 200
    full_par, full_tok, full_rho = oracle.best_first(q, n, 8)
    cost = 1.0 + 0.05 * np.arange(n + 1)   # C(N): a fixed part plus a per-node part
    par, tok, rho = oracle.best_first(q, n, 8, cost=cost)
    N = len(par)
    assert 1 <= N < n
    assert np.array_equal(par, full_par[:N]) and np.array_equal(tok, full_tok[:N])
    A = np.cumsum(full_rho)                   # A[k-1] = sum of the first k scores
    S = [A[k - 1] / cost[k] for k in range(1, n + 1)]
    assert all(S[k] >= S[k - 1] for k in range(1, N))   # growing up to N
    assert S[N] < S[N - 1]                                  # the next node would lower it
