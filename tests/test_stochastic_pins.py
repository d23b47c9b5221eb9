"""Pins of the oracle's stochastic tree acceptance (LLM Primer VI ch. 9, §9.1: a
draft token x from q is accepted with probability min(1, p(x)/q(x)), otherwise the
emitted token comes from the normalized residual (p - q)_+): hand-worked cases, the
greedy limit for one-hot target rows, and the rule's defining property, that the
first emitted token follows the target distribution.  CPU only."""
import numpy as np
import pytest

import oracle
import workloads

P0 = np.array([0.5, 0.3, 0.2])
Q0 = np.array([0.2, 0.5, 0.3])


def run(parent, draft, p_nodes, q_nodes, u, ub, md=4):
    return oracle.accept_stochastic_request(np.array(parent), np.array(draft), P0, Q0,
                                            np.array(p_nodes), np.array(q_nodes),
                                            np.array(u, dtype=float), ub, md)


def test_hand_worked_reject_then_residual():
    # 0.7 * q(1) = 0.35 >= p(1) = 0.3: rejected; (p - q)_+ = [0.3, 0, 0] -> token 0
    L, path, bonus = run([-1], [1], [[0.1, 0.1, 0.8]], [[1 / 3] * 3], [0.7], 0.9)
    assert (L, bonus) == (0, 0) and path.tolist() == [-1, -1, -1, -1]


def test_hand_worked_accept_then_bonus_from_node():
    # 0.5 * 0.5 = 0.25 < 0.3: accepted; the node's p = [0.1, 0.1, 0.8], u = 0.15 -> 1
    L, path, bonus = run([-1], [1], [[0.1, 0.1, 0.8]], [[1 / 3] * 3], [0.5], 0.15)
    assert (L, bonus) == (1, 1) and path.tolist()[:1] == [0]


def test_hand_worked_two_siblings():
    # first sibling (token 1) rejected -> residual [1, 0, 0]; second (token 2) can
    # no longer be accepted (residual 0 there) -> residual of [1,0,0] - q = [0.8,0,0]
    L, path, bonus = run([-1, -1], [1, 2], [[1, 0, 0]] * 2, [[1, 0, 0]] * 2, [0.9, 0.0], 0.99)
    assert (L, bonus) == (0, 0)


def test_one_hot_target_is_greedy():
    rng = np.random.default_rng(3)
    b = workloads.random_batch(rng, [7, 12, 1, 0, 20], 1, 16, 16, decay="scalar", vocab=5,
                               depth_cap=6, max_depth=6)
    V = 5
    onehot = np.eye(V)
    root_p = onehot[b.root_argmax]
    node_p = onehot[b.target]
    q = rng.dirichlet(np.ones(V), size=b.B + b.T)
    ln, path, bonus = oracle.accept_stochastic(b, root_p, node_p, q[:b.B], q[b.B:],
                                               rng.random(b.T), rng.random(b.B))
    g_ln, g_path, g_bonus = oracle.accept_batch(b)
    assert np.array_equal(ln, g_ln) and np.array_equal(path, g_path)
    assert np.array_equal(bonus, g_bonus)


def test_first_token_follows_target_distribution():
    """Two siblings drafted independently from q at the context: the first emitted
    token (the accepted sibling's, else the residual draw) is distributed as p."""
    rng = np.random.default_rng(11)
    V = 4
    p = np.array([0.45, 0.25, 0.2, 0.1])
    q = np.array([0.1, 0.4, 0.3, 0.2])
    trials = 60000
    counts = np.zeros(V)
    leaf = np.full((2, V), 1.0 / V)
    for _ in range(trials):
        x = rng.choice(V, size=2, p=q)
        L, path, bonus = oracle.accept_stochastic_request(
            np.array([-1, -1]), x, p, q, leaf, leaf, rng.random(2), rng.random(), 2)
        counts[x[path[0]] if L else bonus] += 1
    freq = counts / trials
    sigma = np.sqrt(p * (1 - p) / trials)
    assert np.all(np.abs(freq - p) < 5 * sigma), (freq, p)
