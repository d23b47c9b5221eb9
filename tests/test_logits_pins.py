"""Pins of the oracle's target argmax (the greedy rule's "target's own choice",
LLM Primer VI ch. 9, §9.1) against hand-worked rows and a brute-force scan, and
of the logits generator against the planted acceptance paths.  CPU only."""
import math

import numpy as np
import pytest

import oracle
import workloads


def bits(vals):
    return workloads.f32_to_bf16_bits(np.array([vals], dtype=np.float32))


NAN, INF = float("nan"), float("inf")
HAND = [  # (row, index of the largest value; first one among equals)
    ([1.0, 3.0, 3.0, 2.0], 1),
    ([-1.0, -0.5, -2.0], 1),
    ([-INF, -INF], 0),
    ([-0.0, 0.0], 0),            # -0 equals +0: first index
    ([0.0, -0.0, 0.0], 0),
    ([-0.0, -1.0], 0),
    ([1.0, NAN, 5.0, NAN], 1),   # a NaN counts as the largest; first NaN
    ([INF, 3.0e38], 0),
    ([7.0], 0),
    ([-5.0, -5.0, -4.0, -4.0], 2),
]


@pytest.mark.parametrize("row,want", HAND)
def test_argmax_hand_rows(row, want):
    assert int(oracle.argmax_rows(bits(row))[0]) == want


def test_argmax_subnormal_and_zero():
    b = np.array([[0x0001, 0x0000, 0x8001]], dtype=np.uint16)  # +min subnormal, +0, -min
    assert int(oracle.argmax_rows(b)[0]) == 0


def _scan(row):
    """Plain scan: keep the first maximum; a NaN beats every number, first NaN wins."""
    best = 0
    for i in range(1, len(row)):
        a, b = row[i], row[best]
        if math.isnan(b):
            continue
        if math.isnan(a) or a > b:
            best = i
    return best


def test_argmax_brute_force_with_ties_and_nans():
    rng = np.random.default_rng(5)
    for _ in range(300):
        V = int(rng.integers(1, 12))
        vals = rng.integers(-2, 3, V).astype(np.float32)
        vals[rng.random(V) < 0.1] = np.nan
        vals[rng.random(V) < 0.1] = -0.0
        row_bits = workloads.f32_to_bf16_bits(vals[None, :])
        widened = workloads.bf16_bits_to_f32(row_bits[0]).astype(np.float64)
        assert int(oracle.argmax_rows(row_bits)[0]) == _scan(list(widened))


def test_generator_plants_the_targets():
    b = workloads.config2(seed=3)
    root, node = workloads.target_logits(b, 32000, seed=1)
    assert root.shape == (b.B, 32000) and node.shape == (b.T, 32000)
    assert np.array_equal(oracle.argmax_rows(root), b.root_argmax)
    assert np.array_equal(oracle.argmax_rows(node), b.target)


def test_accept_from_logits_reproduces_planted_paths():
    b = workloads.config2(seed=4)
    root, node = workloads.target_logits(b, 32000, seed=2)
    ln, path, bonus, ra, ta = oracle.accept_from_logits(b, root, node)
    l2, p2, b2 = oracle.accept_batch(b)
    assert np.array_equal(ln, l2) and np.array_equal(path, p2) and np.array_equal(bonus, b2)


def test_tied_levels_generator_has_ties():
    b = workloads.config1(seed=2)
    root, node = workloads.target_logits(b, 64, seed=3, levels=3)
    x = workloads.bf16_bits_to_f32(node).astype(np.float64)
    ties = sum(int(np.sum(r == r.max()) > 1) for r in x)
    assert ties == len(x)  # 64 draws from 3 levels: every row ties at its maximum
