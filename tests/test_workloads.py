"""Seeded input generators: shapes, tree validity and the BASTION self-check (CPU)."""
import numpy as np
import pytest

import oracle
import workloads


def _check_batch(b):
    assert b.node_offsets[0] == 0 and np.all(np.diff(b.node_offsets) >= 0)
    T = b.T
    assert b.parent.shape == (T,) and b.depth.shape == (T,)
    for bb in range(b.B):
        s, e = b.node_offsets[bb], b.node_offsets[bb + 1]
        par = b.parent[s:e]
        assert all(-1 <= par[i] < i for i in range(e - s))
        assert np.array_equal(b.depth[s:e], workloads.depths_from_parents(par))
        assert e - s <= b.max_nodes
    assert (b.depth.max() if T else 0) <= b.max_depth
    assert b.q.shape == (T, b.H, b.dk) and b.v.shape == (T, b.H, b.dv)
    assert b.H0.shape == (b.B, b.H, b.dk, b.dv)
    assert b.g.shape == ((T, b.H) if b.decay == "scalar" else (T, b.H, b.dk))
    assert np.all(b.g <= 0)


@pytest.mark.parametrize("c", [1, 2, 3, 4])
def test_config_shapes(c):
    b = workloads.make_config(c)
    _check_batch(b)
    expect = {1: (1, 1, 16, 16), 2: (16, 24, 128, 64), 3: (32, 16, 128, 128), 4: (128, 32, 128, 128)}
    assert (b.B, b.H, b.dk, b.dv) == expect[c]


def test_config5_small_replica_shapes():
    b = workloads.config5(B=2, layers=2, heads=2)
    _check_batch(b)
    assert b.sizes().tolist() == [256, 256] and b.max_depth == 16 and b.decay == "diag"


def test_config2_tree_and_planted_acceptance():
    b = workloads.config2()
    par = b.parent[:16]
    assert par.tolist() == [-1] * 4 + list(range(12))
    ln, path, bonus = oracle.accept_batch(b)
    assert set(ln.tolist()) <= set(range(5)) and len(set(ln.tolist())) > 1
    for bb in range(b.B):
        d = b.draft[b.node_offsets[bb]:b.node_offsets[bb] + 4]
        assert len(set(d.tolist())) == 4


def test_config5_planted_paths_reach_their_nodes():
    b = workloads.config5(B=4, layers=1, heads=1, seed=7)
    ln, path, bonus = oracle.accept_batch(b)
    assert np.all(ln >= 1) and np.all(ln <= 16)


def test_bf16_roundtrip():
    x = np.array([1.0, -2.5, 3.14159, 1e-3, 65504.0, 0.0], np.float32)
    bits = workloads.f32_to_bf16_bits(x)
    y = workloads.bf16_bits_to_f32(bits)
    assert np.all(np.abs(y - x) <= np.abs(x) * 2.0 ** -8)
    assert np.array_equal(workloads.f32_to_bf16_bits(y), bits)


def test_best_first_is_rho_ordered():
    rng = np.random.default_rng(0)
    marg = rng.dirichlet(0.3 * np.ones(8), size=8)
    par, tok, rho = workloads.tree_best_first(marg, 64, 8)
    # insertion order is non-increasing in rho; children never beat their parent
    assert np.all(np.diff(rho) <= 1e-15)
    for i, p in enumerate(par):
        if p >= 0:
            assert rho[i] <= rho[p] + 1e-15
    # the path score is the product of the marginals along the root path
    dep = workloads.depths_from_parents(par)
    for i in range(len(par)):
        j, prod = i, 1.0
        while j >= 0:
            prod *= marg[dep[j] - 1, tok[j]]
            j = par[j]
        assert abs(prod - rho[i]) <= 1e-12


def test_mean_acceptance_matches_bastion_surrogate():
    """Under the planted-continuation generator, E[accept len] = sum_i rho(i)
    (BASTION summary, Method §2 acceptance surrogate); a self-check of the inputs."""
    lens, rhos = [], []
    for seed in range(6):
        b = workloads.config3(seed=seed, H=1)
        ln, _, _ = oracle.accept_batch(b)
        lens.extend(ln.tolist())
        rhos.extend(b.rho_sums)
    lens, rhos = np.array(lens, float), np.array(rhos)
    se = lens.std() / np.sqrt(len(lens))
    assert abs(lens.mean() - rhos.mean()) < 4 * se + 0.05, (lens.mean(), rhos.mean())
