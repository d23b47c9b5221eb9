"""GPU parity of tv_build_tree, best-first draft-tree construction: parents,
tokens and counts bit-exact against the oracle, path scores equal as fp64 values
(both sides form the same products)."""
import numpy as np
import pytest

import oracle

pytestmark = pytest.mark.gpu


@pytest.fixture(scope="module", autouse=True)
def _lib():
    import torch
    if not torch.cuda.is_available():
        pytest.skip("no CUDA device")
    import tree_speculative_verify_tv_gb300 as tv
    tv.build()
    tv.load()


def build(marg, n, cost=None):
    import torch
    import tree_speculative_verify_tv_gb300 as tv
    B, cap, C = marg.shape
    m = torch.from_numpy(np.ascontiguousarray(marg, dtype=np.float64)).cuda()
    c = torch.from_numpy(np.asarray(cost, dtype=np.float64)).cuda() if cost is not None else None
    par = torch.full((max(B, 1), n), -9, dtype=torch.int32, device="cuda")
    tok = torch.full((max(B, 1), n), -9, dtype=torch.int32, device="cuda")
    rho = torch.full((max(B, 1), n), -9.0, dtype=torch.float64, device="cuda")
    cnt = torch.full((max(B, 1),), -9, dtype=torch.int32, device="cuda")
    tv.tv_build_tree(B, C, cap, n, m, c, par, tok, rho, cnt)
    torch.cuda.synchronize()
    return par.cpu().numpy(), tok.cpu().numpy(), rho.cpu().numpy(), cnt.cpu().numpy()


def check(marg, n, cost=None):
    par, tok, rho, cnt = build(marg, n, cost)
    for b in range(marg.shape[0]):
        p, t, r = oracle.best_first(marg[b], n, marg.shape[1], cost=cost)
        N = len(p)
        assert cnt[b] == N
        assert np.array_equal(par[b, :N], p) and np.array_equal(tok[b, :N], t)
        assert np.array_equal(rho[b, :N], r)
        assert np.all(par[b, N:] == -1) and np.all(tok[b, N:] == -1) and np.all(rho[b, N:] == 0.0)


@pytest.mark.parametrize("B,C,cap,n,alpha", [
    (32, 8, 8, 64, 0.3),     # GLA-like layer's trees (64 nodes, depth <= 8, Dirichlet(0.3))
    (8, 8, 16, 256, 0.2),    # large-tree stack's trees (256 nodes, depth <= 16, Dirichlet(0.2))
    (5, 32, 4, 200, 0.5),
    (3, 1, 6, 10, 1.0),      # one candidate: a chain that stops at the depth cap
    (7, 3, 32, 256, 2.0),
    (40, 5, 2, 256, 1.0),    # frontier exhausted before the budget
])
def test_matches_oracle(B, C, cap, n, alpha):
    marg = np.random.default_rng(B * 100 + C).dirichlet(alpha * np.ones(C), size=(B, cap))
    check(marg, n)


def test_equal_scores_follow_frontier_order():
    marg = np.full((4, 5, 4), 0.25)          # every candidate equally likely
    marg[1] = np.full((5, 4), 0.5) * [[1, 1, 0, 0]]   # two tied candidates, two zeros
    check(marg, 60)


@pytest.mark.parametrize("slope", [0.01, 0.05, 0.3])
def test_budget_stop(slope):
    marg = np.random.default_rng(5).dirichlet(0.4 * np.ones(8), size=(6, 8))
    n = 128
    cost = 1.0 + slope * np.arange(n + 1)
    check(marg, n, cost=cost)
