"""GPU parity of tv_accept_stochastic against the oracle's stochastic walk:
lengths, paths and bonus tokens bit-exact.  Both sides decide in fp64 but may sum
a row in different orders; every case asserts first that no decision of the
oracle lies within 1e-9 (relative) of its threshold, so a difference can only be
a fault of the kernel."""
import dataclasses

import numpy as np
import pytest

import oracle
import workloads

pytestmark = pytest.mark.gpu
MARGIN = 1e-9


@pytest.fixture(scope="module", autouse=True)
def _lib():
    import torch
    if not torch.cuda.is_available():
        pytest.skip("no CUDA device")
    import tree_speculative_verify_tv_gb300 as tv
    tv.build()
    tv.load()


def run(batch, inp):
    import torch
    import tree_speculative_verify_tv_gb300 as tv
    d = tv.DeviceBatch(batch)
    cu = lambda x: torch.from_numpy(np.ascontiguousarray(x)).cuda()
    V = inp["root_p"].shape[1]
    T1 = max(batch.T, 1)
    node_p = cu(inp["node_p"] if batch.T else np.zeros((1, V), np.float32))
    node_q = cu(inp["node_q"] if batch.T else np.zeros((1, V), np.float32))
    ua = cu(inp["u_accept"] if batch.T else np.zeros(1))
    d.status.zero_()
    tv.tv_accept_stochastic(batch.B, batch.T, batch.max_nodes, batch.max_depth, V, d.node_offsets,
                            d.parent, cu(inp["draft"] if batch.T else np.zeros(1, np.int32)),
                            cu(inp["root_p"]), node_p, cu(inp["root_q"]), node_q, ua,
                            cu(inp["u_bonus"]), d.accept_len, d.path, d.bonus, d.status)
    torch.cuda.synchronize()
    return (int(d.status[0]), d.accept_len[:batch.B].cpu().numpy(), d.path[:batch.B].cpu().numpy(),
            d.bonus[:batch.B].cpu().numpy())


def check(batch, V, seed, **kw):
    inp = workloads.stochastic_inputs(batch, V, seed=seed, **kw)
    b2 = dataclasses.replace(batch, draft=inp["draft"])
    ln, path, bonus, margin = oracle.accept_stochastic(
        b2, inp["root_p"], inp["node_p"], inp["root_q"], inp["node_q"], inp["u_accept"],
        inp["u_bonus"], with_margin=True)
    assert margin > MARGIN, "choose another seed: a decision is too close to its threshold"
    st, gl, gp, gb = run(b2, inp)
    assert st == 0
    assert np.array_equal(gl, ln) and np.array_equal(gp, path) and np.array_equal(gb, bonus)
    return ln


@pytest.mark.parametrize("c,V,seed", [(1, 32, 2), (2, 32000, 2), (3, 64, 3), (4, 48, 4)])
def test_configs(c, V, seed):
    ln = check(workloads.make_config(c), V, seed)
    assert ln.max() >= 1  # something is accepted somewhere


@pytest.mark.parametrize("V,noise", [(7, 0.2), (100, 1.0), (1000, 3.0), (4096, 0.5)])
def test_ragged_trees_and_vocabularies(V, noise):
    rng = np.random.default_rng(V)
    b = workloads.random_batch(rng, [0, 3, 17, 1, 40, 9], 1, 16, 16, decay="scalar",
                               depth_cap=8, max_depth=8)
    check(b, V, seed=V + 1, draft_noise=noise)


@pytest.mark.parametrize("V,noise,seed", [(50, 3.0, 11), (32000, 4.0, 12)])
def test_wide_trees_many_rejections(V, noise, seed):
    # twelve children of the context and eight of node 0: up to twelve rejections in a
    # row at one node, each a new residual
    sizes = [20, 20, 20, 20]
    b = workloads.random_batch(np.random.default_rng(seed), sizes, 1, 16, 16, decay="scalar",
                               depth_cap=4, max_depth=4)
    par = np.concatenate([[-1] * 12 + [0] * 8] * len(sizes)).astype(np.int32)
    b = dataclasses.replace(b, parent=par, depth=np.where(par < 0, 1, 2).astype(np.int32))
    check(b, V, seed=seed + 100, draft_noise=noise)


def test_empty_trees():
    # no draft nodes at all: every bonus is a draw from the root's target row
    b = workloads.random_batch(np.random.default_rng(8), [0, 0, 0], 1, 16, 16, decay="scalar",
                               depth_cap=4, max_depth=4)
    ln = check(b, 300, seed=9)
    assert np.all(ln == 0)


def test_malformed_draft_token():
    import tree_speculative_verify_tv_gb300 as tv
    b = workloads.random_batch(np.random.default_rng(5), [4, 5], 1, 16, 16, decay="scalar",
                               depth_cap=4, max_depth=4)
    inp = workloads.stochastic_inputs(b, 16, seed=6)
    inp["draft"][b.node_offsets[1] + 1] = 16   # outside the vocabulary
    st, ln, path, bonus = run(dataclasses.replace(b, draft=inp["draft"]), inp)
    assert st == tv.TV_ERR_TREE
    assert ln[1] == 0 and bonus[1] == -1 and np.all(path[1] == -1)
