"""GPU parity of tv_accept_greedy_logits: target argmax of every logits row and
the greedy walk over it, against the oracle's numpy argmax and walk.  Integer
results, compared bit for bit (argmax, length, path, bonus)."""
import numpy as np
import pytest

import workloads

pytestmark = pytest.mark.gpu


@pytest.fixture(scope="module", autouse=True)
def _lib():
    import torch
    if not torch.cuda.is_available():
        pytest.skip("no CUDA device")
    import tree_speculative_verify_tv_gb300 as tv
    tv.build()
    tv.load()


def _dev(x):
    import torch
    return torch.from_numpy(np.ascontiguousarray(x).view(np.int16)).cuda()


def run(batch, root_logits, node_logits, want_argmax=True):
    import torch
    import tree_speculative_verify_tv_gb300 as tv
    d = tv.DeviceBatch(batch)
    V = root_logits.shape[1]
    rl = _dev(root_logits)
    nl = _dev(node_logits if batch.T else np.zeros((1, V), np.uint16))
    ra = torch.full((max(batch.B, 1),), -7, dtype=torch.int32, device="cuda")
    ta = torch.full((max(batch.T, 1),), -7, dtype=torch.int32, device="cuda")
    d.status.zero_()
    d.accept_len.fill_(-9)
    tv.tv_accept_greedy_logits(batch.B, batch.T, batch.max_nodes, batch.max_depth, V,
                               d.node_offsets, d.parent, d.draft, rl, nl,
                               ra if want_argmax else None, ta if want_argmax else None,
                               d.accept_len, d.path, d.bonus, d.status)
    torch.cuda.synchronize()
    return {"status": int(d.status[0]), "len": d.accept_len[:batch.B].cpu().numpy(),
            "path": d.path[:batch.B].cpu().numpy(), "bonus": d.bonus[:batch.B].cpu().numpy(),
            "root": ra[:batch.B].cpu().numpy(), "target": ta[:batch.T].cpu().numpy()}


def check(batch, root_logits, node_logits):
    import oracle
    res = run(batch, root_logits, node_logits)
    ln, path, bonus, ra, ta = oracle.accept_from_logits(batch, root_logits, node_logits)
    assert res["status"] == 0
    assert np.array_equal(res["root"], ra)
    assert np.array_equal(res["target"], ta)
    assert np.array_equal(res["len"], ln)
    assert np.array_equal(res["path"], path)
    assert np.array_equal(res["bonus"], bonus)
    return res


@pytest.mark.parametrize("c,V", [(1, 32), (2, 32000), (3, 64), (4, 32)])
def test_planted_targets(c, V):
    b = workloads.make_config(c)
    root, node = workloads.target_logits(b, V, seed=c)
    res = check(b, root, node)
    assert np.array_equal(res["target"], b.target)  # the planted paths are reproduced


@pytest.mark.parametrize("V", [8, 37, 1000, 32000])
def test_ties_first_index(V):
    """Values from three levels: every row ties; the first index of the maximum wins."""
    b = workloads.random_batch(np.random.default_rng(V), [5, 0, 17, 40], 1, 16, 16,
                               decay="scalar", vocab=min(V, 3), depth_cap=8, max_depth=8)
    root, node = workloads.target_logits(b, V, seed=V, levels=3)
    check(b, root, node)


def test_nan_zero_and_inf_rows():
    b = workloads.random_batch(np.random.default_rng(2), [9, 12], 1, 16, 16, decay="scalar",
                               vocab=4, depth_cap=6, max_depth=6)
    V = 64
    root, node = workloads.target_logits(b, V, seed=5, levels=2)
    rng = np.random.default_rng(7)
    allrows = np.concatenate([root, node])
    for r in range(len(allrows)):
        kind = r % 4
        if kind == 0:
            allrows[r, rng.integers(0, V, 2)] = 0x7FC0          # NaN
        elif kind == 1:
            allrows[r] = 0x8000                                   # all -0
            allrows[r, rng.integers(0, V)] = 0x0000               # one +0: equal, first wins
        elif kind == 2:
            allrows[r] = 0xFF80                                   # all -inf
        else:
            allrows[r, rng.integers(0, V)] = 0x7F80               # +inf
    check(b, allrows[:b.B], allrows[b.B:])


def test_argmax_outputs_are_required():
    import tree_speculative_verify_tv_gb300 as tv
    b = workloads.config2(seed=9)
    root, node = workloads.target_logits(b, 32000, seed=9)
    with pytest.raises(tv.TVError):
        run(b, root, node, want_argmax=False)


def test_malformed_tree():
    b = workloads.random_batch(np.random.default_rng(3), [6, 7, 5], 1, 16, 16, decay="scalar",
                               vocab=4, depth_cap=6, max_depth=6)
    b.parent[b.node_offsets[1] + 2] = 5                          # a parent after its child
    root, node = workloads.target_logits(b, 32, seed=3, levels=4)
    res = run(b, root, node)
    import tree_speculative_verify_tv_gb300 as tv
    assert res["status"] == tv.TV_ERR_TREE
    assert res["len"][1] == 0 and res["bonus"][1] == -1 and np.all(res["path"][1] == -1)
    import oracle
    for bb in (0, 2):
        s, e = b.node_offsets[bb], b.node_offsets[bb + 1]
        ra = oracle.argmax_rows(root[bb:bb + 1])[0]
        ta = oracle.argmax_rows(node[s:e])
        L, p, bo = oracle.accept(b.parent[s:e], b.draft[s:e], ta, ra, b.max_depth)
        assert res["len"][bb] == L and res["bonus"][bb] == bo
        assert np.array_equal(res["path"][bb], p)
