"""GPU parity of tv_commit_verify: the previous step's accepted paths applied to the
state in place, then the current tree verified against the updated state.

Reference: the oracle's greedy walk and commit on the previous batch, then the
oracle's verification of the current batch with the committed state as H0.
States and outputs within 2e-3 normwise relative error; against the separate
tv_commit + tv_verify calls the fused kernel is bit-identical (same operations
in the same order).
"""
import dataclasses

import numpy as np
import pytest

import workloads
from gpu_util import TOL, check_verify, mat_rel_err

pytestmark = pytest.mark.gpu


@pytest.fixture(scope="module", autouse=True)
def _lib():
    import torch
    if not torch.cuda.is_available():
        pytest.skip("no CUDA device")
    import tree_speculative_verify_tv_gb300 as tv
    tv.build()
    tv.load()


def _oracle_two_steps(prev, cur, units=None):
    """Committed state after prev's greedy paths, and cur verified against it."""
    import oracle
    ln, path, _ = oracle.accept_batch(prev)
    Hc = oracle.commit(prev, ln, path, units=units, threads=8)
    H = prev.H0.astype(np.float64).copy()
    for u, m in Hc.items():
        b, h = divmod(u, prev.H)
        H[b, h] = m
    return H, dataclasses.replace(cur, H0=H), ln, path


def _device_two_steps(prev, cur, pending=True):
    import torch
    import tree_speculative_verify_tv_gb300 as tv
    dp, dc = tv.DeviceBatch(prev), tv.DeviceBatch(cur)
    dc.H0.copy_(dp.H0)
    dc.status.zero_()
    dp.status.zero_()
    dp.accept()
    dc.out.fill_(float("nan"))
    dc.commit_verify(dp if pending else None)
    torch.cuda.synchronize()
    return dp, dc


def _check(prev, cur, units=None):
    H_ref, cur_ref, ln, path = _oracle_two_steps(prev, cur, units)
    dp, dc = _device_two_steps(prev, cur)
    assert int(dp.status[0]) == 0 and int(dc.status[0]) == 0, int(dc.status[0])
    assert np.array_equal(dp.accept_len[:prev.B].cpu().numpy(), ln)
    assert np.array_equal(dp.path[:prev.B].cpu().numpy(), path)
    Hd = dc.H0.cpu().numpy().astype(np.float64)
    us = range(prev.B * prev.H) if units is None else units
    worst = max((mat_rel_err(Hd[u // prev.H, u % prev.H], H_ref[u // prev.H, u % prev.H])
                 for u in us), default=0.0)
    assert worst <= TOL, "state rel err %.3e" % worst
    out = dc.out[:cur.T].cpu().numpy().astype(np.float64)
    check_verify(cur_ref, out, units=units)
    return dp, dc


def _pair(make, **kw):
    return make(seed=11, **kw), make(seed=12, **kw)


def test_commit_verify_scalar_dv64_full_size():
    """Mamba-2-like layer (B=16, H=24, dk=128, dv=64, 16-node trees): the fused kernel."""
    _check(*_pair(workloads.config2))


def test_commit_verify_scalar_dv128_full_size():
    """Mixed-budget batch (B=128, H=32, dk=dv=128, up to 128 nodes), sampled units."""
    prev, cur = _pair(workloads.config4)
    rng = np.random.default_rng(0)
    units = np.sort(rng.choice(prev.B * prev.H, 256, replace=False))
    _check(prev, cur, units=units)


@pytest.mark.parametrize("dk,dv", [(64, 64), (64, 128), (128, 64), (128, 128)])
def test_commit_verify_ragged_with_empty_requests(dk, dv):
    """Requests with no current nodes still get their pending commit; requests whose
    previous walk accepted nothing keep their state bit for bit."""
    rng = np.random.default_rng(dk + dv)
    prev = workloads.random_batch(rng, [7, 0, 33, 5, 16], 3, dk, dv, decay="scalar",
                                  max_depth=8, depth_cap=8)
    cur = workloads.random_batch(rng, [0, 9, 21, 0, 40], 3, dk, dv, decay="scalar",
                                 max_depth=8, depth_cap=8)
    dp, dc = _check(prev, cur)
    ln = dp.accept_len[:prev.B].cpu().numpy()
    Hd = dc.H0.cpu().numpy()
    for b in np.where(ln == 0)[0]:
        assert np.array_equal(Hd[b], prev.H0[b])


@pytest.mark.parametrize("c", [1, 3])
def test_commit_verify_other_shapes_run_the_two_kernels(c):
    """Per-channel decay (GLA-like layer) and fp32 single-head trees: commit, then verify."""
    _check(*_pair(lambda seed: workloads.make_config(c, seed)))


def test_commit_verify_without_pending_is_verify():
    import torch
    prev, cur = _pair(workloads.config2)
    dp, dc = _device_two_steps(prev, cur, pending=False)
    assert int(dc.status[0]) == 0
    assert torch.equal(dc.H0, dp.H0)
    check_verify(dataclasses.replace(cur, H0=prev.H0), dc.out[:cur.T].cpu().numpy())


@pytest.mark.parametrize("c", [2, 4])
def test_commit_verify_equals_separate_calls(c):
    import torch
    import tree_speculative_verify_tv_gb300 as tv
    prev, cur = workloads.make_config(c, 21), workloads.make_config(c, 22)
    dp, dc = _device_two_steps(prev, cur)
    assert int(dc.status[0]) == 0
    # the same step as two calls: tv_commit in place, then tv_verify
    d2 = tv.DeviceBatch(cur)
    d2.H0.copy_(torch.from_numpy(prev.H0).cuda())
    d2.status.zero_()
    tv.tv_commit(dp.problem(), d2.H0, dp.g, dp.k, dp.v, dp.path, dp.accept_len, d2.H0, d2.status)
    d2.verify()
    torch.cuda.synchronize()
    assert int(d2.status[0]) == 0
    assert torch.equal(dc.H0, d2.H0)
    assert torch.equal(dc.out[:cur.T], d2.out[:cur.T])


def test_commit_verify_pipeline_three_steps():
    """Steady state: each step applies the previous step's paths, verifies, accepts."""
    import torch
    import oracle
    import tree_speculative_verify_tv_gb300 as tv
    steps = [workloads.config2(seed=30 + s, B=4, H=6) for s in range(3)]
    devs = [tv.DeviceBatch(b) for b in steps]
    state = devs[0].H0
    status = torch.zeros(4, dtype=torch.int32, device="cuda")
    outs = []
    for s, d in enumerate(devs):
        d.status = status
        tv.tv_commit_verify(d.problem(), devs[s - 1].pending() if s else None, state, d.q, d.k,
                            d.v, d.g, d.out, status)
        d.accept()
        torch.cuda.synchronize()
        outs.append(d.out[:steps[s].T].cpu().numpy().astype(np.float64))
    assert int(status[0]) == 0
    H = steps[0].H0.astype(np.float64)
    for s, b in enumerate(steps):
        cur = dataclasses.replace(b, H0=H)
        check_verify(cur, outs[s])
        ln, path, _ = oracle.accept_batch(b)
        assert np.array_equal(devs[s].accept_len[:b.B].cpu().numpy(), ln)
        Hc = oracle.commit(cur, ln, path)
        H = H.copy()
        for u, m in Hc.items():
            H[u // b.H, u % b.H] = m
    # the state after the last step's commit is still pending: apply it alone
    last = devs[-1]
    tv.tv_commit(last.problem(), state, last.g, last.k, last.v, last.path, last.accept_len,
                 state, status)
    torch.cuda.synchronize()
    Hd = state.cpu().numpy().astype(np.float64)
    assert mat_rel_err(Hd, H) <= TOL


@pytest.mark.parametrize("defect", ["not_root_path", "entry_out_of_range", "too_long"])
def test_commit_verify_malformed_pending_path(defect):
    """A bad pending path: TV_ERR_TREE, the request's state untouched and its outputs
    computed from the untouched state; the other requests are committed."""
    import torch
    import oracle
    import tree_speculative_verify_tv_gb300 as tv
    prev, cur = workloads.config2(seed=41, B=3, H=2), workloads.config2(seed=42, B=3, H=2)
    dp, dc = tv.DeviceBatch(prev), tv.DeviceBatch(cur)
    dc.H0.copy_(dp.H0)
    dp.accept()
    torch.cuda.synchronize()
    ln = dp.accept_len[:prev.B].cpu().numpy().copy()
    path = dp.path[:prev.B].cpu().numpy().copy()
    md = prev.max_depth
    if defect == "not_root_path":
        ln[1], path[1] = 2, [0, 5] + [-1] * (md - 2)       # node 5 is not a child of node 0
    elif defect == "entry_out_of_range":
        ln[1], path[1] = 1, [16] + [-1] * (md - 1)         # a request of 16 nodes
    else:
        ln[1] = md + 1
    dp.accept_len[:prev.B].copy_(torch.from_numpy(ln))
    dp.path[:prev.B].copy_(torch.from_numpy(path))
    dc.status.zero_()
    dc.commit_verify(dp)
    torch.cuda.synchronize()
    assert int(dc.status[0]) == tv.TV_ERR_TREE
    good = np.array([0, 2])
    units = [u for u in range(prev.B * prev.H) if u // prev.H in good]
    ln_good = ln.copy()
    ln_good[1] = 0
    Hc = oracle.commit(prev, ln_good, path, units=units)
    H = prev.H0.astype(np.float64).copy()
    for u, m in Hc.items():
        H[u // prev.H, u % prev.H] = m
    Hd = dc.H0.cpu().numpy()
    assert np.array_equal(Hd[1], prev.H0[1])
    for u in units:
        assert mat_rel_err(Hd[u // prev.H, u % prev.H].astype(np.float64),
                           H[u // prev.H, u % prev.H]) <= TOL
    check_verify(dataclasses.replace(cur, H0=H), dc.out[:cur.T].cpu().numpy().astype(np.float64))


def _acv_and_separate(prev, cur):
    """tv_accept_commit_verify, and the same step as tv_accept_greedy then
    tv_commit_verify, on copies of the same inputs: (batch holding the walk's results,
    current batch) for each."""
    import torch
    import tree_speculative_verify_tv_gb300 as tv
    runs = []
    for fused in (True, False):
        dp, dc = tv.DeviceBatch(prev), tv.DeviceBatch(cur)
        dc.H0.copy_(dp.H0)
        dc.status.zero_()
        dp.status.zero_()
        for d in (dp, dc):
            d.accept_len.fill_(-7)
            d.path.fill_(-7)
            d.bonus.fill_(-7)
        dc.out.fill_(float("nan"))
        if fused:
            dc.accept_commit_verify(dp)  # the walk's results land in dc's result buffers
            acc = dc
        else:
            dp.accept()
            dc.commit_verify(dp)
            acc = dp
        torch.cuda.synchronize()
        runs.append((acc, dc))
    return runs


@pytest.mark.parametrize("c", [2, 4])
def test_accept_commit_verify_equals_accept_then_commit_verify(c):
    """Config 2 takes the one-kernel path (the walk runs in every block), config 4 the
    walk kernel and then tv_commit_verify: both bit-identical to the two calls."""
    import torch
    prev, cur = workloads.make_config(c, 51), workloads.make_config(c, 52)
    (fp, fc), (sp, sc) = _acv_and_separate(prev, cur)
    assert int(fc.status[0]) == 0 and int(sc.status[0]) == 0 and int(sp.status[0]) == 0
    B = prev.B
    assert torch.equal(fp.accept_len[:B], sp.accept_len[:B])
    assert torch.equal(fp.path[:B], sp.path[:B])
    assert torch.equal(fp.bonus[:B], sp.bonus[:B])
    assert torch.equal(fc.H0, sc.H0)
    assert torch.equal(fc.out[:cur.T], sc.out[:cur.T])


def test_accept_commit_verify_ragged_trees():
    """Trees of different sizes, so that a request's previous tree does not start at
    b * max_nodes (its arrays are requested again at the actual range): the one-launch
    step still equals tv_accept_greedy then tv_commit_verify bit for bit."""
    import torch
    rng = np.random.default_rng(91)
    kw = dict(decay="scalar", qkv_dtype="bf16", depth_cap=8, vocab=3, max_depth=8)
    prev = workloads.random_batch(rng, [5, 16, 9, 32, 1, 12, 20, 3], 4, 128, 64, **kw)
    cur = workloads.random_batch(rng, [7, 32, 2, 11, 16, 4, 30, 9], 4, 128, 64, **kw)
    (fp, fc), (sp, sc) = _acv_and_separate(prev, cur)
    assert int(fc.status[0]) == 0 and int(sc.status[0]) == 0 and int(sp.status[0]) == 0
    B = prev.B
    assert int(sp.accept_len[:B].max()) > 0
    assert torch.equal(fp.accept_len[:B], sp.accept_len[:B])
    assert torch.equal(fp.path[:B], sp.path[:B])
    assert torch.equal(fp.bonus[:B], sp.bonus[:B])
    assert torch.equal(fc.H0, sc.H0)
    assert torch.equal(fc.out[:cur.T], sc.out[:cur.T])


def test_accept_commit_verify_against_the_oracle():
    prev, cur = _pair(workloads.config2)
    H_ref, cur_ref, ln, path = _oracle_two_steps(prev, cur)
    (fp, fc), _ = _acv_and_separate(prev, cur)
    assert int(fc.status[0]) == 0
    assert np.array_equal(fp.accept_len[:prev.B].cpu().numpy(), ln)
    assert np.array_equal(fp.path[:prev.B].cpu().numpy(), path)
    Hd = fc.H0.cpu().numpy().astype(np.float64)
    worst = max(mat_rel_err(Hd[b, h], H_ref[b, h]) for b in range(prev.B) for h in range(prev.H))
    assert worst <= TOL, "state rel err %.3e" % worst
    check_verify(cur_ref, fc.out[:cur.T].cpu().numpy().astype(np.float64))


def test_accept_commit_verify_malformed_previous_tree():
    """A previous tree with a parent after its child: TV_ERR_TREE, that request gets
    accept_len 0, path -1, bonus -1 and no commit; the other requests are exact."""
    import torch
    import tree_speculative_verify_tv_gb300 as tv
    prev, cur = workloads.config2(seed=61, B=3, H=2), workloads.config2(seed=62, B=3, H=2)
    s = int(prev.node_offsets[1])
    prev.parent[s + 2] = 7
    dp, dc = tv.DeviceBatch(prev), tv.DeviceBatch(cur)
    dc.H0.copy_(dp.H0)
    dc.status.zero_()
    dc.accept_commit_verify(dp)
    torch.cuda.synchronize()
    assert int(dc.status[0]) == tv.TV_ERR_TREE
    assert int(dc.accept_len[1]) == 0 and int(dc.bonus[1]) == -1
    assert torch.all(dc.path[1] == -1)
    assert torch.equal(dc.H0[1], dp.H0[1])
    # the other requests: as the separate calls on an intact copy of their trees
    good = workloads.config2(seed=61, B=3, H=2)
    H_ref, cur_ref, ln, path = _oracle_two_steps(good, cur, units=[0, 1, 4, 5])
    for b in (0, 2):
        assert int(dc.accept_len[b]) == ln[b]
        for h in range(prev.H):
            assert mat_rel_err(dc.H0[b, h].cpu().numpy().astype(np.float64), H_ref[b, h]) <= TOL


@pytest.mark.parametrize("call", ["commit_verify", "accept_commit_verify"])
def test_write_back_of_a_state_only_16_byte_aligned(call):
    """The committed rows go back with 256-bit stores where the state is 32-byte
    aligned and with 128-bit stores where it is only 16-byte aligned: both give the
    same bits."""
    import torch
    import tree_speculative_verify_tv_gb300 as tv
    prev, cur = workloads.make_config(2, 61), workloads.make_config(2, 62)
    res = []
    for shift in (0, 4):
        dp, dc = tv.DeviceBatch(prev), tv.DeviceBatch(cur)
        buf = torch.empty(dc.H0.numel() + 8, dtype=torch.float32, device="cuda")
        H = buf[shift:shift + dc.H0.numel()].view_as(dc.H0)
        assert (H.data_ptr() % 32 == 0) == (shift == 0) and H.data_ptr() % 16 == 0
        H.copy_(dp.H0)
        dc.H0 = H
        dc.status.zero_()
        dp.status.zero_()
        if call == "commit_verify":
            dp.accept()
            dc.commit_verify(dp)
            ln = dp.accept_len
        else:
            dc.accept_commit_verify(dp)
            ln = dc.accept_len
        torch.cuda.synchronize()
        assert int(dc.status[0]) == 0
        assert int(ln[:prev.B].max()) > 0  # some rows are written back
        res.append((dc.H0.clone(), dc.out[:cur.T].clone()))
    assert torch.equal(res[0][0], res[1][0])
    assert torch.equal(res[0][1], res[1][1])
