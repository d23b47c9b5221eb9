"""GPU parity of the fused tensor-core verify kernel (TV_VARIANT_TC_FUSED): the
context term, the pair scores and the tree term of a (request, head) unit all on
tcgen05, one unit per CTA, for scalar-decay trees of up to 32 nodes.  Cases: the
configuration shapes, ragged trees of 0-32 nodes at every dk/dv, deep chains and
wide stars, strong and zero decay, non-finite rows next to a request, malformed
trees between valid ones, canaries around the outputs, compared with the fp64
oracle (2e-3 normwise per row).  Also: the pending commit of tv_commit_verify on
this kernel, and the timeout path (a wait made to expire through
TV_VARIANT_TEST_EXPIRE_WAIT).
"""
import dataclasses

import numpy as np
import pytest

import workloads
from gpu_util import TOL, check_verify, mat_rel_err, row_rel_err, run_library

pytestmark = pytest.mark.gpu

FUSED = 3


@pytest.fixture(scope="module", autouse=True)
def _lib():
    import torch
    if not torch.cuda.is_available():
        pytest.skip("no CUDA device")
    import tree_speculative_verify_tv_gb300 as tv
    tv.build()
    tv.load()
    assert tv.TV_VARIANT_TC_FUSED == FUSED


def _verify(batch, variant=FUSED):
    res = run_library(batch, variant=variant, steps=("verify",))
    return res["status"], res["out"]


def test_fused_mamba2_layer():
    """Mamba-2-like layer, B=16, H=24, 16-node trees: 384 units, all checked."""
    b = workloads.config2(seed=5)
    st, out = _verify(b)
    assert st == 0
    check_verify(b, out)


def test_fused_is_auto_for_the_mamba2_layer():
    import tree_speculative_verify_tv_gb300 as tv
    b = workloads.config2(seed=5)
    d = tv.DeviceBatch(b)
    assert tv.tv_verify_variant(d.problem()) == FUSED


def test_fused_folded_layers_sampled_and_against_one_unit_kernel():
    """32 Mamba-2-like layers folded into the head axis (H = 768, 12288 units), the
    launch the folded measurement times: 128 sampled units against the oracle, every
    unit against the one-unit tensor-core kernel."""
    b = workloads.config2(seed=77, H=24 * 32)
    st, out = _verify(b)
    assert st == 0
    rng = np.random.default_rng(3)
    units = np.sort(rng.choice(b.B * b.H, 128, replace=False))
    check_verify(b, out, units=units)
    st2, out2 = _verify(b, variant=2)
    assert st2 == 0
    # two fp32 evaluations of the same products (each within ~1e-5 of exact)
    assert row_rel_err(out, out2) <= 2e-4


@pytest.mark.parametrize("dk,dv", [(64, 64), (64, 128), (128, 64), (128, 128)])
@pytest.mark.parametrize("cap", [16, 32])
def test_fused_ragged_with_empty_requests(dk, dv, cap):
    """Ragged trees of 0..cap nodes (node tiles of 16 and 32), many per CTA."""
    rng = np.random.default_rng(dk * 3 + dv + cap)
    sizes = rng.integers(0, cap + 1, 90)
    sizes[::7] = 0
    b = workloads.random_batch(rng, sizes, 5, dk, dv, decay="scalar", depth_cap=10,
                               max_depth=10, max_nodes=cap)
    st, out = _verify(b)
    assert st == 0
    check_verify(b, out)


def test_fused_deep_chains_and_wide_stars():
    """Chains of 32 nodes (depth 32, five rounds of pointer doubling) and stars of
    32 roots, interleaved."""
    rng = np.random.default_rng(9)
    b = workloads.random_batch(rng, [32] * 40, 16, 128, 64, decay="scalar", depth_cap=32,
                               max_depth=32)
    for r in range(b.B):
        s = int(b.node_offsets[r])
        par = np.arange(-1, 31, dtype=np.int32) if r % 2 == 0 else np.full(32, -1, np.int32)
        b.parent[s:s + 32] = par
        b.depth[s:s + 32] = workloads.depths_from_parents(par)
    st, out = _verify(b)
    assert st == 0
    check_verify(b, out)


def test_fused_strong_and_zero_decay():
    rng = np.random.default_rng(13)
    b = workloads.random_batch(rng, [16] * 24, 8, 128, 64, decay="scalar", depth_cap=8,
                               max_depth=8)
    g = b.g.reshape(b.T, b.H)
    g[: b.T // 2] = -60.0   # e^{G} underflows to 0 for deep nodes
    g[b.T // 2:] = 0.0
    st, out = _verify(b)
    assert st == 0
    check_verify(b, out)


def test_fused_neighbor_rows_do_not_leak():
    """q/k/v tiles are copied in boxes of 16 nodes, so a request's boxes run into the
    next request's rows: non-finite values there must not reach its outputs."""
    rng = np.random.default_rng(46)
    b = workloads.random_batch(rng, [5, 13, 17, 3, 9], 4, 128, 64, decay="scalar",
                               depth_cap=8, max_depth=8, max_nodes=32)
    s, e = int(b.node_offsets[2]), int(b.node_offsets[3])
    b.v[s:e] = 0x7F80  # bf16 +inf
    b.k[s:e] = 0x7FC0  # bf16 NaN
    b.q[s:e] = 0x7FC0
    st, out = _verify(b)
    assert st == 0
    check_verify(b, out, units=[u for u in range(b.B * b.H) if u // b.H != 2])


def test_fused_malformed_trees_and_offsets_between_valid_ones():
    """Malformed trees zero their rows and set TV_ERR_TREE; the other requests are
    unaffected."""
    rng = np.random.default_rng(12)
    sizes = [int(x) for x in rng.choice([0, 1, 9, 16, 25, 32], 200)]
    b = workloads.random_batch(rng, sizes, 6, 128, 64, decay="scalar", depth_cap=8,
                               max_depth=8, max_nodes=32)
    bad = [r for r in range(b.B) if sizes[r] >= 9][::6]
    for r in bad:
        s = int(b.node_offsets[r])
        b.parent[s + 3] = 5 if r % 2 else 3  # a parent after its child / itself
    st, out = _verify(b)
    assert st == 6  # TV_ERR_TREE
    for r in bad:
        s, e = int(b.node_offsets[r]), int(b.node_offsets[r + 1])
        assert np.all(out[s:e] == 0.0)
    check_verify(b, out, units=[u for u in range(b.B * b.H) if u // b.H not in bad])


def test_fused_depth_mismatch_and_too_deep():
    rng = np.random.default_rng(15)
    b = workloads.random_batch(rng, [12, 12, 12, 12], 3, 128, 64, decay="scalar", depth_cap=6,
                               max_depth=6)
    s1, s2 = int(b.node_offsets[1]), int(b.node_offsets[2])
    b.depth[s1 + 4] += 1
    chain = np.arange(-1, 11, dtype=np.int32)
    b.parent[s2:s2 + 12] = chain                    # depth 12 > max_depth 6
    b.depth[s2:s2 + 12] = workloads.depths_from_parents(chain)
    st, out = _verify(b)
    assert st == 6
    assert np.all(out[s1:int(b.node_offsets[3])] == 0.0)
    check_verify(b, out, units=[u for u in range(b.B * b.H) if u // b.H in (0, 3)])


def test_fused_outputs_stay_inside_their_buffers():
    """Canaries before and after out: the epilogue writes only the request's rows."""
    import torch
    import tree_speculative_verify_tv_gb300 as tv
    b = workloads.config2(seed=19, B=5, H=7)
    d = tv.DeviceBatch(b)
    pad = 4096
    big = torch.full((pad + d.out.numel() + pad,), 12345.0, device="cuda")
    out = big[pad:pad + d.out.numel()].view_as(d.out)
    d.status.zero_()
    tv.tv_verify(d.problem(), d.H0, d.q, d.k, d.v, d.g, out, d.status, variant=FUSED)
    torch.cuda.synchronize()
    assert int(d.status[0]) == 0
    assert torch.all(big[:pad] == 12345.0) and torch.all(big[pad + out.numel():] == 12345.0)
    check_verify(b, out[:b.T].cpu().numpy().astype(np.float64))


def _two_step(prev, cur, units=None):
    import torch
    import oracle
    import tree_speculative_verify_tv_gb300 as tv
    ln, path, _ = oracle.accept_batch(prev)
    Hc = oracle.commit(prev, ln, path, units=units, threads=8)
    H = prev.H0.astype(np.float64).copy()
    for u, m in Hc.items():
        b, h = divmod(u, prev.H)
        H[b, h] = m
    dp, dc = tv.DeviceBatch(prev), tv.DeviceBatch(cur)
    dc.H0.copy_(dp.H0)
    dp.status.zero_()
    dc.status.zero_()
    dp.accept()
    dc.out.fill_(float("nan"))
    dc.commit_verify(dp)
    torch.cuda.synchronize()
    assert int(dp.status[0]) == 0 and int(dc.status[0]) == 0
    Hd = dc.H0.cpu().numpy().astype(np.float64)
    us = range(prev.B * prev.H) if units is None else units
    worst = max(mat_rel_err(Hd[u // prev.H, u % prev.H], H[u // prev.H, u % prev.H]) for u in us)
    assert worst <= TOL, worst
    check_verify(dataclasses.replace(cur, H0=H), dc.out[:cur.T].cpu().numpy().astype(np.float64),
                 units=units)
    return dp, dc, ln


@pytest.mark.parametrize("dk,dv", [(64, 64), (128, 64), (128, 128)])
def test_fused_commit_verify_ragged_with_empty_requests(dk, dv):
    """Requests with no current nodes still get their pending commit; requests whose
    previous walk accepted nothing keep their state bit for bit."""
    rng = np.random.default_rng(dk + 7 * dv)
    sizes_p = [int(x) for x in rng.choice([0, 3, 16, 29, 32], 60)]
    sizes_c = [int(x) for x in rng.choice([0, 5, 16, 31], 60)]
    prev = workloads.random_batch(rng, sizes_p, 3, dk, dv, decay="scalar", max_depth=8,
                                  depth_cap=8, max_nodes=32)
    cur = workloads.random_batch(rng, sizes_c, 3, dk, dv, decay="scalar", max_depth=8,
                                 depth_cap=8, max_nodes=32)
    dp, dc, ln = _two_step(prev, cur)
    Hd = dc.H0.cpu().numpy()
    for b in np.where(ln == 0)[0]:
        assert np.array_equal(Hd[b], prev.H0[b])


def test_fused_commit_verify_folded_sampled():
    prev = workloads.config2(seed=41, H=24 * 8)
    cur = workloads.config2(seed=42, H=24 * 8)
    rng = np.random.default_rng(1)
    _two_step(prev, cur, units=np.sort(rng.choice(prev.B * prev.H, 96, replace=False)))


def test_fused_commit_verify_bad_path_reports_and_skips_commit():
    """A pending path that is not a root path of the previous tree: TV_ERR_TREE and
    that request's state unchanged; the other requests commit and verify."""
    import torch
    import oracle
    import tree_speculative_verify_tv_gb300 as tv
    prev = workloads.config2(seed=51, B=6, H=4)
    cur = workloads.config2(seed=52, B=6, H=4)
    dp, dc = tv.DeviceBatch(prev), tv.DeviceBatch(cur)
    dc.H0.copy_(dp.H0)
    dp.status.zero_()
    dp.accept()
    torch.cuda.synchronize()
    ln = dp.accept_len[:prev.B].cpu().numpy()
    r = int(np.argmax(ln >= 2))
    assert ln[r] >= 2
    path = dp.path.clone()
    path[r, 0], path[r, 1] = path[r, 1].item(), path[r, 0].item()  # no longer a root path
    dp.path.copy_(path)
    dc.status.zero_()
    dc.commit_verify(dp)
    torch.cuda.synchronize()
    assert int(dc.status[0]) == 6
    assert torch.equal(dc.H0[r], dp.H0[r])


def test_fused_timeout_path_then_normal_call():
    """The test hook makes each CTA's first wait for a state chunk expire: the call
    reports TV_ERR_TIMEOUT (after waiting for its copies and products in flight and
    freeing its tensor memory); the next ordinary call on the same stream is exact."""
    import torch
    import tree_speculative_verify_tv_gb300 as tv
    b = workloads.config2(seed=61, H=24 * 4)
    d = tv.DeviceBatch(b)
    d.status.zero_()
    tv.tv_verify(d.problem(), d.H0, d.q, d.k, d.v, d.g, d.out, d.status,
                 variant=FUSED | tv.TV_VARIANT_TEST_EXPIRE_WAIT)
    torch.cuda.synchronize()
    assert int(d.status[0]) == tv.TV_ERR_TIMEOUT
    for _ in range(2):
        d.status.zero_()
        d.out.fill_(float("nan"))
        tv.tv_verify(d.problem(), d.H0, d.q, d.k, d.v, d.g, d.out, d.status, variant=FUSED)
        torch.cuda.synchronize()
        assert int(d.status[0]) == 0
    rng = np.random.default_rng(2)
    units = np.sort(rng.choice(b.B * b.H, 64, replace=False))
    check_verify(b, d.out[:b.T].cpu().numpy().astype(np.float64), units=units)
