"""GPU parity of the large-tree per-channel-decay member of TV_VARIANT_TC_FUSED: trees
of up to 256 nodes and depth 16, dv = 128, the context product on tcgen05 (q~ hi/lo
against the state rows hi/lo) and the tree term by fp32 walks of each node's root
path.  Cases: the large-tree stack at reduced size (every unit against the fp64
oracle) and against the staged large-tree kernel, ragged trees of 0-256 nodes (one
and two 128-row tiles) at dk = 64 and 128, chains of depth 16 and stars of 256
roots, path sums far below -69 (e^{G} under the fp32 range: the walk sums each
pair's decay, so no factor leaves the range), growing decay, non-finite rows next to
a request (copy boxes of 32 nodes), malformed trees and depth errors among many units
per persistent CTA, canaries around the outputs, and the timeout path
(TV_VARIANT_TEST_EXPIRE_WAIT)."""
import numpy as np
import pytest

import workloads
from gpu_util import check_verify, row_rel_err, run_library

pytestmark = pytest.mark.gpu

FUSED = 3
TILED = 4


@pytest.fixture(scope="module", autouse=True)
def _lib():
    import torch
    if not torch.cuda.is_available():
        pytest.skip("no CUDA device")
    import tree_speculative_verify_tv_gb300 as tv
    tv.build()
    tv.load()


def _verify(batch, variant=FUSED):
    res = run_library(batch, variant=variant, steps=("verify",))
    return res["status"], res["out"]


def _diag(rng, sizes, H, dk, *, depth_cap=8, max_depth=16, max_nodes=256):
    return workloads.random_batch(rng, sizes, H, dk, 128, decay="diag", depth_cap=depth_cap,
                                  max_depth=max_depth, max_nodes=max_nodes)


def test_fwalk_large_tree_stack_reduced_all_units():
    """B=2, 2 layers x 4 heads of the large-tree stack (256-node best-first trees,
    depth <= 16): every unit against the oracle."""
    b = workloads.config5(B=2, layers=2, heads=4, seed=21)
    st, out = _verify(b)
    assert st == 0
    check_verify(b, out, threads=16)


def test_fwalk_is_auto_and_matches_the_staged_kernel():
    import tree_speculative_verify_tv_gb300 as tv
    b = workloads.config5(B=3, layers=4, heads=8, seed=22)
    assert tv.tv_verify_variant(tv.DeviceBatch(b).problem()) == FUSED
    st, out = _verify(b)
    st2, out2 = _verify(b, variant=TILED)
    assert st == 0 and st2 == 0
    # two fp32 evaluations of the same sums, each within ~1e-5 of exact
    assert row_rel_err(out, out2) <= 2e-4


@pytest.mark.parametrize("dk", [64, 128])
@pytest.mark.parametrize("cap", [100, 256])
def test_fwalk_ragged_with_empty_requests(dk, cap):
    """Ragged trees of 0..cap nodes: one 128-row tile or two, partial copy boxes."""
    rng = np.random.default_rng(dk + cap)
    sizes = rng.integers(0, cap + 1, 40)
    sizes[::7] = 0
    sizes[1] = cap
    sizes[2] = min(129, cap)
    sizes[3] = min(128, cap)
    b = _diag(rng, sizes, 3, dk, depth_cap=12, max_depth=16, max_nodes=cap)
    st, out = _verify(b)
    assert st == 0
    check_verify(b, out, threads=16)


def test_fwalk_chains_of_16_and_stars_of_256():
    """256-node trees made of sixteen chains of depth 16 (every path slot used), and
    stars of 256 roots (a path of one node each), interleaved."""
    rng = np.random.default_rng(9)
    b = _diag(rng, [256] * 6, 3, 128, depth_cap=16, max_depth=16)
    chains = np.concatenate([np.concatenate([[-1], np.arange(16 * c, 16 * c + 15)])
                             for c in range(16)]).astype(np.int32)
    for r in range(b.B):
        s = int(b.node_offsets[r])
        par = chains if r % 2 == 0 else np.full(256, -1, np.int32)
        b.parent[s:s + 256] = par
        b.depth[s:s + 256] = workloads.depths_from_parents(par)
    st, out = _verify(b)
    assert st == 0
    check_verify(b, out, threads=16)


def test_fwalk_path_sums_far_below_the_fp32_range():
    """Requests whose path sums fall to -150 or -360 in some channels next to requests
    with moderate decay: pair decays are summed along the walk, so the outputs stay
    exact where a factor e^{-G} would overflow."""
    rng = np.random.default_rng(13)
    b = _diag(rng, [140, 256, 17, 200, 33, 5], 4, 128, depth_cap=10, max_depth=16)
    g = b.g.reshape(b.T, b.H, b.dk)
    o = b.node_offsets
    g[o[0]:o[1], :, 5] = -15.0        # one channel: G down to -150
    g[o[1]:o[2]] = -12.0              # every channel
    g[o[3]:o[4], 1, 100] = -30.0      # one head, one channel
    g[o[4]:o[5]] = 0.0                # no decay
    st, out = _verify(b)
    assert st == 0
    check_verify(b, out, threads=16)


def test_fwalk_growing_decay_in_range():
    rng = np.random.default_rng(14)
    b = _diag(rng, [130, 256, 12], 4, 128, depth_cap=10, max_depth=16)
    g = b.g.reshape(b.T, b.H, b.dk)
    g[:] = np.abs(g) * 4.0
    st, out = _verify(b)
    assert st == 0
    check_verify(b, out)


def test_fwalk_neighbor_rows_do_not_leak():
    """q/k/g/v rows are copied in boxes of 32 nodes, so a request's boxes run into the
    next request's rows: non-finite values there must not reach its outputs."""
    rng = np.random.default_rng(46)
    b = _diag(rng, [70, 13, 150, 3, 90], 4, 128, max_nodes=256)
    s, e = int(b.node_offsets[2]), int(b.node_offsets[3])
    b.v[s:e] = 0x7F80  # bf16 +inf
    b.k[s:e] = 0x7FC0  # bf16 NaN
    b.q[s:e] = 0x7FC0
    b.g.reshape(b.T, b.H, b.dk)[s:e] = np.inf
    st, out = _verify(b)
    assert st == 0
    check_verify(b, out, units=[u for u in range(b.B * b.H) if u // b.H != 2])


def test_fwalk_malformed_trees_among_many_units():
    """About 1000 units, so each persistent CTA takes several in turn, with empty
    requests and malformed trees between valid ones."""
    rng = np.random.default_rng(12)
    sizes = [int(x) for x in rng.choice([0, 1, 9, 100, 129, 256], 120)]
    b = _diag(rng, sizes, 8, 128, max_nodes=256)
    bad = [r for r in range(b.B) if sizes[r] >= 9][::5]
    for r in bad:
        s = int(b.node_offsets[r])
        b.parent[s + 3] = 5 if r % 2 else 3  # a parent after its child / itself
    st, out = _verify(b)
    assert st == 6  # TV_ERR_TREE
    for r in bad:
        s, e = int(b.node_offsets[r]), int(b.node_offsets[r + 1])
        assert np.all(out[s:e] == 0.0)
    check_verify(b, out, units=[u for u in range(b.B * b.H) if u // b.H not in bad], threads=16)


def test_fwalk_depth_mismatch_and_too_deep():
    rng = np.random.default_rng(15)
    b = _diag(rng, [140, 140, 140, 140], 3, 128, depth_cap=6, max_depth=12)
    s1, s2 = int(b.node_offsets[1]), int(b.node_offsets[2])
    b.depth[s1 + 4] += 1
    chain = np.arange(-1, 13, dtype=np.int32)                # depth 14 > max_depth 12
    b.parent[s2:s2 + 14] = chain
    b.depth[s2:s2 + 14] = workloads.depths_from_parents(chain)
    st, out = _verify(b)
    assert st == 6
    assert np.all(out[s1:int(b.node_offsets[3])] == 0.0)
    check_verify(b, out, units=[u for u in range(b.B * b.H) if u // b.H in (0, 3)])


def test_fwalk_deeper_trees_take_the_staged_kernel():
    """A declared max_depth above 16 leaves the walk kernel: AUTO picks the staged
    large-tree kernel, and TV_VARIANT_TC_FUSED reports TV_ERR_UNSUPPORTED."""
    import tree_speculative_verify_tv_gb300 as tv
    rng = np.random.default_rng(16)
    b = _diag(rng, [200, 90], 2, 128, depth_cap=8, max_depth=17)
    d = tv.DeviceBatch(b)
    assert tv.tv_verify_variant(d.problem()) == TILED
    assert tv.tv_verify_supports(d.problem(), FUSED) == 0


def test_fwalk_outputs_stay_inside_their_buffers():
    import torch
    import tree_speculative_verify_tv_gb300 as tv
    b = workloads.config5(B=2, layers=1, heads=5, seed=19)
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


def test_fwalk_timeout_path_then_normal_call():
    """The test hook makes each CTA's first wait for a group's inputs expire: the call
    reports TV_ERR_TIMEOUT (after its copies and products in flight are done and its
    tensor memory is freed); the next ordinary calls on the same stream are exact."""
    import torch
    import tree_speculative_verify_tv_gb300 as tv
    b = workloads.config5(B=2, layers=2, heads=4, seed=61)
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
    check_verify(b, d.out[:b.T].cpu().numpy().astype(np.float64))
