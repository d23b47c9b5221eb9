"""GPU parity of the per-channel-decay kernel of TV_VARIANT_TC_FUSED: the three
products of a (request, head) unit on tcgen05 with the decay folded into the factors
(q~ = e^{G} q, k~ = e^{-G} k, hi/lo split), key channels in groups of 64, trees of up
to 64 nodes, dv = 128.  Cases: the GLA-like configuration (all units against the
fp64 oracle, and against the staged large-tree kernel), ragged trees of 0-64 nodes at
dk = 64 and 128, 64-node chains and stars, path sums outside the factors' range (the
walk that replaces the score product then), growing decay, non-finite rows next to a
request, malformed trees between valid ones, canaries around the outputs, and the
timeout path (TV_VARIANT_TEST_EXPIRE_WAIT)."""
import numpy as np
import pytest

import workloads
from gpu_util import check_verify, row_rel_err, run_library

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


def _verify(batch, variant=FUSED):
    res = run_library(batch, variant=variant, steps=("verify",))
    return res["status"], res["out"]


def _diag(rng, sizes, H, dk, *, depth_cap=8, max_depth=8, max_nodes=None):
    return workloads.random_batch(rng, sizes, H, dk, 128, decay="diag", depth_cap=depth_cap,
                                  max_depth=max_depth, max_nodes=max_nodes)


def test_fdiag_gla_layer_all_units():
    """GLA-like layer, B=32, H=16, 64-node best-first trees: 512 units, all checked."""
    b = workloads.config3()
    st, out = _verify(b)
    assert st == 0
    check_verify(b, out, threads=16)


def test_fdiag_is_auto_for_the_gla_layer_and_matches_the_staged_kernel():
    import tree_speculative_verify_tv_gb300 as tv
    b = workloads.config3(seed=7)
    assert tv.tv_verify_variant(tv.DeviceBatch(b).problem()) == FUSED
    st, out = _verify(b)
    st2, out2 = _verify(b, variant=4)
    assert st == 0 and st2 == 0
    # two fp32 evaluations of the same sums, each within ~1e-5 of exact
    assert row_rel_err(out, out2) <= 2e-4


@pytest.mark.parametrize("dk", [64, 128])
@pytest.mark.parametrize("cap", [16, 32, 64])
def test_fdiag_ragged_with_empty_requests(dk, cap):
    """Ragged trees of 0..cap nodes (node tiles of 16, 32 and 64)."""
    rng = np.random.default_rng(dk + cap)
    sizes = rng.integers(0, cap + 1, 70)
    sizes[::9] = 0
    b = _diag(rng, sizes, 3, dk, depth_cap=10, max_depth=10, max_nodes=cap)
    st, out = _verify(b)
    assert st == 0
    check_verify(b, out)


def test_fdiag_chains_and_stars_of_64():
    """64-node trees made of two chains of 32 (the deepest trees the library takes:
    path sums over 32 rows, five rounds of pointer doubling, ancestors on both halves
    of the 64-bit masks) and stars of 64 roots, interleaved."""
    rng = np.random.default_rng(9)
    b = _diag(rng, [64] * 12, 4, 128, depth_cap=32, max_depth=32)
    chains = np.concatenate([np.arange(-1, 31), np.concatenate([[-1], np.arange(32, 63)])])
    for r in range(b.B):
        s = int(b.node_offsets[r])
        par = chains.astype(np.int32) if r % 2 == 0 else np.full(64, -1, np.int32)
        b.parent[s:s + 64] = par
        b.depth[s:s + 64] = workloads.depths_from_parents(par)
    st, out = _verify(b)
    assert st == 0
    check_verify(b, out)


def test_fdiag_path_sums_out_of_range_take_the_walk():
    """Requests whose path sums leave +-69 in some channel (strong decay in one
    channel, or in all) next to requests in range: the walk gives their weights."""
    rng = np.random.default_rng(13)
    b = _diag(rng, [40, 64, 17, 64, 33, 5], 4, 128, depth_cap=8, max_depth=8)
    g = b.g.reshape(b.T, b.H, b.dk)
    o = b.node_offsets
    g[o[0]:o[1], :, 5] = -15.0        # one channel: G down to -120
    g[o[1]:o[2]] = -12.0              # every channel
    g[o[3]:o[4], 1, 100] = -30.0      # one head, one channel
    g[o[4]:o[5]] = 0.0                # no decay
    st, out = _verify(b)
    assert st == 0
    check_verify(b, out)


def test_fdiag_growing_decay_in_range():
    """g > 0 (growth) with path sums inside the range: factors above and below 1."""
    rng = np.random.default_rng(14)
    b = _diag(rng, [30, 64, 12], 4, 128, depth_cap=8, max_depth=8)
    g = b.g.reshape(b.T, b.H, b.dk)
    g[:] = np.abs(g) * 4.0
    st, out = _verify(b)
    assert st == 0
    check_verify(b, out)


def test_fdiag_neighbor_rows_do_not_leak():
    """q/k/g/v columns are copied in boxes of 16 nodes, so a request's boxes run into
    the next request's rows: non-finite values there must not reach its outputs."""
    rng = np.random.default_rng(46)
    b = _diag(rng, [5, 13, 17, 3, 9], 4, 128, max_nodes=32)
    s, e = int(b.node_offsets[2]), int(b.node_offsets[3])
    b.v[s:e] = 0x7F80  # bf16 +inf
    b.k[s:e] = 0x7FC0  # bf16 NaN
    b.q[s:e] = 0x7FC0
    b.g.reshape(b.T, b.H, b.dk)[s:e] = np.inf
    st, out = _verify(b)
    assert st == 0
    check_verify(b, out, units=[u for u in range(b.B * b.H) if u // b.H != 2])


def test_fdiag_malformed_trees_between_valid_ones():
    rng = np.random.default_rng(12)
    sizes = [int(x) for x in rng.choice([0, 1, 9, 33, 64], 60)]
    b = _diag(rng, sizes, 3, 128, max_nodes=64)
    bad = [r for r in range(b.B) if sizes[r] >= 9][::5]
    for r in bad:
        s = int(b.node_offsets[r])
        b.parent[s + 3] = 5 if r % 2 else 3  # a parent after its child / itself
    st, out = _verify(b)
    assert st == 6  # TV_ERR_TREE
    for r in bad:
        s, e = int(b.node_offsets[r]), int(b.node_offsets[r + 1])
        assert np.all(out[s:e] == 0.0)
    check_verify(b, out, units=[u for u in range(b.B * b.H) if u // b.H not in bad])


def test_fdiag_depth_mismatch_and_too_deep():
    rng = np.random.default_rng(15)
    b = _diag(rng, [12, 12, 12, 12], 3, 128, depth_cap=6, max_depth=6)
    s1, s2 = int(b.node_offsets[1]), int(b.node_offsets[2])
    b.depth[s1 + 4] += 1
    chain = np.arange(-1, 11, dtype=np.int32)
    b.parent[s2:s2 + 12] = chain                    # depth 12 > max_depth 6
    b.depth[s2:s2 + 12] = workloads.depths_from_parents(chain)
    st, out = _verify(b)
    assert st == 6
    assert np.all(out[s1:int(b.node_offsets[3])] == 0.0)
    check_verify(b, out, units=[u for u in range(b.B * b.H) if u // b.H in (0, 3)])


def test_fdiag_outputs_stay_inside_their_buffers():
    import torch
    import tree_speculative_verify_tv_gb300 as tv
    b = workloads.config3(seed=19, B=5, H=7)
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


def test_fdiag_timeout_path_then_normal_call():
    """The test hook makes each CTA's first wait for a state chunk expire: the call
    reports TV_ERR_TIMEOUT (after its copies and products in flight are done and its
    tensor memory is freed); the next ordinary call on the same stream is exact."""
    import torch
    import tree_speculative_verify_tv_gb300 as tv
    b = workloads.config3(seed=61, B=8)
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
