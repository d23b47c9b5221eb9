"""GPU parity: the CUDA library against the fp64 oracle, called through the C ABI.

Outputs and committed states within 2e-3 normwise relative error (per node row,
per (request, head) matrix); acceptance length, path and bonus bit-exact.
"""
import numpy as np
import pytest

import workloads
from gpu_util import (TOL, check_accept, check_commit, check_verify, mat_rel_err, row_rel_err,
                      run_library)

pytestmark = pytest.mark.gpu

VARIANTS = {"auto": 0, "simt": 1, "tc": 2, "tiled": 4}


@pytest.fixture(scope="module", autouse=True)
def _lib():
    import torch
    if not torch.cuda.is_available():
        pytest.skip("no CUDA device")
    import tree_speculative_verify_tv_gb300 as tv
    tv.build()
    tv.load()


def _tc_supported(batch):
    """Whether the library takes this shape on the one-unit tcgen05 kernel (it
    reports TV_ERR_UNSUPPORTED for a forced tensor-core run otherwise)."""
    import tree_speculative_verify_tv_gb300 as tv
    p = tv.make_problem(batch.B, batch.H, batch.dk, batch.dv, batch.T, batch.max_nodes,
                        batch.max_depth, tv.TV_DECAY_DIAG if batch.decay == "diag" else 0,
                        tv.TV_BF16 if batch.qkv_dtype == "bf16" else tv.TV_F32, 16, 16, 16)
    return tv.tv_verify_supports(p, tv.TV_VARIANT_TC) == 1


def _full_check(batch, variant="auto", units=None):
    if variant == "tc" and not _tc_supported(batch):
        pytest.skip("shape outside the tensor-core kernel")
    res = run_library(batch, variant=VARIANTS[variant])
    assert res["status"] == 0, res["status"]
    ev = check_verify(batch, res["out"], units=units)
    ln, path = check_accept(batch, res)
    ec = check_commit(batch, res["H_new"], ln, path, units=units)
    return ev, ec


@pytest.mark.parametrize("variant", ["simt", "auto"])
@pytest.mark.parametrize("c", [1, 2, 3, 4])
def test_config_full_size(c, variant):
    _full_check(workloads.make_config(c), variant)


@pytest.mark.parametrize("c", [2, 3, 4])
def test_config_full_size_tensor_core(c):
    b = workloads.make_config(c)
    assert _tc_supported(b)
    _full_check(b, "tc")


@pytest.mark.parametrize("dk,dv", [(64, 64), (64, 128), (128, 64), (128, 128)])
def test_tensor_core_ragged_scalar(dk, dv):
    rng = np.random.default_rng(dk + 7 * dv)
    sizes = [1, 16, 17, 0, 72, 64, 31, 128, 5]   # 128 nodes: the largest the forced runs use
    b = workloads.random_batch(rng, sizes, 3, dk, dv, decay="scalar", qkv_dtype="bf16",
                               depth_cap=16, max_depth=16, max_nodes=128)
    assert _tc_supported(b)
    _full_check(b, "tc")


@pytest.mark.parametrize("dk,dv", [(64, 64), (64, 128), (128, 64), (128, 128)])
def test_tensor_core_ragged_diagonal(dk, dv):
    rng = np.random.default_rng(3 * dk + dv)
    sizes = [1, 16, 17, 0, 64, 31, 5, 48]
    b = workloads.random_batch(rng, sizes, 3, dk, dv, decay="diag", qkv_dtype="bf16",
                               depth_cap=16, max_depth=16, max_nodes=64)
    assert _tc_supported(b)
    _full_check(b, "tc")


def test_tensor_core_agrees_with_simt():
    b = workloads.config2(seed=3)
    r_tc = run_library(b, variant=2, steps=("verify",))
    r_simt = run_library(b, variant=1, steps=("verify",))
    assert r_tc["status"] == 0 and r_simt["status"] == 0
    assert row_rel_err(r_tc["out"], r_simt["out"]) <= 1e-4


def test_tensor_core_rejects_unsupported_shapes():
    import tree_speculative_verify_tv_gb300 as tv
    b = workloads.config5(B=1, layers=1, heads=2)   # 256-node diagonal-decay trees
    assert not _tc_supported(b)
    with pytest.raises(tv.TVError) as ei:
        run_library(b, variant=2, steps=("verify",))
    assert ei.value.code == tv.TV_ERR_UNSUPPORTED


@pytest.mark.parametrize("seed", range(10))
def test_config1_seeds(seed):
    _full_check(workloads.config1(seed=seed), "simt")


@pytest.mark.parametrize("seed", range(3))
@pytest.mark.parametrize("variant", ["simt", "auto"])
def test_config2_seeds(seed, variant):
    _full_check(workloads.config2(seed=seed), variant)


def _auto_variant(batch):
    import tree_speculative_verify_tv_gb300 as tv
    p = tv.make_problem(batch.B, batch.H, batch.dk, batch.dv, batch.T, batch.max_nodes,
                        batch.max_depth, tv.TV_DECAY_DIAG if batch.decay == "diag" else 0,
                        tv.TV_BF16 if batch.qkv_dtype == "bf16" else tv.TV_F32, 16, 16, 16)
    return tv.tv_verify_variant(p)


def test_automatic_kernel_choice():
    """TV_VARIANT_AUTO: the fused kernels for scalar-decay trees of <= 32 nodes and
    per-channel trees at dv = 128 of <= 64 nodes or of <= 256 nodes and depth 16, the
    one-unit kernel for larger scalar-decay trees and other small per-channel trees,
    the staged large-tree kernel for trees too large for those."""
    import tree_speculative_verify_tv_gb300 as tv
    assert _auto_variant(workloads.make_config(2)) == tv.TV_VARIANT_TC_FUSED
    assert _auto_variant(workloads.make_config(3)) == tv.TV_VARIANT_TC_FUSED
    assert _auto_variant(workloads.make_config(4)) == tv.TV_VARIANT_TC
    assert _auto_variant(workloads.config5(B=2, layers=1, heads=2)) == tv.TV_VARIANT_TC_FUSED
    small = workloads.random_batch(np.random.default_rng(50), [32, 20], 2, 128, 128, decay="diag",
                                   qkv_dtype="bf16", depth_cap=8, max_depth=8, max_nodes=32)
    assert _auto_variant(small) == tv.TV_VARIANT_TC_FUSED
    small64 = workloads.random_batch(np.random.default_rng(51), [32, 20], 2, 128, 64,
                                     decay="diag", qkv_dtype="bf16", depth_cap=8, max_depth=8,
                                     max_nodes=32)
    assert _auto_variant(small64) == tv.TV_VARIANT_TC
    assert _auto_variant(workloads.make_config(1)) == tv.TV_VARIANT_SIMT


@pytest.mark.parametrize("variant", ["simt", "auto"])
def test_config5_reduced(variant):
    _full_check(workloads.config5(B=2, layers=2, heads=4, seed=11), variant)


def test_config5_full_size_every_unit():
    """B=8, 36 layers x 32 heads, 256-node trees, the launch the benchmark times: every
    one of the 9216 (request, head) units compared with the oracle (outputs and
    committed states), the oracle threaded over all host cores and run in eight
    slices of units to bound its memory."""
    import os
    b = workloads.config5()
    res = run_library(b, variant=VARIANTS["auto"])
    assert res["status"] == 0, res["status"]
    ln, path = check_accept(b, res)
    threads = os.cpu_count() or 8
    units = np.arange(b.B * b.H, dtype=np.int32)
    for part in np.array_split(units, 8):
        check_verify(b, res["out"], units=part, threads=threads)
        check_commit(b, res["H_new"], ln, path, units=part, threads=threads)


SHAPES = [  # (dk, dv, decay, dtype)
    (8, 8, "scalar", "f32"), (16, 24, "diag", "f32"), (32, 16, "scalar", "bf16"),
    (64, 64, "diag", "bf16"), (64, 128, "scalar", "bf16"), (128, 64, "diag", "bf16"),
    (96, 40, "scalar", "bf16"), (128, 128, "diag", "f32"), (256, 256, "scalar", "bf16"),
    (256, 32, "diag", "bf16"),
]


@pytest.mark.parametrize("variant", ["simt", "auto"])
@pytest.mark.parametrize("shape", SHAPES, ids=lambda s: "%dx%d-%s-%s" % s)
def test_random_shapes_ragged(shape, variant):
    dk, dv, decay, dt = shape
    rng = np.random.default_rng(dk * 1000 + dv)
    sizes = [0, 1, 37, 5, 256, 64, 0, 33, 100, 2]
    b = workloads.random_batch(rng, sizes, 3, dk, dv, decay=decay, qkv_dtype=dt, depth_cap=32,
                               max_depth=32, max_nodes=256)
    _full_check(b, variant)


@pytest.mark.parametrize("variant", ["simt", "auto"])
def test_deepest_chain_and_widest_star(variant):
    rng = np.random.default_rng(3)
    chain = np.arange(-1, 31, dtype=np.int32)          # depth 32
    star = np.full(256, -1, dtype=np.int32)            # 256 children of the context
    parents = [chain, star]
    b = workloads.assemble(rng, parents, 4, 128, 64, decay="diag", qkv_dtype="bf16",
                           g_kind="logsig16", h0_std=0.05, vocab=2, max_depth=32, max_nodes=256)
    # plant a full-depth acceptance along the chain
    b.draft[:32] = 1
    b.target[:32] = 1
    b.root_argmax[0] = 1
    _full_check(b, variant)
    res = run_library(b, variant=VARIANTS[variant])
    assert res["len"][0] == 32


def test_strong_decay_and_zero_decay():
    rng = np.random.default_rng(9)
    for g_kind, scale in (("zero", 0.0), ("softplus01", 30.0)):
        b = workloads.random_batch(rng, [17, 40], 2, 64, 64, decay="diag", qkv_dtype="bf16",
                                   g_kind="softplus01", depth_cap=12, max_depth=12)
        b.g = (b.g * scale).astype(np.float32)
        _full_check(b, "simt")
        _full_check(b, "auto")


@pytest.mark.parametrize("c", [1, 2, 3, 4])
def test_accept_commit_fused_matches_oracle(c):
    b = workloads.make_config(c)
    res = run_library(b, steps=("verify", "accept_commit"))
    assert res["status"] == 0
    ln, path = check_accept(b, res)
    check_commit(b, res["H_new"], ln, path)


def test_accept_commit_fused_equals_separate_calls():
    b = workloads.config5(B=2, layers=2, heads=4, seed=3)
    r1 = run_library(b, steps=("accept", "commit"))
    r2 = run_library(b, steps=("accept_commit",))
    assert r1["status"] == 0 and r2["status"] == 0
    for key in ("len", "path", "bonus"):
        assert np.array_equal(r1[key], r2[key])
    assert np.array_equal(r1["H_new"], r2["H_new"])
    r3 = run_library(b, steps=("accept_commit",), commit_in_place=True)
    assert np.array_equal(r1["H_new"], r3["H_new"])


def test_accept_commit_fused_malformed_tree():
    b = _bad_tree_batch()
    s0 = b.node_offsets[1]
    b.parent[s0 + 2] = 4                                  # request 1: parent after child
    import torch
    import tree_speculative_verify_tv_gb300 as tv
    d = tv.DeviceBatch(b)
    d.status.zero_()
    d.H_new.fill_(5.0)
    d.accept_commit()
    torch.cuda.synchronize()
    assert int(d.status[0]) == 6
    assert int(d.accept_len[1]) == 0 and int(d.bonus[1]) == -1
    assert bool(torch.all(d.path[1] == -1))
    assert bool(torch.all(d.H_new[1] == 5.0))             # request 1 untouched
    # requests 0 and 2 are committed as the oracle does
    import oracle
    keep = [0, 2]
    ln = d.accept_len[:b.B].cpu().numpy()
    path = d.path[:b.B].cpu().numpy()
    for bb in keep:
        s, e = b.node_offsets[bb], b.node_offsets[bb + 1]
        L, p, bo = oracle.accept(b.parent[s:e], b.draft[s:e], b.target[s:e], b.root_argmax[bb],
                                 b.max_depth)
        assert L == ln[bb] and np.array_equal(p, path[bb]) and bo == int(d.bonus[bb])
    ref = oracle.commit(b, ln, path, units=[u for u in range(b.B * b.H) if u // b.H in keep])
    Hn = d.H_new.cpu().numpy().astype(np.float64)
    for u, Hr in ref.items():
        bb, h = divmod(u, b.H)
        assert mat_rel_err(Hn[bb, h], Hr) <= TOL


def test_commit_in_place():
    b = workloads.config2(seed=4)
    res = run_library(b, commit_in_place=True)
    assert res["status"] == 0
    ln, path = check_accept(b, res)
    check_commit(b, res["H_new"], ln, path)


def test_outputs_stay_inside_their_buffers():
    """Canary check: verify and commit write exactly their own rows."""
    import torch
    import tree_speculative_verify_tv_gb300 as tv
    b = workloads.random_batch(np.random.default_rng(1), [3, 9, 1], 2, 64, 64, decay="scalar")
    d = tv.DeviceBatch(b)
    canary = 12345.0
    out = torch.full((b.T + 8, b.H, b.dv), canary, device="cuda")
    Hn = torch.full((b.B + 2, b.H, b.dk, b.dv), canary, device="cuda")
    d.status.zero_()
    tv.tv_verify(d.problem(), d.H0, d.q, d.k, d.v, d.g, out, d.status)
    d.accept()
    tv.tv_commit(d.problem(), d.H0, d.g, d.k, d.v, d.path, d.accept_len, Hn, d.status)
    torch.cuda.synchronize()
    assert int(d.status[0]) == 0
    assert torch.all(out[b.T:] == canary) and torch.all(Hn[b.B:] == canary)
    assert not torch.any(out[:b.T] == canary)


# ------------------------------------------------------------------ device-detected errors


@pytest.mark.parametrize("decay", ["diag", "scalar"])
def test_tiled_tensor_core_ragged(decay):
    """The node-tiled tcgen05 kernel on ragged trees: empty, single-node, one tile
    exactly, one node over a tile, several tiles and the largest tree."""
    rng = np.random.default_rng(41 if decay == "diag" else 42)
    b = workloads.random_batch(rng, [0, 1, 63, 64, 65, 130, 256], 2, 128, 128, decay=decay,
                               qkv_dtype="bf16", depth_cap=12, max_depth=16)
    _full_check(b, "tiled")


def test_tiled_tensor_core_config3():
    """The GLA-like configuration (64-node best-first trees, per-channel decay) on
    the node-tiled kernel."""
    _full_check(workloads.make_config(3), "tiled")


def test_tiled_tensor_core_deepest_chain():
    b = workloads.random_batch(np.random.default_rng(43), [32, 200], 2, 128, 128,
                               decay="diag", qkv_dtype="bf16", depth_cap=32, max_depth=32)
    s = int(b.node_offsets[0])
    b.parent[s:s + 32] = np.arange(-1, 31, dtype=np.int32)
    b.depth[s:s + 32] = np.arange(1, 33, dtype=np.int32)
    _full_check(b, "tiled")


def test_tiled_tensor_core_malformed_tree():
    rng = np.random.default_rng(44)
    b = workloads.random_batch(rng, [6, 70, 7], 2, 128, 128, decay="diag", qkv_dtype="bf16",
                               depth_cap=6, max_depth=6)
    s = b.node_offsets[1]
    b.parent[s + 66] = 68
    res = run_library(b, variant=4, steps=("verify",))
    assert res["status"] == 6  # TV_ERR_TREE
    e = b.node_offsets[2]
    assert np.all(res["out"][s:e] == 0.0)
    import oracle
    units = [u for u in range(b.B * b.H) if u // b.H != 1]
    ref = oracle.verify(b, units=units)
    for u, o in ref.items():
        bb, h = divmod(u, b.H)
        ss, ee = b.node_offsets[bb], b.node_offsets[bb + 1]
        assert row_rel_err(res["out"][ss:ee, h], o) <= TOL


@pytest.mark.parametrize("decay", ["diag", "scalar"])
def test_tiled_tensor_core_neighbor_rows_do_not_leak(decay):
    """The large-tree kernels copy k, g and v rows in boxes of 32 nodes, so a
    request's boxes run into the next request's rows: non-finite values there must
    not reach its outputs."""
    rng = np.random.default_rng(46)
    b = workloads.random_batch(rng, [5, 40, 17, 70], 2, 128, 128, decay=decay, qkv_dtype="bf16",
                               depth_cap=8, max_depth=16)
    s, e = int(b.node_offsets[2]), int(b.node_offsets[3])
    b.v[s:e] = 0x7F80  # bf16 +inf
    b.k[s:e] = 0x7FC0  # bf16 NaN
    b.g[s:e] = np.float32(np.inf)
    res = run_library(b, variant=4, steps=("verify",))
    assert res["status"] == 0
    check_verify(b, res["out"], units=[u for u in range(b.B * b.H) if u // b.H != 2])


@pytest.mark.parametrize("decay", ["diag", "scalar"])
def test_tiled_tensor_core_many_units_with_empty_and_malformed(decay):
    """The staged kernel runs one CTA per SM over the (request, head) units in turn:
    512 units, so every CTA takes several, with empty requests and malformed trees
    between valid ones (units that skip their phases must keep every later unit's
    copies and barriers in step)."""
    rng = np.random.default_rng(48 if decay == "diag" else 49)
    sizes = [int(x) for x in rng.choice([0, 1, 17, 64, 100, 128], 64)]
    b = workloads.random_batch(rng, sizes, 8, 128, 128, decay=decay, qkv_dtype="bf16",
                               depth_cap=10, max_depth=12, max_nodes=128)
    bad = [r for r in range(b.B) if sizes[r] >= 17][::5]
    for r in bad:  # a parent after its child
        s = int(b.node_offsets[r])
        b.parent[s + 3] = 9
    res = run_library(b, variant=4, steps=("verify",))
    assert res["status"] == 6  # TV_ERR_TREE
    for r in bad:
        s, e = int(b.node_offsets[r]), int(b.node_offsets[r + 1])
        assert np.all(res["out"][s:e] == 0.0)
    check_verify(b, res["out"], units=[u for u in range(b.B * b.H) if u // b.H not in bad])


@pytest.mark.parametrize("md", [21, 22])
def test_tiled_tensor_core_staged_depth_limit(md):
    """256-node trees as deep as the staged kernel's shared-memory plan allows (21)
    and one deeper (the node-tiled kernel), each with a chain to the deepest level."""
    rng = np.random.default_rng(47 + md)
    b = workloads.random_batch(rng, [256, 200], 2, 128, 128, decay="diag", qkv_dtype="bf16",
                               depth_cap=8, max_depth=md)
    s = int(b.node_offsets[0])
    par = np.empty(256, np.int32)
    par[:md] = np.arange(-1, md - 1)
    par[md:] = rng.integers(-1, md - 1, 256 - md)
    dep = np.zeros(256, np.int32)
    for i in range(256):
        dep[i] = 1 if par[i] < 0 else dep[par[i]] + 1
    assert dep.max() == md
    b.parent[s:s + 256], b.depth[s:s + 256] = par, dep
    res = run_library(b, variant=4, steps=("verify",))
    assert res["status"] == 0
    check_verify(b, res["out"])


def test_tiled_tensor_core_rejects_other_dims():
    b = workloads.random_batch(np.random.default_rng(45), [4], 1, 64, 64, decay="diag",
                               qkv_dtype="bf16")
    with pytest.raises(Exception):
        run_library(b, variant=4, steps=("verify",))


def _bad_tree_batch():
    rng = np.random.default_rng(2)
    return workloads.random_batch(rng, [6, 5, 7], 2, 64, 64, decay="scalar", qkv_dtype="bf16",
                                  depth_cap=6, max_depth=6)


@pytest.mark.parametrize("variant", ["simt", "auto", "tc"])
@pytest.mark.parametrize("defect", ["parent_forward", "parent_self", "depth_mismatch",
                                    "too_deep"])
def test_malformed_tree_sets_status_and_zero_rows(defect, variant):
    b = _bad_tree_batch()
    s = b.node_offsets[1]                      # corrupt request 1 only
    if defect == "parent_forward":
        b.parent[s + 2] = 4
    elif defect == "parent_self":
        b.parent[s + 3] = 3
    elif defect == "depth_mismatch":
        b.depth[s + 4] += 1
    else:
        b.max_depth = int(b.depth[s:b.node_offsets[2]].max()) - 1
        if b.max_depth < 1:
            pytest.skip("tree too shallow")
    res = run_library(b, variant=VARIANTS[variant], steps=("verify",))
    assert res["status"] == 6  # TV_ERR_TREE
    e = b.node_offsets[2]
    assert np.all(res["out"][s:e] == 0.0)
    # the other requests are still correct
    import oracle
    units = [u for u in range(b.B * b.H) if u // b.H != 1]
    if defect == "too_deep":
        return
    ref = oracle.verify(b, units=units)
    for u, o in ref.items():
        bb, h = divmod(u, b.H)
        ss, ee = b.node_offsets[bb], b.node_offsets[bb + 1]
        assert row_rel_err(res["out"][ss:ee, h], o) <= TOL


def test_bad_offsets_set_status():
    b = _bad_tree_batch()
    b.node_offsets = b.node_offsets.copy()
    b.node_offsets[2] = b.node_offsets[1] - 1   # negative length for request 1
    res = run_library(b, steps=("verify",))
    assert res["status"] == 6


def test_accept_path_longer_than_bound_sets_status():
    n = 6
    chain = np.arange(-1, n - 1, dtype=np.int32)
    rng = np.random.default_rng(0)
    b = workloads.assemble(rng, [chain, chain], 1, 16, 16, decay="scalar", qkv_dtype="f32",
                           g_kind="softplus01", h0_std=0.1, vocab=2, max_depth=n)
    b.draft[:] = 1
    b.target[:] = 1
    b.root_argmax[:] = [1, 0]
    b.max_depth = 4                              # walk of request 0 would reach depth 6
    res = run_library(b, steps=("accept",))
    assert res["status"] == 6
    assert res["len"][0] == 0 and res["bonus"][0] == -1 and np.all(res["path"][0] == -1)
    assert res["len"][1] == 0 and res["bonus"][1] == 0  # request 1: nothing matches


def test_commit_rejects_path_that_is_not_a_root_path():
    import torch
    import tree_speculative_verify_tv_gb300 as tv
    b = workloads.config2(seed=1, B=2, H=2)
    d = tv.DeviceBatch(b)
    d.status.zero_()
    d.accept_len.copy_(torch.tensor([2, 1], dtype=torch.int32))
    d.path.copy_(torch.tensor([[0, 5, -1, -1], [3, -1, -1, -1]], dtype=torch.int32))  # 5 is not a child of 0
    d.H_new.fill_(7.0)
    d.commit()
    torch.cuda.synchronize()
    assert int(d.status[0]) == 6
    Hn = d.H_new.cpu().numpy()
    assert np.all(Hn[0] == 7.0)                  # request 0 untouched
    import oracle
    r = oracle.commit(b, np.array([0, 1], np.int32), np.array([[0, -1, -1, -1], [3, -1, -1, -1]],
                                                              np.int32), units=[2, 3])
    assert mat_rel_err(Hn[1, 0], r[2]) <= TOL and mat_rel_err(Hn[1, 1], r[3]) <= TOL


def test_empty_requests_and_empty_batch():
    b = workloads.random_batch(np.random.default_rng(4), [0, 0, 3, 0], 2, 16, 16,
                               decay="scalar", qkv_dtype="f32")
    _full_check(b, "simt")
    b0 = workloads.random_batch(np.random.default_rng(4), [0, 0], 2, 16, 16, decay="scalar",
                                qkv_dtype="f32")
    res = run_library(b0)
    assert res["status"] == 0 and np.all(res["len"] == 0)
    assert np.array_equal(res["bonus"], b0.root_argmax)
    assert mat_rel_err(res["H_new"], b0.H0.astype(np.float64)) == 0.0
