"""GPU parity of tv_tree_attention against the oracle's tree-masked softmax
attention (fp64).  Tolerance: the library's output bar, 2e-3 normwise relative
error per (node, head) output row, measured as for the verify outputs: the
largest |difference| over the row's d channels divided by the row's largest
|reference| value.  The kernel forms scores and sums in fp32 from exact bf16
inputs and feeds the softmax weights to the value sum as a bf16 hi + lo pair
(|p - hi - lo| <= 2^-16 p), so the weights add no error of the bf16 size."""

import numpy as np
import pytest

import oracle
import workloads

pytestmark = pytest.mark.gpu
TOL = 2e-3


@pytest.fixture(scope="module", autouse=True)
def _lib():
    import torch
    if not torch.cuda.is_available():
        pytest.skip("no CUDA device")
    import tree_speculative_verify_tv_gb300 as tv
    tv.build()
    tv.load()


def run(batch, a, H, Hkv, d, P, workspace=True, parent=None, ctx=None):
    import torch
    import tree_speculative_verify_tv_gb300 as tv
    cu = lambda x: torch.from_numpy(np.ascontiguousarray(x)).cuda()
    T = batch.T
    par = batch.parent if parent is None else parent
    out = torch.full((max(T, 1), H, d), float("nan"), dtype=torch.float32, device="cuda")
    st = torch.zeros(1, dtype=torch.int32, device="cuda")
    wsb = tv.tv_tree_attention_workspace_bytes(batch.B, T, batch.max_nodes, H, Hkv, d, P)
    ws = torch.empty(max(wsb // 4, 1), dtype=torch.float32, device="cuda") if workspace and wsb \
        else None
    rc = tv.tv_tree_attention(batch.B, T, batch.max_nodes, H, Hkv, d, P, cu(batch.node_offsets),
                              cu(par if T else np.zeros(1, np.int32)),
                              cu(a["ctx_len"] if ctx is None else ctx),
                              cu(a["q"]), cu(a["k_cache"]), cu(a["v_cache"]), cu(a["k_tree"]),
                              cu(a["v_tree"]), a["scale"], out, ws, wsb if ws is not None else 0,
                              st)
    assert rc == 0
    torch.cuda.synchronize()
    return int(st[0]), out[:T].cpu().numpy().astype(np.float64), wsb


def reference(batch, a):
    return oracle.tree_attention(batch.node_offsets, batch.parent, a["q_f32"], a["k_cache_f32"],
                                 a["v_cache_f32"], a["ctx_len"], a["k_tree_f32"], a["v_tree_f32"],
                                 a["scale"])


def row_errors(got, ref):
    num = np.max(np.abs(got - ref), axis=-1)
    den = np.maximum(np.max(np.abs(ref), axis=-1), 1e-30)
    return num / den


def check(batch, H, Hkv, d, ctx, seed, P=None, spike=0.0, tail_nan=False, workspace=True):
    a = workloads.attention_inputs(batch, H, Hkv, d, ctx, P=P, seed=seed, spike=spike,
                                   tail_nan=tail_nan)
    P = a["k_cache"].shape[2]
    st, got, wsb = run(batch, a, H, Hkv, d, P, workspace=workspace)
    assert st == 0
    ref = reference(batch, a)
    assert np.all(np.isfinite(got))
    err = row_errors(got, ref)
    assert err.max() < TOL, "worst row error %.3e" % err.max()
    return err.max(), wsb


def test_config2_tree_ragged_context_with_jumps():
    # 16 requests x the 16-node top-4 tree, 32 query heads over 8 KV heads, d = 128;
    # contexts of 0..1100 positions (ragged last tiles), planted large scores
    b = workloads.make_config(2)
    ctx = np.random.default_rng(1).integers(0, 1100, b.B)
    ctx[0], ctx[1], ctx[2] = 0, 128, 129
    check(b, 32, 8, 128, ctx, seed=2, P=1152, spike=8.0)


@pytest.mark.parametrize("workspace", [True, False])
def test_split_context_small_batch(workspace):
    # two units: the context is split over many CTAs when a workspace is given
    b = workloads.random_batch(np.random.default_rng(3), [11, 40], 1, 16, 16, depth_cap=6,
                               max_depth=8)
    _, wsb = check(b, 8, 1, 128, [3000, 1333], seed=4, P=3072, spike=6.0, workspace=workspace)
    assert wsb > 0


@pytest.mark.parametrize("H,Hkv,d", [(4, 4, 64), (16, 1, 64), (32, 2, 128), (8, 8, 128)])
def test_head_groupings_and_widths(H, Hkv, d):
    b = workloads.random_batch(np.random.default_rng(H + d), [0, 9, 33, 1, 64], 1, 16, 16,
                               depth_cap=10, max_depth=16)
    check(b, H, Hkv, d, [50, 0, 700, 128, 257], seed=H * d, spike=4.0)


def test_256_node_trees():
    # two tree tiles per request, eight M tiles of 128 query rows
    b = workloads.random_batch(np.random.default_rng(5), [256, 130], 1, 16, 16, depth_cap=16,
                               max_depth=16)
    check(b, 4, 1, 128, [400, 0], seed=6)


def test_cache_tail_holds_nan():
    b = workloads.random_batch(np.random.default_rng(7), [5, 17, 2], 1, 16, 16, depth_cap=6,
                               max_depth=8)
    check(b, 8, 2, 128, [77, 300, 1], seed=8, P=512, tail_nan=True)


def test_bench_workload_sampled():
    # the benchmarked shape: 16 requests, 4096-position contexts
    b = workloads.make_config(2)
    check(b, 32, 8, 128, [4096] * b.B, seed=9, P=4096)


def test_malformed_parent_and_context_length():
    import tree_speculative_verify_tv_gb300 as tv
    b = workloads.random_batch(np.random.default_rng(9), [4, 6], 1, 16, 16, depth_cap=4,
                               max_depth=4)
    a = workloads.attention_inputs(b, 4, 2, 64, [10, 20], P=64, seed=10)
    par = b.parent.copy()
    par[b.node_offsets[1] + 2] = 5  # a parent after its child
    st, got, _ = run(b, a, 4, 2, 64, 64, parent=par)
    assert st == tv.TV_ERR_TREE
    s = int(b.node_offsets[1])
    assert np.all(got[s:] == 0)
    ref = reference(b, a)
    assert row_errors(got[:s], ref[:s]).max() < TOL
    st, got, _ = run(b, a, 4, 2, 64, 64, ctx=np.array([10, 65], np.int32))
    assert st == tv.TV_ERR_SHAPE
    assert np.all(got[s:] == 0)
