"""Pins of the oracle's tree-masked softmax attention (oracle.tree_attention) to
results fixed by something other than its own code: PyTorch's
scaled_dot_product_attention on the flattened root path of each node (CPU, fp64),
causal attention for a chain, closed forms for a zero scale, constant values and a
context-free root node.  The page passages are cited in the oracle."""
import numpy as np
import pytest

import oracle
import workloads

torch = pytest.importorskip("torch")
F = torch.nn.functional


def inputs(sizes, H, Hkv, d, ctx, seed, spike=0.0, P=None):
    rng = np.random.default_rng(seed)
    b = workloads.random_batch(rng, sizes, 1, 16, 16, depth_cap=6, max_depth=8)
    a = workloads.attention_inputs(b, H, Hkv, d, ctx, P=P, seed=seed + 1, spike=spike)
    return b, a


def run_oracle(b, a, scale=None):
    return oracle.tree_attention(b.node_offsets, b.parent, a["q_f32"], a["k_cache_f32"],
                                 a["v_cache_f32"], a["ctx_len"], a["k_tree_f32"],
                                 a["v_tree_f32"], a["scale"] if scale is None else scale)


def root_path(parent, s, i):
    """Request-local node indices from the child of the context down to i."""
    path = []
    while i >= 0:
        path.append(i)
        i = int(parent[s + i])
    return path[::-1]


@pytest.mark.parametrize("sizes,H,Hkv,d,ctx,spike", [
    ([5, 1, 9], 4, 2, 16, [7, 0, 12], 0.0),
    ([12, 3], 8, 2, 32, [40, 5], 6.0),
    ([16], 6, 6, 8, [3], 0.0),
])
def test_each_node_equals_attention_over_its_flattened_path(sizes, H, Hkv, d, ctx, spike):
    # node i's output is plain (unmasked) attention of its query over the context
    # followed by its own root path
    b, a = inputs(sizes, H, Hkv, d, ctx, seed=sum(sizes) + H, spike=spike)
    out = run_oracle(b, a)
    grp = H // Hkv
    for r in range(b.B):
        s, e = int(b.node_offsets[r]), int(b.node_offsets[r + 1])
        L = int(a["ctx_len"][r])
        for i in range(e - s):
            path = [s + j for j in root_path(b.parent, s, i)]
            for h in range(H):
                kvh = h // grp
                K = np.concatenate([a["k_cache_f32"][r, kvh, :L], a["k_tree_f32"][path, kvh]])
                V = np.concatenate([a["v_cache_f32"][r, kvh, :L], a["v_tree_f32"][path, kvh]])
                qt = torch.from_numpy(a["q_f32"][s + i, h].astype(np.float64))[None, None, None]
                kt = torch.from_numpy(K.astype(np.float64))[None, None]
                vt = torch.from_numpy(V.astype(np.float64))[None, None]
                ref = F.scaled_dot_product_attention(qt, kt, vt, scale=a["scale"])[0, 0, 0]
                np.testing.assert_allclose(out[s + i, h], ref.numpy(), rtol=1e-12, atol=1e-13)


def test_chain_is_causal_attention_over_prefix_and_chain():
    n, L, H, d = 10, 23, 2, 16
    b = workloads.random_batch(np.random.default_rng(3), [n], 1, 16, 16, depth_cap=n,
                               max_depth=n)
    b.parent[:] = np.arange(-1, n - 1, dtype=np.int32)
    a = workloads.attention_inputs(b, H, H, d, [L], seed=4)
    out = run_oracle(b, a)
    for h in range(H):
        K = np.concatenate([a["k_cache_f32"][0, h, :L], a["k_tree_f32"][:, h]]).astype(np.float64)
        V = np.concatenate([a["v_cache_f32"][0, h, :L], a["v_tree_f32"][:, h]]).astype(np.float64)
        Q = np.zeros((L + n, d))
        Q[L:] = a["q_f32"][:, h]
        ref = F.scaled_dot_product_attention(torch.from_numpy(Q)[None, None],
                                             torch.from_numpy(K)[None, None],
                                             torch.from_numpy(V)[None, None], is_causal=True,
                                             scale=a["scale"])[0, 0]
        np.testing.assert_allclose(out[:, h], ref[L:].numpy(), rtol=1e-12, atol=1e-13)


def test_zero_scale_gives_the_mean_of_visible_values():
    b, a = inputs([7, 4], 4, 2, 8, [5, 0], seed=11)
    out = run_oracle(b, a, scale=0.0)
    for r in range(b.B):
        s, e = int(b.node_offsets[r]), int(b.node_offsets[r + 1])
        L = int(a["ctx_len"][r])
        for i in range(e - s):
            path = [s + j for j in root_path(b.parent, s, i)]
            for h in range(4):
                tot = a["v_cache_f32"][r, h // 2, :L].astype(np.float64).sum(axis=0) + \
                    a["v_tree_f32"][path, h // 2].astype(np.float64).sum(axis=0)
                np.testing.assert_allclose(out[s + i, h], tot / (L + len(path)), rtol=1e-12,
                                           atol=1e-14)


def test_constant_values_per_kv_head_come_back_unchanged():
    # every visible value of KV head c is the vector (c+1) * u: each query head gets
    # its own group's vector, whatever the scores
    b, a = inputs([6, 9], 8, 4, 16, [30, 2], seed=21, spike=4.0)
    u = np.linspace(-1, 1, 16).astype(np.float32)
    for c in range(4):
        a["v_cache_f32"][:, c] = (c + 1) * u
        a["v_tree_f32"][:, c] = (c + 1) * u
    out = run_oracle(b, a)
    for h in range(8):
        want = ((h // 2 + 1) * u).astype(np.float32).astype(np.float64)
        np.testing.assert_allclose(out[:, h], np.broadcast_to(want, out[:, h].shape),
                                   rtol=1e-12, atol=1e-13)


def test_root_node_without_context_returns_its_own_value():
    b, a = inputs([5], 2, 1, 8, [0], seed=31)
    out = run_oracle(b, a)
    for i in range(5):
        if b.parent[i] == -1:
            for h in range(2):
                np.testing.assert_allclose(out[i, h], a["v_tree_f32"][i, 0], rtol=0, atol=1e-15)


def test_large_scores_do_not_overflow():
    # scores of several hundred: the max subtraction keeps exp finite
    b, a = inputs([8], 2, 1, 16, [20], seed=41)
    out = run_oracle(b, a, scale=200.0)
    assert np.all(np.isfinite(out))
