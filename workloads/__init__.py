"""Seeded synthetic inputs for tree verification through a gated linear recurrence.

This module only *builds inputs*: draft trees, token ids, per-node factors
(q, k, v, g) and the committed context state H0.  It holds none of the
verification arithmetic (no recurrence, no acceptance walk, no commit); both the
fp64 oracle and the CUDA library consume what it returns.

Workload shapes follow the five benchmark configurations of the Bole
tree-speculation study (summary page "Bole: hybrid-attention tree speculation",
sections "Tree-Structured Closed Form" and "Evaluation"), and the best-first
tree construction of BASTION (summary page "BASTION", Method §1 path score
rho(i) = prod_k q_k(x_ik) and §2 best-first expansion).  All draws use
``numpy.random.default_rng(seed)``; the default seed of configuration c is
1000 + c.

Encodings
---------
* bf16 tensors are stored as ``uint16`` bit patterns (round-to-nearest-even
  of the float32 draw); :func:`bf16_bits_to_f32` widens them exactly.
* Trees are packed per request: ``node_offsets[B+1]`` (int32), ``parent[T]``
  local to the request (-1 = child of the committed context), ``depth[T]``
  (1 for a child of the context).  Parents precede children.
"""
from __future__ import annotations

import dataclasses
import heapq
from typing import List, Optional, Sequence

import numpy as np

# ---------------------------------------------------------------- encodings


def f32_to_bf16_bits(x: np.ndarray) -> np.ndarray:
    """Round float32 values to bfloat16 (nearest, ties to even); return the bits.
    A NaN stays a NaN (quiet, same sign)."""
    x = np.ascontiguousarray(x, dtype=np.float32)
    u = x.view(np.uint32)
    lsb = (u >> np.uint32(16)) & np.uint32(1)
    with np.errstate(over="ignore"):
        r = ((u + np.uint32(0x7FFF) + lsb) >> np.uint32(16)).astype(np.uint16)
    nan = np.isnan(x)
    if nan.any():
        r[nan] = ((u[nan] >> np.uint32(16)) | np.uint32(0x0040)).astype(np.uint16)
    return r


def bf16_bits_to_f32(b: np.ndarray) -> np.ndarray:
    """Widen bfloat16 bit patterns to float32 (exact)."""
    b = np.ascontiguousarray(b, dtype=np.uint16)
    return (b.astype(np.uint32) << np.uint32(16)).view(np.float32)


def softplus(x: np.ndarray) -> np.ndarray:
    return np.logaddexp(0.0, x)


def logsigmoid(x: np.ndarray) -> np.ndarray:
    return -np.logaddexp(0.0, -x)


# ---------------------------------------------------------------- container


@dataclasses.dataclass
class Batch:
    """One verification batch: B requests, each with its own draft tree, H heads."""

    B: int
    H: int
    dk: int
    dv: int
    decay: str            # "scalar" (g: [T,H]) or "diag" (g: [T,H,dk])
    qkv_dtype: str        # "bf16" (uint16 bits) or "f32"
    node_offsets: np.ndarray  # int32 [B+1]
    parent: np.ndarray        # int32 [T]
    depth: np.ndarray         # int32 [T]
    q: np.ndarray             # [T,H,dk]
    k: np.ndarray             # [T,H,dk]
    v: np.ndarray             # [T,H,dv]
    g: np.ndarray             # float32 [T,H] or [T,H,dk]
    H0: np.ndarray            # float32 [B,H,dk,dv]
    draft: np.ndarray         # int32 [T]   draft token of each node
    target: np.ndarray        # int32 [T]   target argmax after each node
    root_argmax: np.ndarray   # int32 [B]   target argmax at the committed context
    max_nodes: int
    max_depth: int
    name: str = ""

    @property
    def T(self) -> int:
        return int(self.node_offsets[-1])

    def sizes(self) -> np.ndarray:
        return np.diff(self.node_offsets)

    def qkv_f32(self, a: np.ndarray) -> np.ndarray:
        """Exact float32 view of a q/k/v array (bf16 bits widened)."""
        if self.qkv_dtype == "bf16":
            return bf16_bits_to_f32(a)
        return np.ascontiguousarray(a, dtype=np.float32)

    def node_heads(self) -> int:
        return self.T * self.H


# ---------------------------------------------------------------- trees


def depths_from_parents(parent: Sequence[int]) -> np.ndarray:
    """Depth of each node (1 for a child of the context); parents precede children."""
    d = np.zeros(len(parent), dtype=np.int32)
    for i, p in enumerate(parent):
        d[i] = 1 if p < 0 else d[p] + 1
    return d


def tree_random_recursive(rng, n: int) -> np.ndarray:
    """parent[0] = -1, parent[i] ~ U[0, i) for i > 0."""
    par = np.empty(n, dtype=np.int32)
    if n == 0:
        return par
    par[0] = -1
    for i in range(1, n):
        par[i] = rng.integers(0, i)
    return par


def tree_random_capped(rng, n: int, depth_cap: int) -> np.ndarray:
    """parent[0] = -1, parent[i] uniform over earlier nodes whose depth is below the cap."""
    par = np.empty(n, dtype=np.int32)
    dep = np.empty(n, dtype=np.int32)
    if n == 0:
        return par
    par[0], dep[0] = -1, 1
    for i in range(1, n):
        ok = np.nonzero(dep[:i] < depth_cap)[0]
        j = int(ok[rng.integers(0, len(ok))])
        par[i], dep[i] = j, dep[j] + 1
    return par


def tree_topk_chains(width: int, chain_len: int) -> np.ndarray:
    """`width` roots, each continued by a chain: nodes numbered level by level."""
    n = width * chain_len
    par = np.empty(n, dtype=np.int32)
    for i in range(n):
        par[i] = -1 if i < width else i - width
    return par


def tree_best_first(marginals: np.ndarray, n: int, depth_cap: int):
    """Best-first prefix tree from position-wise marginals (BASTION Method §1–§2).

    marginals: [depth_cap, C] draft distributions q_k over C candidates.
    Each node i at depth d carries the path score rho(i) = prod_{k<=d} q_k(x_ik).
    Repeatedly insert the frontier node with the largest rho (ties by push
    order); node index = insertion order, so parents precede children.
    Returns (parent[n], token[n], rho[n]).
    """
    C = marginals.shape[1]
    heap = []
    push = 0
    for x in range(C):
        heapq.heappush(heap, (-float(marginals[0, x]), push, -1, 1, x))
        push += 1
    parent, token, rho, depth = [], [], [], []
    while len(parent) < n and heap:
        negr, _, p, d, x = heapq.heappop(heap)
        idx = len(parent)
        parent.append(p)
        token.append(x)
        rho.append(-negr)
        depth.append(d)
        if d < depth_cap:
            for y in range(C):
                heapq.heappush(heap, (negr * float(marginals[d, y]), push, idx, d + 1, y))
                push += 1
    return (np.array(parent, dtype=np.int32), np.array(token, dtype=np.int32),
            np.array(rho, dtype=np.float64))


# ---------------------------------------------------------------- assembly


def _normal_scaled(rng, shape, std) -> np.ndarray:
    return (rng.standard_normal(shape, dtype=np.float32) * np.float32(std)).astype(np.float32)


def assemble(rng, parents: List[np.ndarray], H: int, dk: int, dv: int, *, decay: str,
             qkv_dtype: str, g_kind: str, h0_std: float, draft=None, target=None,
             root_argmax=None, vocab: int = 32, max_depth: Optional[int] = None,
             max_nodes: Optional[int] = None, name: str = "", values: bool = True) -> Batch:
    """Pack per-request trees and draw the per-node factors.

    values=False skips the factors and the state (q, k, v, g, H0 come back as empty
    arrays of the right dtype): the trees and tokens only, for a caller that fills
    the factors itself (the benchmark's timing of large configurations).

    g_kind: "softplus01"  g = -softplus(N(0,1))          (scalar decay, c1)
            "softplus_m1" g = -softplus(N(-1, 0.5))      (scalar decay, c2/c4)
            "logsig16"    g = logsigmoid(N(2,1)) / 16    (diagonal decay, c3/c5)
            "zero"        g = 0
    """
    B = len(parents)
    sizes = np.array([len(p) for p in parents], dtype=np.int64)
    offs = np.zeros(B + 1, dtype=np.int32)
    offs[1:] = np.cumsum(sizes)
    T = int(offs[-1])
    parent = np.concatenate(parents).astype(np.int32) if T else np.zeros(0, np.int32)
    depth = (np.concatenate([depths_from_parents(p) for p in parents]).astype(np.int32)
             if T else np.zeros(0, np.int32))
    if not values:
        e16 = np.zeros(0, np.uint16 if qkv_dtype == "bf16" else np.float32)
        return Batch(B=B, H=H, dk=dk, dv=dv, decay=decay, qkv_dtype=qkv_dtype,
                     node_offsets=offs, parent=parent, depth=depth, q=e16, k=e16, v=e16,
                     g=np.zeros(0, np.float32), H0=np.zeros(0, np.float32),
                     draft=np.zeros(T, np.int32) if draft is None else np.asarray(draft, np.int32),
                     target=np.zeros(T, np.int32) if target is None else np.asarray(target, np.int32),
                     root_argmax=(np.zeros(B, np.int32) if root_argmax is None
                                  else np.asarray(root_argmax, np.int32)),
                     max_nodes=int(max_nodes if max_nodes is not None
                                   else max(1, int(sizes.max()) if B else 1)),
                     max_depth=int(max_depth if max_depth is not None
                                   else (int(depth.max()) if T else 1)), name=name)
    sc = 1.0 / np.sqrt(dk)
    q = _normal_scaled(rng, (T, H, dk), sc)
    k = _normal_scaled(rng, (T, H, dk), sc)
    v = _normal_scaled(rng, (T, H, dv), sc)
    gshape = (T, H) if decay == "scalar" else (T, H, dk)
    if g_kind == "softplus01":
        g = -softplus(rng.standard_normal(gshape))
    elif g_kind == "softplus_m1":
        g = -softplus(rng.normal(-1.0, 0.5, gshape))
    elif g_kind == "logsig16":
        g = logsigmoid(rng.normal(2.0, 1.0, gshape)) / 16.0
    elif g_kind == "zero":
        g = np.zeros(gshape)
    else:
        raise ValueError(g_kind)
    g = g.astype(np.float32)
    H0 = _normal_scaled(rng, (B, H, dk, dv), h0_std)
    if qkv_dtype == "bf16":
        q, k, v = f32_to_bf16_bits(q), f32_to_bf16_bits(k), f32_to_bf16_bits(v)
    if draft is None:
        draft = rng.integers(0, vocab, T).astype(np.int32)
    if target is None:
        target = rng.integers(0, vocab, T).astype(np.int32)
    if root_argmax is None:
        root_argmax = rng.integers(0, vocab, B).astype(np.int32)
    md = int(depth.max()) if T else 1
    return Batch(B=B, H=H, dk=dk, dv=dv, decay=decay, qkv_dtype=qkv_dtype,
                 node_offsets=offs, parent=parent, depth=depth, q=q, k=k, v=v, g=g,
                 H0=H0, draft=np.asarray(draft, np.int32), target=np.asarray(target, np.int32),
                 root_argmax=np.asarray(root_argmax, np.int32),
                 max_nodes=int(max_nodes if max_nodes is not None else max(1, int(sizes.max()) if B else 1)),
                 max_depth=int(max_depth if max_depth is not None else md), name=name)


# ---------------------------------------------------------------- configs


def _plant_path(rng, parent: np.ndarray, draft: np.ndarray, target: np.ndarray,
                path: Sequence[int], no_match_token: int):
    """Set target tokens so that the greedy walk follows `path` and stops after it.

    Root token = draft of the path's first node (or a non-matching token when the
    path is empty); each path node's target = draft of the next path node; the
    last node's target is a token no child of it carries.  Returns root token.
    """
    n = len(parent)
    children = [[] for _ in range(n + 1)]  # slot n = virtual root
    for i in range(n):
        children[n if parent[i] < 0 else parent[i]].append(i)
    if len(path) == 0:
        used = {int(draft[c]) for c in children[n]}
        tok = no_match_token
        while tok in used:
            tok += 1
        return tok
    root_tok = int(draft[path[0]])
    for a, b in zip(path[:-1], path[1:]):
        target[a] = draft[b]
    last = path[-1]
    used = {int(draft[c]) for c in children[last]}
    tok = no_match_token
    while tok in used:
        tok += 1
    target[last] = tok
    return root_tok


def config1(seed: Optional[int] = None, values: bool = True) -> Batch:
    """c1: one request, one head, dk=dv=16, fp32 q/k/v, random recursive 8-node tree."""
    rng = np.random.default_rng(1001 if seed is None else seed)
    par = tree_random_recursive(rng, 8)
    return assemble(rng, [par], 1, 16, 16, decay="scalar", qkv_dtype="f32",
                    g_kind="softplus01", h0_std=0.1, vocab=32, max_depth=8, name="c1",
                    values=values)


def config2(seed: Optional[int] = None, B: int = 16, H: int = 24, values: bool = True) -> Batch:
    """c2: Mamba-2-like layer.  B=16, H=24, dk=128, dv=64, bf16, scalar decay.

    Fixed top-k tree: 4 children of the context, each continued by a chain of
    3 more nodes (16 nodes, BFS numbering).  Vocabulary 32000; depth-1 drafts
    are distinct; a planted path of length L ~ U{0..4} along one chain.
    """
    rng = np.random.default_rng(1002 if seed is None else seed)
    par = tree_topk_chains(4, 4)
    n = len(par)
    parents, drafts, targets, roots = [], [], [], []
    for _ in range(B):
        d = rng.integers(0, 32000, n).astype(np.int32)
        d[:4] = rng.choice(32000, 4, replace=False)
        t = rng.integers(0, 32000, n).astype(np.int32)
        chain = int(rng.integers(0, 4))
        L = int(rng.integers(0, 5))
        path = [chain + 4 * m for m in range(L)]
        roots.append(_plant_path(rng, par, d, t, path, no_match_token=int(rng.integers(0, 32000))))
        parents.append(par)
        drafts.append(d)
        targets.append(t)
    return assemble(rng, parents, H, 128, 64, decay="scalar", qkv_dtype="bf16",
                    g_kind="softplus_m1", h0_std=0.05, draft=np.concatenate(drafts),
                    target=np.concatenate(targets), root_argmax=np.array(roots), max_depth=4,
                    name="c2", values=values)


def _best_first_requests(rng, B: int, n: int, depth_cap: int, alpha: float, C: int = 8):
    """Per request: Dirichlet marginals, best-first tree, draft = candidate id,
    target continuation t_k ~ q_k; target argmax t_{d+1} on the matching path and
    U[0,C) off it; root argmax t_1.  Returns parents, drafts, targets, roots, rho sums."""
    parents, drafts, targets, roots, rhos = [], [], [], [], []
    for _ in range(B):
        marg = rng.dirichlet(alpha * np.ones(C), size=depth_cap)
        par, tok, rho = tree_best_first(marg, n, depth_cap)
        cont = np.array([rng.choice(C, p=marg[kk]) for kk in range(depth_cap)]
                        + [rng.integers(0, C)], dtype=np.int32)
        dep = depths_from_parents(par)
        on = np.zeros(len(par), dtype=bool)
        for i in range(len(par)):
            up = on[par[i]] if par[i] >= 0 else True
            on[i] = up and tok[i] == cont[dep[i] - 1]
        tgt = rng.integers(0, C, len(par)).astype(np.int32)
        tgt[on] = cont[dep[on]]
        parents.append(par)
        drafts.append(tok)
        targets.append(tgt)
        roots.append(int(cont[0]))
        rhos.append(float(rho.sum()))
    return parents, drafts, targets, roots, rhos


def config3(seed: Optional[int] = None, B: int = 32, H: int = 16, values: bool = True) -> Batch:
    """c3: GLA-like layer, diagonal decay.  B=32, H=16, dk=dv=128, bf16; best-first
    64-node trees of depth <= 8 from Dirichlet(0.3) marginals over 8 candidates."""
    rng = np.random.default_rng(1003 if seed is None else seed)
    parents, drafts, targets, roots, rhos = _best_first_requests(rng, B, 64, 8, 0.3)
    b = assemble(rng, parents, H, 128, 128, decay="diag", qkv_dtype="bf16", g_kind="logsig16",
                 h0_std=0.05, draft=np.concatenate(drafts), target=np.concatenate(targets),
                 root_argmax=np.array(roots), max_depth=8, name="c3", values=values)
    b.rho_sums = rhos  # type: ignore[attr-defined]
    return b


def config4(seed: Optional[int] = None, B: int = 128, H: int = 32, values: bool = True) -> Batch:
    """c4: mixed-budget batch.  B=128, H=32, dk=dv=128, bf16, scalar decay; tree
    sizes ~ U{4,8,16,32,64,128}; random parents with depth cap 12."""
    rng = np.random.default_rng(1004 if seed is None else seed)
    sizes = rng.choice([4, 8, 16, 32, 64, 128], B)
    parents = [tree_random_capped(rng, int(n), 12) for n in sizes]
    return assemble(rng, parents, H, 128, 128, decay="scalar", qkv_dtype="bf16",
                    g_kind="softplus_m1", h0_std=0.05, vocab=32, max_depth=12,
                    max_nodes=128, name="c4", values=values)


def config5(seed: Optional[int] = None, B: int = 8, layers: int = 36, heads: int = 32,
            values: bool = True) -> Batch:
    """c5: large-tree stack.  B=8, 36 layers x 32 heads folded into H=1152,
    dk=dv=128, bf16, diagonal decay; best-first 256-node trees of depth <= 16 from
    Dirichlet(0.2) marginals; one planted accepted path per request to a uniform
    random node (shared by every layer and head of the request)."""
    rng = np.random.default_rng(1005 if seed is None else seed)
    parents, drafts, _, _, _ = _best_first_requests(rng, B, 256, 16, 0.2)
    targets, roots = [], []
    for b in range(B):
        par, d = parents[b], drafts[b]
        t = rng.integers(0, 8, len(par)).astype(np.int32)
        u = int(rng.integers(0, len(par)))
        path = []
        j = u
        while j >= 0:
            path.append(j)
            j = int(par[j])
        path.reverse()
        roots.append(_plant_path(rng, par, d, t, path, no_match_token=8))
        targets.append(t)
    return assemble(rng, parents, layers * heads, 128, 128, decay="diag", qkv_dtype="bf16",
                    g_kind="logsig16", h0_std=0.05, draft=np.concatenate(drafts),
                    target=np.concatenate(targets), root_argmax=np.array(roots),
                    max_depth=16, name="c5", values=values)


CONFIGS = {1: config1, 2: config2, 3: config3, 4: config4, 5: config5}


def make_config(c: int, seed: Optional[int] = None, **kw) -> Batch:
    return CONFIGS[c](seed, **kw)


def target_logits(batch: Batch, vocab: int, seed: Optional[int] = None, *,
                  levels: Optional[int] = None):
    """bf16 target logits for the greedy walk (uint16 bits): root_logits [B][vocab]
    at the committed context and node_logits [T][vocab] after each node.

    Default: values N(0, 2) with the row's target token (batch.root_argmax /
    batch.target) set 1 above the row's largest other value, so the argmax of each
    row is that token and the planted acceptance paths are reproduced.
    levels=k: values drawn from k equally spaced levels (many ties, targets not
    planted), for exercising the first-index rule."""
    rng = np.random.default_rng(0 if seed is None else seed)
    rows = batch.B + batch.T

    def draw(n):
        if levels:
            return rng.integers(0, levels, (n, vocab)).astype(np.float32) * np.float32(0.5)
        return rng.normal(0.0, 2.0, (n, vocab)).astype(np.float32)

    x = draw(rows)
    if not levels:
        tok = np.concatenate([batch.root_argmax, batch.target]).astype(np.int64)
        if rows and int(tok.max()) >= vocab:
            raise ValueError("a target token is outside the vocabulary")
        r = np.arange(rows)
        x[r, tok] = -np.inf
        x[r, tok] = np.max(x, axis=1) + np.float32(1.0)
    bits = f32_to_bf16_bits(x)
    return bits[:batch.B], bits[batch.B:]


def stochastic_inputs(batch: Batch, vocab: int, seed: Optional[int] = None,
                      spread: float = 2.0, draft_noise: float = 1.0):
    """Inputs of the stochastic acceptance rule for `batch`'s trees: target and draft
    probability rows (float32) at the context (root_p, root_q [B][vocab]) and after
    every node (node_p, node_q [T][vocab]), draft tokens drawn from the parent's
    draft row, uniforms for every acceptance test (u_accept [T]) and every bonus
    draw (u_bonus [B]), both float64 in [0, 1).  Target logits are N(0, spread);
    draft logits add N(0, draft_noise) to them.  Returns a dict; the batch's own
    draft tokens are left unchanged (the dict carries the new ones)."""
    rng = np.random.default_rng(0 if seed is None else seed)
    rows = batch.B + batch.T

    def softmax(z):
        z = z - z.max(axis=1, keepdims=True)
        e = np.exp(z)
        return e / e.sum(axis=1, keepdims=True)

    zt = rng.normal(0.0, spread, (rows, vocab))
    pt = softmax(zt).astype(np.float32)
    pq = softmax(zt + rng.normal(0.0, draft_noise, (rows, vocab))).astype(np.float32)
    draft = np.zeros(batch.T, np.int32)
    for r in range(batch.B):
        s, e = int(batch.node_offsets[r]), int(batch.node_offsets[r + 1])
        for i in range(s, e):
            p = int(batch.parent[i])
            row = pq[r] if p < 0 else pq[batch.B + s + p]
            w = row.astype(np.float64)
            draft[i] = rng.choice(vocab, p=w / w.sum())
    return dict(root_p=pt[:batch.B], node_p=pt[batch.B:], root_q=pq[:batch.B],
                node_q=pq[batch.B:], draft=draft,
                u_accept=rng.random(batch.T), u_bonus=rng.random(batch.B))


def attention_inputs(batch: Batch, H: int, Hkv: int, d: int, ctx_len: Sequence[int],
                     P: Optional[int] = None, seed: Optional[int] = None, spike: float = 0.0,
                     tail_nan: bool = False, widen: bool = True):
    """Inputs of one attention layer over `batch`'s draft trees (its tree only; its
    linear-layer factors are not used): queries q [T][H][d], the shared-prefix KV
    cache k_cache, v_cache [B][Hkv][P][d] with ctx_len[b] valid positions, and the
    tree nodes' own keys and values k_tree, v_tree [T][Hkv][d].  Every value is
    N(0, 1) rounded to bf16 (uint16 bits; the "_f32" entries are the exact widened
    values), so scale * q.k with scale = 1/sqrt(d) is about N(0, 1).
    spike > 0: one cached key in 64 per (request, KV head) is replaced by
    spike * (the mean of the group's first query head over the request's nodes) /
    |that mean| * sqrt(d), giving scores of about +-spike that make the row maximum
    jump between key tiles.  tail_nan: cache positions at and beyond ctx_len hold
    NaN (they must not be read into the result).  widen=False leaves out the
    "_f32" entries."""
    rng = np.random.default_rng(0 if seed is None else seed)
    B, T = batch.B, batch.T
    ctx = np.asarray(ctx_len, dtype=np.int32).reshape(B)
    P = int(max(1, ctx.max() if B else 1)) if P is None else int(P)
    if B and int(ctx.max()) > P:
        raise ValueError("ctx_len exceeds the cache capacity P")
    draw = lambda shape: rng.standard_normal(shape, dtype=np.float32)
    q = draw((T, H, d))
    kc = draw((B, Hkv, P, d))
    vc = draw((B, Hkv, P, d))
    kt = draw((T, Hkv, d))
    vt = draw((T, Hkv, d))
    grp = H // Hkv
    if spike > 0:
        for b in range(B):
            s, e = int(batch.node_offsets[b]), int(batch.node_offsets[b + 1])
            if e == s or ctx[b] == 0:
                continue
            for kv in range(Hkv):
                m = q[s:e, kv * grp].astype(np.float64).mean(axis=0)
                m = m / max(np.linalg.norm(m), 1e-30) * np.sqrt(d) * spike
                pos = rng.choice(int(ctx[b]), size=max(1, int(ctx[b]) // 64), replace=False)
                sign = np.where(rng.random(len(pos)) < 0.5, -1.0, 1.0)
                kc[b, kv, pos] = (sign[:, None] * m[None, :]).astype(np.float32)
    if tail_nan:
        for b in range(B):
            kc[b, :, int(ctx[b]):] = np.nan
            vc[b, :, int(ctx[b]):] = np.nan
    out = dict(ctx_len=ctx, scale=float(1.0 / np.sqrt(d)))
    for name, a in (("q", q), ("k_cache", kc), ("v_cache", vc), ("k_tree", kt), ("v_tree", vt)):
        bits = f32_to_bf16_bits(a)
        out[name] = bits
        if widen:
            out[name + "_f32"] = bf16_bits_to_f32(bits)
    return out


def random_batch(rng, sizes: Sequence[int], H: int, dk: int, dv: int, *, decay="scalar",
                 qkv_dtype="bf16", g_kind=None, depth_cap: int = 32, vocab: int = 4,
                 h0_std: float = 0.05, max_depth: Optional[int] = None,
                 max_nodes: Optional[int] = None) -> Batch:
    """Ragged batch with random capped trees, for parity sweeps over shapes."""
    parents = [tree_random_capped(rng, int(n), depth_cap) for n in sizes]
    if g_kind is None:
        g_kind = "softplus_m1" if decay == "scalar" else "logsig16"
    return assemble(rng, parents, H, dk, dv, decay=decay, qkv_dtype=qkv_dtype, g_kind=g_kind,
                    h0_std=h0_std, vocab=vocab, max_depth=max_depth, max_nodes=max_nodes,
                    name="random")
