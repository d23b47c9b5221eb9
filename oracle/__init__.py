"""fp64 CPU oracle for tree verification -- TEST INFRASTRUCTURE ONLY.

Only the tests, ``__graft_entry__.smoke()`` and the benchmark's CPU-baseline
leg import this package.  The CUDA library never calls it and it never calls
the CUDA library; the two share only the seeded input generators
(``workloads``).

The arithmetic lives in ``oracle.c`` (plain C, double precision): the naive
serial tree walk that materialises one state matrix per draft node (Bole
summary page, "Core techniques" §1-§2 and the naive baseline it compares
against), the greedy acceptance walk (LLM Primer VI ch. 9, §9.1) and the
commit of the accepted path's state (Bole §2).  This file builds the C source,
marshals arrays and splits work over threads; the functions for the wider rows
of the path are plain numpy here: the argmax of logits rows, best-first tree
construction, stochastic acceptance and tree-masked softmax attention.

Parity pins for each function are in ``tests/test_oracle_pins.py``.
"""
from __future__ import annotations

import ctypes
import heapq
import os
import subprocess
import threading
from concurrent.futures import ThreadPoolExecutor
from typing import Optional, Sequence

import numpy as np

_HERE = os.path.dirname(os.path.abspath(__file__))
_SRC = os.path.join(_HERE, "oracle.c")
_LIB = os.path.join(_HERE, "liboracle.so")
_lock = threading.Lock()
_lib = None

_I32P = np.ctypeslib.ndpointer(dtype=np.int32, flags="C_CONTIGUOUS")
_F32P = np.ctypeslib.ndpointer(dtype=np.float32, flags="C_CONTIGUOUS")
_F64P = np.ctypeslib.ndpointer(dtype=np.float64, flags="C_CONTIGUOUS")


def build(force: bool = False) -> str:
    """Compile oracle.c into liboracle.so (gcc, -O2, no fast-math)."""
    if force or not os.path.exists(_LIB) or os.path.getmtime(_LIB) < os.path.getmtime(_SRC):
        tmp = _LIB + ".%d.tmp" % os.getpid()
        subprocess.check_call(["gcc", "-O2", "-std=c99", "-fPIC", "-shared", "-fno-fast-math",
                               "-ffp-contract=off", "-o", tmp, _SRC, "-lm"])
        os.replace(tmp, _LIB)
    return _LIB


def load(path: str):
    """Load a compiled oracle library (the default build, or a test's variant)."""
    L = ctypes.CDLL(path)
    i = ctypes.c_int
    L.orc_check_tree.argtypes = [i, _I32P]
    L.orc_verify_unit.argtypes = [i, _I32P, i, i, i, _F64P, _F64P, _F64P, _F64P, _F64P,
                                  _F64P, ctypes.c_void_p]
    L.orc_accept.argtypes = [i, _I32P, _I32P, _I32P, ctypes.c_int32, i, _I32P, _I32P,
                             _I32P]
    L.orc_commit_unit.argtypes = [i, _I32P, i, i, i, _F64P, _F64P, _F64P, _F64P, _F64P]
    L.orc_verify_batch.argtypes = [i, i, i, i, i, _I32P, _I32P, _F32P, _F32P, _F32P,
                                   _F32P, _F32P, i, _I32P, _F64P]
    L.orc_accept_batch.argtypes = [i, _I32P, _I32P, _I32P, _I32P, _I32P, i, _I32P, _I32P,
                                   _I32P]
    L.orc_commit_batch.argtypes = [i, i, i, i, i, _I32P, _F32P, _F32P, _F32P, _F32P,
                                   _I32P, _I32P, i, i, _I32P, _F64P]
    for f in (L.orc_check_tree, L.orc_verify_unit, L.orc_accept, L.orc_commit_unit,
              L.orc_verify_batch, L.orc_accept_batch, L.orc_commit_batch):
        f.restype = ctypes.c_int
    return L


def lib():
    global _lib
    with _lock:
        if _lib is None:
            _lib = load(build())
    return _lib


_override = threading.local()


def _L():
    return getattr(_override, "lib", None) or lib()


class using:
    """Context manager: route this thread's oracle calls to another build."""

    def __init__(self, L):
        self.L = L

    def __enter__(self):
        self.prev = getattr(_override, "lib", None)
        _override.lib = self.L

    def __exit__(self, *a):
        _override.lib = self.prev


class OracleError(RuntimeError):
    pass


def _rc(rc: int, what: str):
    if rc != 0:
        raise OracleError("%s failed with code %d" % (what, rc))


def _f64(a) -> np.ndarray:
    return np.ascontiguousarray(a, dtype=np.float64)


# ------------------------------------------------------------------ unit level


def verify_unit(parent, q, k, v, g, H0, *, diag: bool, return_states: bool = False):
    """Naive serial walk for one (request, head).  q,k: [n,dk]; v: [n,dv];
    g: [n] or [n,dk]; H0: [dk,dv].  Returns out [n,dv] (and states [n,dk,dv])."""
    parent = np.ascontiguousarray(parent, dtype=np.int32)
    n = len(parent)
    q, k, v, g, H0 = _f64(q), _f64(k), _f64(v), _f64(g), _f64(H0)
    dk, dv = H0.shape
    out = np.zeros((n, dv), dtype=np.float64)
    states = np.zeros((max(n, 1), dk, dv), dtype=np.float64)
    _rc(_L().orc_verify_unit(n, parent, dk, dv, int(diag), g.reshape(-1) if n else np.zeros(1),
                              q.reshape(-1) if n else np.zeros(1),
                              k.reshape(-1) if n else np.zeros(1),
                              v.reshape(-1) if n else np.zeros(1), H0.reshape(-1),
                              out.reshape(-1) if n else np.zeros(1),
                              states.ctypes.data_as(ctypes.c_void_p)), "verify_unit")
    return (out, states[:n]) if return_states else out


def accept(parent, draft, target, root_tok: int, max_depth: int):
    """Greedy walk for one request: returns (len, path[max_depth], bonus)."""
    parent = np.ascontiguousarray(parent, dtype=np.int32)
    ln = np.zeros(1, np.int32)
    bonus = np.zeros(1, np.int32)
    path = np.zeros(max(max_depth, 1), np.int32)
    _rc(_L().orc_accept(len(parent), parent, np.ascontiguousarray(draft, np.int32),
                         np.ascontiguousarray(target, np.int32), int(root_tok), max_depth, ln,
                         path, bonus), "accept")
    return int(ln[0]), path[:max_depth], int(bonus[0])


def commit_unit(path, L: int, k, v, g, H0, *, diag: bool):
    """Replay the recurrence from H0 along path[:L]; returns H_new [dk,dv]."""
    H0 = _f64(H0)
    dk, dv = H0.shape
    out = np.zeros((dk, dv), np.float64)
    k, v, g = _f64(k), _f64(v), _f64(g)
    _rc(_L().orc_commit_unit(L, np.ascontiguousarray(path, np.int32), dk, dv, int(diag),
                              g.reshape(-1) if g.size else np.zeros(1),
                              k.reshape(-1) if k.size else np.zeros(1),
                              v.reshape(-1) if v.size else np.zeros(1), H0.reshape(-1),
                              out.reshape(-1)), "commit_unit")
    return out


# ------------------------------------------------------------------ batch level


class _Packed:
    """float32 views of a workloads.Batch, as the C batch drivers read them."""

    def __init__(self, batch):
        self.b = batch
        self.q = np.ascontiguousarray(batch.qkv_f32(batch.q)).reshape(-1)
        self.k = np.ascontiguousarray(batch.qkv_f32(batch.k)).reshape(-1)
        self.v = np.ascontiguousarray(batch.qkv_f32(batch.v)).reshape(-1)
        self.g = np.ascontiguousarray(batch.g, dtype=np.float32).reshape(-1)
        self.H0 = np.ascontiguousarray(batch.H0, dtype=np.float32).reshape(-1)
        self.offs = np.ascontiguousarray(batch.node_offsets, np.int32)
        self.parent = np.ascontiguousarray(batch.parent, np.int32)
        for name in ("q", "k", "v", "g", "parent"):
            a = getattr(self, name)
            if a.size == 0:
                setattr(self, name, np.zeros(1, a.dtype))


def _split(seq: np.ndarray, parts: int):
    parts = max(1, min(parts, len(seq)))
    return [s for s in np.array_split(seq, parts) if len(s)]


def verify(batch, units: Optional[Sequence[int]] = None, threads: int = 1, packed=None):
    """Outputs of the listed units (u = b*H + h; default all).

    Returns a dict u -> out [N_b, dv] (float64)."""
    b = batch
    P = packed or _Packed(b)
    if units is None:
        units = np.arange(b.B * b.H, dtype=np.int32)
    units = np.ascontiguousarray(units, dtype=np.int32)
    sizes = np.diff(b.node_offsets)
    res = {}

    def run(chunk):
        rows = int(sum(sizes[u // b.H] for u in chunk))
        out = np.zeros((max(rows, 1), b.dv), np.float64)
        _rc(_L().orc_verify_batch(b.B, b.H, b.dk, b.dv, int(b.decay == "diag"), P.offs,
                                   P.parent, P.g, P.q, P.k, P.v, P.H0, len(chunk),
                                   np.ascontiguousarray(chunk, np.int32), out.reshape(-1)),
            "verify_batch")
        r = 0
        part = {}
        for u in chunk:
            n = int(sizes[u // b.H])
            part[int(u)] = out[r:r + n]
            r += n
        return part

    chunks = _split(units, threads * 4)
    if threads <= 1 or len(chunks) == 1:
        for c in chunks:
            res.update(run(c))
    else:
        with ThreadPoolExecutor(threads) as ex:
            for part in ex.map(run, chunks):
                res.update(part)
    return res


def verify_dense(batch, threads: int = 1) -> np.ndarray:
    """All outputs as a packed [T,H,dv] float64 array."""
    res = verify(batch, threads=threads)
    out = np.zeros((batch.T, batch.H, batch.dv), np.float64)
    for u, o in res.items():
        bb, h = divmod(u, batch.H)
        s, e = batch.node_offsets[bb], batch.node_offsets[bb + 1]
        out[s:e, h, :] = o
    return out


def accept_batch(batch, max_depth: Optional[int] = None, root_argmax=None, target=None):
    """Greedy walk for every request: (len[B], path[B,max_depth], bonus[B])."""
    b = batch
    md = b.max_depth if max_depth is None else max_depth
    ln = np.zeros(max(b.B, 1), np.int32)
    bonus = np.zeros(max(b.B, 1), np.int32)
    path = np.zeros(max(b.B * md, 1), np.int32)
    root = np.ascontiguousarray(b.root_argmax if root_argmax is None else root_argmax, np.int32)
    tgt = np.ascontiguousarray(b.target if target is None else target, np.int32)
    par = np.ascontiguousarray(b.parent, np.int32)
    drf = np.ascontiguousarray(b.draft, np.int32)
    if par.size == 0:
        par, drf, tgt = np.zeros(1, np.int32), np.zeros(1, np.int32), np.zeros(1, np.int32)
    _rc(_L().orc_accept_batch(b.B, np.ascontiguousarray(b.node_offsets, np.int32), par, drf, tgt,
                               root if root.size else np.zeros(1, np.int32), md, ln, path, bonus),
        "accept_batch")
    return ln[:b.B], path[:b.B * md].reshape(b.B, md), bonus[:b.B]


def argmax_rows(bits) -> np.ndarray:
    """Target argmax of every row of bf16 logits (uint16 bit patterns, [rows][V]).

    The greedy rule takes the target's most likely token (LLM Primer VI ch. 9,
    §9.1).  Written as numpy's argmax over the exactly widened values: the first
    index among equal maxima; a NaN counts as larger than any number (the first
    NaN wins); -0 equals +0."""
    b = np.ascontiguousarray(bits, dtype=np.uint16)
    if b.ndim != 2 or b.shape[1] == 0:
        raise OracleError("argmax_rows needs a [rows][V] array with V >= 1")
    x = (b.astype(np.uint32) << np.uint32(16)).view(np.float32).astype(np.float64)
    return np.argmax(x, axis=1).astype(np.int32)


def accept_from_logits(batch, root_logits, node_logits, max_depth: Optional[int] = None):
    """Greedy walk with the target's choices taken as the argmax of its logits:
    root_logits [B][V] at the committed context, node_logits [T][V] after each
    node.  Returns (len[B], path[B,max_depth], bonus[B], root_argmax[B],
    target_argmax[T])."""
    root = argmax_rows(root_logits) if batch.B else np.zeros(0, np.int32)
    tgt = argmax_rows(node_logits) if batch.T else np.zeros(0, np.int32)
    ln, path, bonus = accept_batch(batch, max_depth=max_depth, root_argmax=root, target=tgt)
    return ln, path, bonus, root, tgt


def best_first(marginals, n: int, depth_cap: int, cost=None):
    """Draft tree of one request by best-first expansion (BASTION page, Method §1-§3).

    marginals [depth_cap][C]: the drafter's distribution q_k over C candidates at
    position k.  A node at depth d holding candidates x_1..x_d has path score
    rho = prod_k q_k(x_k).  The frontier starts as the C children of the context;
    the frontier node with the largest rho is added next (equal scores: the one that
    joined the frontier first; a node's C children join, in candidate order, when it
    is added and its depth is below depth_cap).  Node index = order of addition.
    cost (optional) [n+1]: the step cost C(N) with N nodes; the tree then stops
    growing once the estimated speed-up sum(rho) / C(N) would drop (§3).
    Returns (parent[N], token[N], rho[N]) with N <= n nodes (float64 rho)."""
    q = np.asarray(marginals, dtype=np.float64)
    C = q.shape[1]
    frontier = []  # (-rho, joined, parent, depth, token)
    joined = 0
    for x in range(C):
        heapq.heappush(frontier, (-float(q[0, x]), joined, -1, 1, x))
        joined += 1
    parent, token, rho = [], [], []
    total = 0.0
    while len(parent) < n and frontier:
        negr, _, p, d, x = frontier[0]
        r = -negr
        if cost is not None and parent:
            N = len(parent)
            if (total + r) / float(cost[N + 1]) < total / float(cost[N]):
                break
        heapq.heappop(frontier)
        i = len(parent)
        parent.append(p)
        token.append(x)
        rho.append(r)
        total += r
        if d < depth_cap:
            for y in range(C):
                heapq.heappush(frontier, (negr * float(q[d, y]), joined, i, d + 1, y))
                joined += 1
    return (np.array(parent, dtype=np.int32), np.array(token, dtype=np.int32),
            np.array(rho, dtype=np.float64))


def accept_stochastic_request(parent, draft, p_root, q_root, p_nodes, q_nodes, u_accept,
                              u_bonus: float, max_depth: int, with_margin: bool = False):
    """Stochastic acceptance of one request's draft tree (LLM Primer VI ch. 9, §9.1).

    The rule on a chain: a token x drawn from the draft distribution q is accepted
    with probability min(1, p(x)/q(x)), tested as u * q(x) < p(x) with the node's
    uniform u; after a rejection the target distribution becomes the normalized
    residual (p - q)_+ and the emitted token is drawn from it.  On a tree (reading):
    the children of the current node are tried in index order, each against the
    current residual; the first accepted child becomes the current node (its own
    p, q); if none is accepted, the bonus token is drawn from the current residual
    by inverse CDF: the first index whose running sum exceeds u_bonus * total.  A
    residual that sums to 0 (p <= q everywhere) leaves p unchanged.  fp64 throughout.
    Returns (L, path[max_depth], bonus), and the smallest decision margin if asked."""
    par = np.asarray(parent)
    n = len(par)
    p = np.asarray(p_root, dtype=np.float64)
    q = np.asarray(q_root, dtype=np.float64)
    cur, path, margin = -1, [], np.inf
    while True:
        accepted = False
        for c in range(cur + 1, n):
            if par[c] != cur:
                continue
            x = int(draft[c])
            lhs, rhs = float(u_accept[c]) * q[x], p[x]
            margin = min(margin, abs(lhs - rhs) / max(abs(lhs), abs(rhs), 1e-300))
            if lhs < rhs:
                if len(path) >= max_depth:
                    raise OracleError("accepted path longer than max_depth")
                path.append(c)
                cur = c
                p = np.asarray(p_nodes[c], dtype=np.float64)
                q = np.asarray(q_nodes[c], dtype=np.float64)
                accepted = True
                break
            r = np.maximum(p - q, 0.0)
            z = r.sum()
            if z > 0.0:
                p = r / z
        if not accepted:
            break
    cs = np.cumsum(p)
    target = float(u_bonus) * cs[-1]
    idx = int(np.searchsorted(cs, target, side="right"))
    if idx >= len(p):
        idx = int(np.nonzero(p > 0)[0][-1])
    if with_margin:
        gaps = np.abs(cs - target)
        margin = min(margin, float(gaps.min()) / max(cs[-1], 1e-300))
    out = np.full(max(max_depth, 1), -1, np.int32)
    out[:len(path)] = path
    if with_margin:
        return len(path), out, idx, margin
    return len(path), out, idx


def accept_stochastic(batch, root_p, node_p, root_q, node_q, u_accept, u_bonus,
                      max_depth: Optional[int] = None, with_margin: bool = False):
    """accept_stochastic_request for every request: (len[B], path[B,md], bonus[B])
    (and the smallest decision margin over the batch if asked)."""
    b = batch
    md = b.max_depth if max_depth is None else max_depth
    ln = np.zeros(b.B, np.int32)
    path = np.full((b.B, md), -1, np.int32)
    bonus = np.zeros(b.B, np.int32)
    margin = np.inf
    for r in range(b.B):
        s, e = int(b.node_offsets[r]), int(b.node_offsets[r + 1])
        res = accept_stochastic_request(b.parent[s:e], b.draft[s:e], root_p[r], root_q[r],
                                        node_p[s:e], node_q[s:e], u_accept[s:e], u_bonus[r],
                                        md, with_margin=True)
        ln[r], path[r], bonus[r] = res[0], res[1], res[2]
        margin = min(margin, res[3])
    if with_margin:
        return ln, path, bonus, margin
    return ln, path, bonus


def tree_attention(node_offsets, parent, q, k_cache, v_cache, ctx_len, k_tree, v_tree,
                   scale: float):
    """Softmax attention of one layer over draft trees with the tree mask -- the
    attention half of a hybrid model's verification pass.

    Pages: the target verifies all candidates in one forward pass over the prefix
    followed by the candidates (LLM Primer VI ch. 9, §9.1); a candidate tree is
    verified in one attention pass with a custom mask (§9.2); every branch shares
    the prefix's KV and adds only its own (Bole summary page, "Why existing tree
    speculation fails on hybrid models").  Reading: node i of request b, query head
    h, sees the b's first ctx_len[b] cached positions of KV head h // (H / Hkv) and
    the tree nodes on its own root path, itself included:
        o[i, h] = sum_j softmax_j(scale * q[i, h] . k_j) v_j.
    Shapes: q [T][H][d]; k_cache, v_cache [B][Hkv][P][d]; ctx_len [B];
    k_tree, v_tree [T][Hkv][d]; node_offsets [B+1]; parent [T] local to the request
    (-1 = child of the context, parents precede children).  fp64; returns [T][H][d].
    The mask is written out as a full 0/1 matrix and the softmax takes the row
    maximum out before exponentiating (exact in real arithmetic)."""
    q = np.asarray(q, dtype=np.float64)
    kc = np.asarray(k_cache, dtype=np.float64)
    vc = np.asarray(v_cache, dtype=np.float64)
    kt = np.asarray(k_tree, dtype=np.float64)
    vt = np.asarray(v_tree, dtype=np.float64)
    T, H, d = q.shape
    B, Hkv = kc.shape[0], kc.shape[1]
    if H % Hkv:
        raise OracleError("query heads must be a multiple of KV heads")
    grp = H // Hkv
    out = np.zeros((T, H, d), dtype=np.float64)
    for b in range(B):
        s, e = int(node_offsets[b]), int(node_offsets[b + 1])
        n, L = e - s, int(ctx_len[b])
        if n == 0:
            continue
        # anc[i, j] = 1 iff node j is on node i's root path (i included)
        anc = np.zeros((n, n), dtype=bool)
        for i in range(n):
            j = i
            while j >= 0:
                if j > i or int(parent[s + j]) >= j:
                    raise OracleError("parents must precede children")
                anc[i, j] = True
                j = int(parent[s + j])
        visible = np.concatenate([np.ones((n, L), dtype=bool), anc], axis=1)
        for h in range(H):
            kv = h // grp
            K = np.concatenate([kc[b, kv, :L], kt[s:e, kv]], axis=0)
            V = np.concatenate([vc[b, kv, :L], vt[s:e, kv]], axis=0)
            S = scale * (q[s:e, h] @ K.T)
            S = np.where(visible, S, -np.inf)
            S = S - S.max(axis=1, keepdims=True)
            W = np.exp(S)
            W = W / W.sum(axis=1, keepdims=True)
            out[s:e, h] = W @ V
    return out


def commit(batch, accept_len, path, units: Optional[Sequence[int]] = None, threads: int = 1,
           packed=None):
    """H_new of the listed units: dict u -> [dk, dv] float64."""
    b = batch
    P = packed or _Packed(b)
    if units is None:
        units = np.arange(b.B * b.H, dtype=np.int32)
    units = np.ascontiguousarray(units, dtype=np.int32)
    path = np.ascontiguousarray(path, np.int32)
    md = path.shape[1] if path.ndim == 2 else b.max_depth
    ln = np.ascontiguousarray(accept_len, np.int32)
    res = {}

    def run(chunk):
        out = np.zeros((len(chunk), b.dk, b.dv), np.float64)
        _rc(_L().orc_commit_batch(b.B, b.H, b.dk, b.dv, int(b.decay == "diag"), P.offs, P.g,
                                   P.k, P.v, P.H0, ln, path.reshape(-1), md, len(chunk),
                                   np.ascontiguousarray(chunk, np.int32), out.reshape(-1)),
            "commit_batch")
        return {int(u): out[i] for i, u in enumerate(chunk)}

    chunks = _split(units, threads * 4)
    if threads <= 1 or len(chunks) == 1:
        for c in chunks:
            res.update(run(c))
    else:
        with ThreadPoolExecutor(threads) as ex:
            for part in ex.map(run, chunks):
                res.update(part)
    return res
