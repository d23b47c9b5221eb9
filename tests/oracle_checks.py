"""Independent checks that pin the fp64 oracle to the mathematics.

Each check compares the oracle with something other than itself:
  * a hand-worked example (tests/golden/hand_tree_3node.txt),
  * the textbook parallel ("attention") form of gated linear attention on a chain,
  * tree-masked causal linear attention (g = 0, H0 = 0) with the mask found by
    brute-force reachability,
  * the closed form o_i = H0^T (e^{G_i} * q_i) when k = v = 0,
  * the tree closed form and a per-node root-path replay on every tree of <= 5 nodes,
  * invariances (linearity, sibling symmetry, relabelling, re-rooting),
  * an exhaustive characterisation of the greedy walk (lexicographically first
    maximal matching root path), and
  * the commit against the materialised state of the accepted node.

Operations: Bole summary page, "Core techniques" §1 (h_{t+1} = S_t h_t + u_t with
S = diag(exp g), u = k v^T, o = H^T q) and §2 (commit the accepted path's state);
LLM Primer VI ch. 9 §9.1 (greedy acceptance).

The checks are plain functions so that tests/test_oracle_pins.py can also run
them against deliberately broken builds of the oracle and see them fail.
"""
from __future__ import annotations

import itertools
import os

import numpy as np

import oracle

GOLDEN = os.path.join(os.path.dirname(os.path.abspath(__file__)), "golden")


# ------------------------------------------------------------------ helpers (independent)


def ancestors(parent):
    """anc*(i): nodes reachable from i by following parent links, i included."""
    n = len(parent)
    out = []
    for i in range(n):
        s, j, steps = [], i, 0
        while j >= 0:
            s.append(j)
            j = int(parent[j])
            steps += 1
            assert steps <= n, "cycle"
        out.append(s)
    return out


def root_path(parent, i):
    return list(reversed(ancestors(parent)[i]))


def closed_form(parent, q, k, v, g, H0, diag):
    """Tree closed form: o_i = H0^T(e^{G_i} q_i) + sum_{j in anc*(i)} (sum_c q_ic k_jc
    e^{G_ic - G_jc}) v_j, with G_i the sum of g over anc*(i)."""
    n, dk = q.shape
    gg = g if diag else np.repeat(np.asarray(g, np.float64)[:, None], dk, axis=1)
    anc = ancestors(parent)
    G = np.array([gg[a].sum(axis=0) for a in anc]) if n else np.zeros((0, dk))
    out = np.zeros((n, H0.shape[1]))
    for i in range(n):
        out[i] = H0.T @ (np.exp(G[i]) * q[i])
        for j in anc[i]:
            out[i] += np.sum(q[i] * k[j] * np.exp(G[i] - G[j])) * v[j]
    return out


def path_replay(parent, q, k, v, g, H0, diag):
    """Per node: run the plain sequential recurrence over its root path."""
    n, dk = q.shape
    out = np.zeros((n, H0.shape[1]))
    for i in range(n):
        S = H0.copy()
        for j in root_path(parent, i):
            a = np.exp(g[j]) if diag else np.exp(g[j]) * np.ones(dk)
            S = a[:, None] * S + np.outer(k[j], v[j])
        out[i] = S.T @ q[i]
    return out


def gla_parallel_chain(q, k, v, g, H0, diag):
    """Textbook parallel form of gated linear attention on a sequence (no tree):
    Gc = cumsum(g); O = ((Q e^{Gc}) (K e^{-Gc})^T * causal) V + (Q e^{Gc}) H0."""
    n, dk = q.shape
    gg = g if diag else np.repeat(np.asarray(g, np.float64)[:, None], dk, axis=1)
    Gc = np.cumsum(gg, axis=0)
    Qt = q * np.exp(Gc)
    Kt = k * np.exp(-Gc)
    A = np.tril(Qt @ Kt.T)
    return A @ v + Qt @ H0


def rand_unit(rng, n, dk, dv, diag, gscale=1.0):
    q = rng.standard_normal((n, dk))
    k = rng.standard_normal((n, dk))
    v = rng.standard_normal((n, dv))
    g = -gscale * rng.random((n, dk) if diag else n)
    H0 = rng.standard_normal((dk, dv))
    return q, k, v, g, H0


def close(a, b, tol=1e-10):
    a, b = np.asarray(a, np.float64), np.asarray(b, np.float64)
    scale = max(1.0, float(np.max(np.abs(b))) if b.size else 1.0)
    return a.shape == b.shape and float(np.max(np.abs(a - b)) if a.size else 0.0) <= tol * scale


# ------------------------------------------------------------------ golden fixture


def _fields(val):
    """'a=1 2 b=3 c=' -> {'a': ['1','2'], 'b': ['3'], 'c': []}."""
    out, cur = {}, None
    for tok in val.split():
        if "=" in tok:
            cur, _, first = tok.partition("=")
            out[cur] = [first] if first else []
        else:
            out[cur].append(tok)
    return out


def load_golden():
    cases, walks, acc, cur = [], [], None, None
    with open(os.path.join(GOLDEN, "hand_tree_3node.txt")) as f:
        for line in f:
            line = line.split("#", 1)[0].strip()
            if not line:
                continue
            key, _, val = line.partition(":")
            key, val = key.strip(), val.strip()
            if key == "case":
                cur = {"name": val}
                cases.append(cur)
            elif key == "accept":
                d = _fields(val)
                acc = {"draft": [int(x) for x in d["draft"]],
                       "target": [int(x) for x in d["target"]]}
            elif key == "walk":
                d = _fields(val)
                walks.append({"root": int(d["root"][0]), "len": int(d["len"][0]),
                              "path": [int(x) for x in d["path"]],
                              "bonus": int(d["bonus"][0]), "commit": d["commit"][0]})
            else:
                cur[key] = [float(x) for x in val.split()]
    return cases, acc, walks


def check_golden():
    cases, acc, walks = load_golden()
    assert len(cases) == 2 and len(walks) == 3
    for c in cases:
        parent = np.array(c["parent"], np.int32)
        n = len(parent)
        dk, dv = int(c["dk"][0]), int(c["dv"][0])
        diag = c["name"] == "diag"
        H0 = np.array(c["H0"]).reshape(dk, dv)
        k = np.array(c["k"]).reshape(n, dk)
        v = np.array(c["v"]).reshape(n, dv)
        q = np.array(c["q"]).reshape(n, dk)
        a = np.array(c["decay_factors"]).reshape((n, dk) if diag else (n,))
        g = np.log(a)
        out, states = oracle.verify_unit(parent, q, k, v, g, H0, diag=diag, return_states=True)
        assert close(out, np.array(c["out"]).reshape(n, dv), 1e-12), (c["name"], out)
        for i in range(n):
            assert close(states[i], np.array(c["state%d" % i]).reshape(dk, dv), 1e-12)
        for w in walks:
            L, path, bonus = oracle.accept(parent, acc["draft"], acc["target"], w["root"], 4)
            assert L == w["len"] and list(path[:L]) == w["path"] and bonus == w["bonus"], w
            assert all(p == -1 for p in path[L:])
            Hn = oracle.commit_unit(path, L, k, v, g, H0, diag=diag)
            ref = H0 if w["commit"] == "H0" else np.array(c[w["commit"]]).reshape(dk, dv)
            assert close(Hn, ref, 1e-12), (c["name"], w)


# ------------------------------------------------------------------ recurrence pins


def check_chain_is_gla(seed=0):
    rng = np.random.default_rng(seed)
    for diag in (False, True):
        for n, dk, dv in ((1, 3, 2), (7, 4, 5), (12, 8, 3)):
            q, k, v, g, H0 = rand_unit(rng, n, dk, dv, diag)
            parent = np.arange(-1, n - 1, dtype=np.int32)
            out = oracle.verify_unit(parent, q, k, v, g, H0, diag=diag)
            assert close(out, gla_parallel_chain(q, k, v, g, H0, diag), 1e-9), (diag, n)


def check_masked_linear_attention(seed=1):
    rng = np.random.default_rng(seed)
    for n in (1, 5, 9, 16):
        parent = np.array([-1] + [int(rng.integers(-1, i)) for i in range(1, n)], np.int32)
        q, k, v, _, _ = rand_unit(rng, n, 6, 4, False)
        M = np.zeros((n, n))
        for i, a in enumerate(ancestors(parent)):
            M[i, a] = 1.0
        ref = (M * (q @ k.T)) @ v
        for diag in (False, True):
            g = np.zeros((n, 6)) if diag else np.zeros(n)
            out = oracle.verify_unit(parent, q, k, v, g, np.zeros((6, 4)), diag=diag)
            assert close(out, ref, 1e-10), (n, diag)


def check_no_update_closed_form(seed=2):
    rng = np.random.default_rng(seed)
    for diag in (False, True):
        n, dk, dv = 10, 5, 7
        parent = np.array([-1] + [int(rng.integers(-1, i)) for i in range(1, n)], np.int32)
        q, _, _, g, H0 = rand_unit(rng, n, dk, dv, diag)
        gg = g if diag else np.repeat(g[:, None], dk, axis=1)
        G = np.array([gg[a].sum(axis=0) for a in ancestors(parent)])
        ref = (q * np.exp(G)) @ H0
        out = oracle.verify_unit(parent, q, np.zeros((n, dk)), np.zeros((n, dv)), g, H0,
                                 diag=diag)
        assert close(out, ref, 1e-10), diag


def check_linearity_and_scaling(seed=3):
    rng = np.random.default_rng(seed)
    n, dk, dv = 9, 4, 6
    parent = np.array([-1, 0, 0, 1, -1, 4, 3, 2, 6], np.int32)
    for diag in (False, True):
        q, k, v, g, H0 = rand_unit(rng, n, dk, dv, diag)
        _, _, v2, _, H02 = rand_unit(rng, n, dk, dv, diag)
        f = lambda H, vv, qq=q: oracle.verify_unit(parent, qq, k, vv, g, H, diag=diag)
        assert close(f(H0 + H02, v + v2), f(H0, v) + f(H02, v2), 1e-10)
        assert close(f(2.5 * H0, 2.5 * v), 2.5 * f(H0, v), 1e-10)
        assert close(f(H0, v, -3.0 * q), -3.0 * f(H0, v), 1e-10)


def check_siblings_and_relabel(seed=4):
    rng = np.random.default_rng(seed)
    dk, dv = 4, 3
    # nodes 1 and 2 are siblings (children of 0) with identical factors
    parent = np.array([-1, 0, 0, 1, 2], np.int32)
    for diag in (False, True):
        q, k, v, g, H0 = rand_unit(rng, 5, dk, dv, diag)
        for arr in (q, k, v, g):
            arr[2] = arr[1]
            arr[4] = arr[3]
        out = oracle.verify_unit(parent, q, k, v, g, H0, diag=diag)
        assert close(out[1], out[2], 1e-12) and close(out[3], out[4], 1e-12)
    # topology-preserving relabel (parents still precede children) permutes outputs
    n = 8
    parent = np.array([-1, 0, -1, 1, 0, 2, 3, 5], np.int32)
    # a random linear extension of the tree order: every parent still precedes its child
    placed, order = set(), []
    while len(order) < n:
        ready = [i for i in range(n) if i not in placed and (parent[i] < 0 or parent[i] in placed)]
        pick = ready[int(rng.integers(0, len(ready)))]
        placed.add(pick)
        order.append(pick)
    assert order != list(range(n))
    perm = np.empty(n, np.int64)
    perm[order] = np.arange(n)                 # new index of old node i
    inv = np.array(order)                      # old node at new index
    new_parent = np.array([perm[parent[o]] if parent[o] >= 0 else -1 for o in inv], np.int32)
    assert all(new_parent[i] < i for i in range(n))
    for diag in (False, True):
        q, k, v, g, H0 = rand_unit(rng, n, dk, dv, diag)
        out = oracle.verify_unit(parent, q, k, v, g, H0, diag=diag)
        out2 = oracle.verify_unit(new_parent, q[inv], k[inv], v[inv], g[inv], H0, diag=diag)
        assert close(out2, out[inv], 1e-12)


def all_parent_arrays(n):
    """Every parent array with parent[i] in {-1, 0, .., i-1}: (n)! trees incl. forests."""
    return itertools.product(*[range(-1, i) for i in range(n)])


def check_bruteforce_small(max_n=5, seed=5):
    rng = np.random.default_rng(seed)
    for n in range(1, max_n + 1):
        for diag in (False, True):
            q, k, v, g, H0 = rand_unit(rng, n, 3, 2, diag)
            for par in all_parent_arrays(n):
                parent = np.array(par, np.int32)
                out = oracle.verify_unit(parent, q, k, v, g, H0, diag=diag)
                assert close(out, closed_form(parent, q, k, v, g, H0, diag), 1e-10), par
                assert close(out, path_replay(parent, q, k, v, g, H0, diag), 1e-10), par


def check_bruteforce_sampled_n8(trials=60, seed=6):
    rng = np.random.default_rng(seed)
    for _ in range(trials):
        diag = bool(rng.integers(0, 2))
        parent = np.array([int(rng.integers(-1, i)) for i in range(8)], np.int32)
        q, k, v, g, H0 = rand_unit(rng, 8, 4, 3, diag)
        out = oracle.verify_unit(parent, q, k, v, g, H0, diag=diag)
        assert close(out, closed_form(parent, q, k, v, g, H0, diag), 1e-10)
        assert close(out, path_replay(parent, q, k, v, g, H0, diag), 1e-10)


# ------------------------------------------------------------------ accept / commit pins


def greedy_by_enumeration(parent, draft, target, root_tok):
    """Lexicographically first maximal matching root path (exhaustive)."""
    n = len(parent)
    matching = []
    for i in range(n):
        p = root_path(parent, i)
        ok = draft[p[0]] == root_tok and all(target[a] == draft[b] for a, b in zip(p, p[1:]))
        if ok:
            matching.append(tuple(p))
    mset = set(matching)
    maximal = [p for p in matching
               if not any(parent[c] == p[-1] and (p + (c,)) in mset for c in range(n))]
    if not maximal:
        return (), root_tok
    best = min(maximal)
    return best, target[best[-1]]


def check_accept_exhaustive(trials=400, seed=7):
    rng = np.random.default_rng(seed)
    for t in range(trials):
        n = int(rng.integers(0, 12))
        parent = np.array([int(rng.integers(-1, i)) for i in range(n)], np.int32)
        vocab = int(rng.integers(1, 4))           # small vocab: many duplicate siblings
        draft = rng.integers(0, vocab, n).astype(np.int32)
        target = rng.integers(0, vocab, n).astype(np.int32)
        root = int(rng.integers(0, vocab))
        md = int(max([len(root_path(parent, i)) for i in range(n)] + [1]))
        L, path, bonus = oracle.accept(parent, draft, target, root, md)
        ref, rbonus = greedy_by_enumeration(parent, draft, target, root)
        assert tuple(path[:L]) == ref and bonus == rbonus, (t, parent, draft, target, root)
        assert all(x == -1 for x in path[L:])


def check_accept_special_cases():
    # chain where every target matches the next draft: accept the whole depth
    n = 6
    parent = np.arange(-1, n - 1, dtype=np.int32)
    draft = np.arange(10, 10 + n, dtype=np.int32)
    target = np.arange(11, 11 + n, dtype=np.int32)
    L, path, bonus = oracle.accept(parent, draft, target, 10, n)
    assert L == n and list(path) == list(range(n)) and bonus == 10 + n
    # no child of the context matches: nothing accepted, bonus = root token
    L, path, bonus = oracle.accept(parent, draft, target, 99, n)
    assert L == 0 and bonus == 99 and all(p == -1 for p in path)
    # empty tree
    L, path, bonus = oracle.accept(np.zeros(0, np.int32), [], [], 5, 3)
    assert L == 0 and bonus == 5


def check_commit_is_accepted_state(seed=8):
    rng = np.random.default_rng(seed)
    for trial in range(30):
        n = int(rng.integers(1, 14))
        diag = bool(trial % 2)
        parent = np.array([int(rng.integers(-1, i)) for i in range(n)], np.int32)
        q, k, v, g, H0 = rand_unit(rng, n, 4, 5, diag)
        _, states = oracle.verify_unit(parent, q, k, v, g, H0, diag=diag, return_states=True)
        u = int(rng.integers(0, n))
        p = root_path(parent, u)
        Hn = oracle.commit_unit(np.array(p, np.int32), len(p), k, v, g, H0, diag=diag)
        assert close(Hn, states[u], 1e-12)
        assert close(oracle.commit_unit(np.zeros(1, np.int32), 0, k, v, g, H0, diag=diag), H0, 0)


def check_reroot(seed=9):
    """Verifying u's subtree from H0' = commit(H0, path to u) reproduces its outputs."""
    rng = np.random.default_rng(seed)
    for diag in (False, True):
        n = 12
        parent = np.array([-1, 0, 0, 1, 1, 2, 3, 3, 4, 6, 7, 5], np.int32)
        q, k, v, g, H0 = rand_unit(rng, n, 5, 4, diag)
        out = oracle.verify_unit(parent, q, k, v, g, H0, diag=diag)
        u = 1
        p = root_path(parent, u)
        H0u = oracle.commit_unit(np.array(p, np.int32), len(p), k, v, g, H0, diag=diag)
        sub = [i for i in range(n) if u in ancestors(parent)[i] and i != u]
        idx = {o: s for s, o in enumerate(sub)}
        sp = np.array([idx[parent[o]] if parent[o] != u else -1 for o in sub], np.int32)
        out2 = oracle.verify_unit(sp, q[sub], k[sub], v[sub], g[sub], H0u, diag=diag)
        assert close(out2, out[sub], 1e-11)


QUICK_CHECKS = [check_golden, check_chain_is_gla, check_masked_linear_attention,
                check_no_update_closed_form, check_linearity_and_scaling,
                check_siblings_and_relabel, lambda: check_bruteforce_small(4),
                check_accept_exhaustive, check_accept_special_cases,
                check_commit_is_accepted_state, check_reroot]
