"""Pins of the fp64 oracle (CPU only).

The oracle is checked against a hand-worked example, textbook reductions, brute
force over every small tree and invariances (see tests/oracle_checks.py).  The
mutation test then plants plausible mistakes in copies of the oracle's C source
and shows that each one fails at least one of these pins.
"""
import os
import shutil
import subprocess

import numpy as np
import pytest

import oracle
import oracle_checks as oc
import workloads


def test_golden_hand_example():
    oc.check_golden()


def test_chain_tree_equals_parallel_gla():
    oc.check_chain_is_gla()


def test_zero_decay_zero_state_is_tree_masked_linear_attention():
    oc.check_masked_linear_attention()


def test_no_updates_gives_decayed_context_readout():
    oc.check_no_update_closed_form()


def test_linearity_and_scaling():
    oc.check_linearity_and_scaling()


def test_siblings_and_relabelling():
    oc.check_siblings_and_relabel()


def test_bruteforce_every_tree_up_to_7_nodes():
    oc.check_bruteforce_small(7)


def test_bruteforce_sampled_8_node_trees():
    oc.check_bruteforce_sampled_n8(trials=2000)


def test_accept_matches_exhaustive_enumeration():
    oc.check_accept_exhaustive(trials=3000)


def test_accept_special_cases():
    oc.check_accept_special_cases()


def test_commit_is_state_of_accepted_node():
    oc.check_commit_is_accepted_state()


def test_reroot_invariance():
    oc.check_reroot()


def test_oracle_rejects_malformed_trees():
    bad = [np.array([0], np.int32), np.array([-1, 1], np.int32), np.array([-2], np.int32),
           np.array([-1, 0, 3, 1], np.int32)]
    for parent in bad:
        n = len(parent)
        with pytest.raises(oracle.OracleError):
            oracle.verify_unit(parent, np.zeros((n, 2)), np.zeros((n, 2)), np.zeros((n, 2)),
                               np.zeros(n), np.zeros((2, 2)), diag=False)


def test_batch_drivers_match_unit_routines():
    b = workloads.random_batch(np.random.default_rng(3), [5, 0, 9, 1], 3, 8, 16, decay="diag")
    res = oracle.verify(b)
    q, k, v = b.qkv_f32(b.q), b.qkv_f32(b.k), b.qkv_f32(b.v)
    for u, out in res.items():
        bb, h = divmod(u, b.H)
        s, e = b.node_offsets[bb], b.node_offsets[bb + 1]
        ref = oracle.verify_unit(b.parent[s:e], q[s:e, h], k[s:e, h], v[s:e, h], b.g[s:e, h],
                                 b.H0[bb, h], diag=True)
        assert np.array_equal(out, ref)
    ln, path, bonus = oracle.accept_batch(b)
    for bb in range(b.B):
        s, e = b.node_offsets[bb], b.node_offsets[bb + 1]
        L, p, bo = oracle.accept(b.parent[s:e], b.draft[s:e], b.target[s:e], b.root_argmax[bb],
                                 b.max_depth)
        assert (L, bo) == (ln[bb], bonus[bb]) and np.array_equal(p, path[bb])
    Hn = oracle.commit(b, ln, path)
    for u, H in Hn.items():
        bb, h = divmod(u, b.H)
        s, e = b.node_offsets[bb], b.node_offsets[bb + 1]
        ref = oracle.commit_unit(path[bb], int(ln[bb]), k[s:e, h], v[s:e, h], b.g[s:e, h],
                                 b.H0[bb, h], diag=True)
        assert np.array_equal(H, ref)


# ------------------------------------------------------------------ planted mistakes

MUTANTS = {
    "output read before the node's own update": (
        "acc += S[(size_t)r * dv + c] * q", "acc += prev[(size_t)r * dv + c] * q"),
    "decay applied after adding the update": (
        "S[(size_t)r * dv + c] = a * prev[(size_t)r * dv + c]\n"
        "                                      + k[(size_t)i * dk + r] * v[(size_t)i * dv + c];",
        "S[(size_t)r * dv + c] = a * (prev[(size_t)r * dv + c]\n"
        "                                      + k[(size_t)i * dk + r] * v[(size_t)i * dv + c]);"),
    "decay with the wrong sign": ("exp(diag ? g[(size_t)i * dk + r] : g[i])",
                                  "exp(-(diag ? g[(size_t)i * dk + r] : g[i]))"),
    "dropped update term": (
        "                                      + k[(size_t)i * dk + r] * v[(size_t)i * dv + c];",
        "                                      + 0.0 * k[(size_t)i * dk + r];"),
    "parent ignored (sequence instead of tree)": (
        "parent[i] < 0 ? H0 : states + (size_t)parent[i] * dk * dv",
        "i == 0 ? H0 : states + (size_t)(i - 1) * dk * dv"),
    "greedy keeps the last matching child": ("{ c = i; break; }", "{ c = i; }"),
    "bonus is the root token": ("*bonus = t;", "*bonus = root_tok;"),
    "commit drops the last path node": ("for (int m = 0; m < L; ++m) {\n        int i = path[m];",
                                        "for (int m = 0; m < L - 1; ++m) {\n        int i = path[m];"),
    "scalar decay read from the wrong node": ("exp(diag ? g[(size_t)i * dk + r] : g[i])",
                                              "exp(diag ? g[(size_t)i * dk + r] : g[i > 0 ? i - 1 : i])"),
}


@pytest.mark.parametrize("name", sorted(MUTANTS))
def test_pins_catch_planted_mistake(name, tmp_path):
    if shutil.which("gcc") is None:
        pytest.skip("gcc not available")
    src = open(os.path.join(os.path.dirname(oracle.__file__), "oracle.c")).read()
    old, new = MUTANTS[name]
    assert src.count(old) >= 1, "mutation anchor not found: " + name
    mut = src.replace(old, new)
    cfile = tmp_path / "mutant.c"
    cfile.write_text(mut)
    so = tmp_path / "libmutant.so"
    subprocess.check_call(["gcc", "-O1", "-std=c99", "-fPIC", "-shared", "-o", str(so), str(cfile),
                           "-lm"])
    L = oracle.load(str(so))
    failed = []
    with oracle.using(L):
        for chk in oc.QUICK_CHECKS:
            try:
                chk()
            except (AssertionError, oracle.OracleError, IndexError):
                failed.append(getattr(chk, "__name__", "check"))
    assert failed, "no pin caught: " + name
