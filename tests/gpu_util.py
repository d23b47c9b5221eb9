"""Helpers for the GPU parity tests: run the library on a host batch, compare
with the oracle.  Tolerance: normwise relative error <= 2e-3 per output row
(max |diff| over dv / max |ref| over dv) and per committed (request, head)
state matrix; acceptance results bit-exact."""
from __future__ import annotations

import numpy as np

TOL = 2e-3


def run_library(batch, variant=0, commit_in_place=False, steps=("verify", "accept", "commit")):
    import torch
    import tree_speculative_verify_tv_gb300 as tv

    d = tv.DeviceBatch(batch)
    d.status.zero_()
    if "verify" in steps:
        d.out.fill_(float("nan"))
        d.verify(variant=variant)
    if "accept" in steps:
        d.accept()
    if "commit" in steps:
        if not commit_in_place:
            d.H_new.fill_(float("nan"))
        d.commit(in_place=commit_in_place)
    if "accept_commit" in steps:
        if not commit_in_place:
            d.H_new.fill_(float("nan"))
        d.accept_commit(in_place=commit_in_place)
    torch.cuda.synchronize()
    res = {"status": int(d.status[0].item())}
    if "verify" in steps:
        res["out"] = d.out[:batch.T].cpu().numpy().astype(np.float64)
    if "accept" in steps or "accept_commit" in steps:
        res["len"] = d.accept_len[:batch.B].cpu().numpy()
        res["path"] = d.path[:batch.B].cpu().numpy()
        res["bonus"] = d.bonus[:batch.B].cpu().numpy()
    if "commit" in steps or "accept_commit" in steps:
        res["H_new"] = (d.H0 if commit_in_place else d.H_new).cpu().numpy().astype(np.float64)
    return res


def row_rel_err(got: np.ndarray, ref: np.ndarray) -> float:
    """max over rows of max|got-ref| / max|ref| (rows along the last axis)."""
    got = got.reshape(-1, got.shape[-1])
    ref = ref.reshape(-1, ref.shape[-1])
    if got.size == 0:
        return 0.0
    num = np.max(np.abs(got - ref), axis=1)
    den = np.maximum(np.max(np.abs(ref), axis=1), 1e-30)
    bad = ~np.isfinite(got).all(axis=1)
    e = num / den
    e[bad] = np.inf
    return float(e.max())


def mat_rel_err(got: np.ndarray, ref: np.ndarray) -> float:
    if got.size == 0:
        return 0.0
    if not np.isfinite(got).all():
        return float("inf")
    return float(np.max(np.abs(got - ref)) / max(np.max(np.abs(ref)), 1e-30))


def check_verify(batch, out, units=None, tol=TOL, threads=8):
    import oracle
    ref = oracle.verify(batch, units=units, threads=threads)
    worst = 0.0
    for u, o in ref.items():
        b, h = divmod(u, batch.H)
        s, e = batch.node_offsets[b], batch.node_offsets[b + 1]
        worst = max(worst, row_rel_err(out[s:e, h, :], o))
    assert worst <= tol, "verify rel err %.3e > %.1e" % (worst, tol)
    return worst


def check_accept(batch, res):
    import oracle
    ln, path, bonus = oracle.accept_batch(batch)
    assert np.array_equal(res["len"], ln), (res["len"], ln)
    assert np.array_equal(res["path"], path)
    assert np.array_equal(res["bonus"], bonus)
    return ln, path


def check_commit(batch, H_new, ln, path, units=None, tol=TOL, threads=8):
    import oracle
    ref = oracle.commit(batch, ln, path, units=units, threads=threads)
    worst = 0.0
    for u, Hr in ref.items():
        b, h = divmod(u, batch.H)
        worst = max(worst, mat_rel_err(H_new[b, h], Hr))
    assert worst <= tol, "commit rel err %.3e > %.1e" % (worst, tol)
    return worst
