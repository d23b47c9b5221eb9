"""GPU parity of the persistent tensor-core verify kernel (TV_VARIANT_TC_STREAM):
each CTA streams several (request, head) units through two shared-memory stages,
so these cases run more units than resident CTAs (both stages and both barrier
phases in use) and compare with the fp64 oracle (2e-3 normwise per row) and, bit
for bit, with the one-unit tensor-core kernel, which does the same arithmetic.
"""
import numpy as np
import pytest

import workloads
from gpu_util import check_verify, run_library

pytestmark = pytest.mark.gpu

STREAM = 3


@pytest.fixture(scope="module", autouse=True)
def _lib():
    import torch
    if not torch.cuda.is_available():
        pytest.skip("no CUDA device")
    import tree_speculative_verify_tv_gb300 as tv
    tv.build()
    tv.load()
    assert tv.TV_VARIANT_TC_STREAM == STREAM


def _verify(batch, variant):
    res = run_library(batch, variant=variant, steps=("verify",))
    return res["status"], res["out"]


def test_stream_mamba2_layer():
    """Mamba-2-like layer, B=16, H=24: 384 units over the resident CTAs."""
    b = workloads.config2(seed=5)
    st, out = _verify(b, STREAM)
    assert st == 0
    check_verify(b, out)


def test_stream_folded_layers_sampled():
    """32 Mamba-2-like layers folded into the head axis (H = 768, 12288 units), the
    launch the folded measurement times; 96 sampled units against the oracle."""
    b = workloads.config2(seed=77, H=24 * 32)
    st, out = _verify(b, STREAM)
    assert st == 0
    rng = np.random.default_rng(3)
    units = np.sort(rng.choice(b.B * b.H, 96, replace=False))
    check_verify(b, out, units=units)


def test_stream_equals_one_unit_kernel():
    b = workloads.config2(seed=8, H=24 * 8)
    s1, o1 = _verify(b, STREAM)
    s2, o2 = _verify(b, 2)
    assert s1 == 0 and s2 == 0
    assert np.array_equal(o1, o2)


@pytest.mark.parametrize("dk,dv", [(64, 64), (64, 128), (128, 64), (128, 128)])
def test_stream_ragged_with_empty_requests(dk, dv):
    rng = np.random.default_rng(dk * 3 + dv)
    sizes = rng.integers(0, 41, 60)
    sizes[::7] = 0
    b = workloads.random_batch(rng, sizes, 12, dk, dv, decay="scalar", depth_cap=10,
                               max_depth=10)
    st, out = _verify(b, STREAM)
    assert st == 0
    check_verify(b, out)


def test_stream_deep_chains():
    rng = np.random.default_rng(9)
    b = workloads.random_batch(rng, [32] * 40, 16, 128, 64, decay="scalar", depth_cap=32)
    st, out = _verify(b, STREAM)
    assert st == 0
    check_verify(b, out)


def test_stream_malformed_tree_and_offsets():
    """A malformed tree zeroes its request's rows and sets TV_ERR_TREE; the other
    requests (streamed through the same CTAs) are unaffected."""
    import torch
    import oracle
    import tree_speculative_verify_tv_gb300 as tv
    rng = np.random.default_rng(12)
    b = workloads.random_batch(rng, [9] * 50, 16, 128, 64, decay="scalar", depth_cap=8,
                               max_depth=8)
    bad = 7
    s0 = b.node_offsets[bad]
    b.parent[s0 + 3] = 5                       # a parent after its child
    d = tv.DeviceBatch(b)
    d.status.zero_()
    d.out.fill_(float("nan"))
    d.verify(variant=STREAM)
    torch.cuda.synchronize()
    assert int(d.status[0]) == tv.TV_ERR_TREE
    out = d.out[:b.T].cpu().numpy().astype(np.float64)
    assert np.all(out[s0:b.node_offsets[bad + 1]] == 0.0)
    good = [u for u in range(b.B * b.H) if u // b.H != bad]
    ref = oracle.verify(b, units=good, threads=8)
    for u, o in ref.items():
        bb, h = divmod(u, b.H)
        got = out[b.node_offsets[bb]:b.node_offsets[bb + 1], h]
        assert np.max(np.abs(got - o)) <= 2e-3 * max(np.max(np.abs(o)), 1e-30)
