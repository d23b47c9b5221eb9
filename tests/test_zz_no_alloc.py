"""tv_verify_serial_static, the entry point for callers that cannot allocate
device memory: it keeps the per-node states in the library's built-in 16 MiB
scratch array instead of a caller workspace.  Through the C ABI, two calls in a
row (different problems, so the second reuses the array the first wrote) must
each give the outputs of tv_verify_serial with a caller workspace, within the
2e-3 normwise tolerance of the other parity tests.  This file is collected last
on purpose: a run that stops at the first failure has run every other test."""
import numpy as np
import pytest

import workloads
from gpu_util import TOL, row_rel_err

pytestmark = pytest.mark.gpu


@pytest.fixture(scope="module", autouse=True)
def _lib():
    import torch
    if not torch.cuda.is_available():
        pytest.skip("no CUDA device")
    import tree_speculative_verify_tv_gb300 as tv
    tv.build()
    tv.load()


def _outputs(batch):
    """(outputs with a workspace, outputs from the built-in scratch array)."""
    import torch
    import tree_speculative_verify_tv_gb300 as tv
    d = tv.DeviceBatch(batch)
    p = d.problem()
    need = tv.tv_verify_serial_workspace_bytes(p)
    assert 0 < need <= tv.TV_SERIAL_STATIC_BYTES
    ws = torch.empty(need // 4, dtype=torch.float32, device="cuda")
    d.status.zero_()
    tv.tv_verify_serial(p, d.H0, d.q, d.k, d.v, d.g, d.out, ws, need, d.status)
    torch.cuda.synchronize()
    assert int(d.status[0]) == 0
    ref = d.out[:batch.T].clone()
    d.out.fill_(float("nan"))
    rc = tv.tv_verify_serial_static(p, d.H0, d.q, d.k, d.v, d.g, d.out, d.status, check=False)
    torch.cuda.synchronize()
    assert rc == tv.TV_OK, tv.status_string(rc)
    assert int(d.status[0]) == 0
    return ref.cpu().numpy().astype(np.float64), d.out[:batch.T].cpu().numpy().astype(np.float64)


def test_static_scratch_matches_workspace_on_two_calls():
    first = workloads.config2(seed=61, B=1)   # one Mamba-2-like request: 12 MiB of states
    second = workloads.random_batch(np.random.default_rng(62), [9, 0, 30, 4], 2, 64, 128,
                                    decay="diag", depth_cap=10, max_depth=10)
    for batch in (first, second):
        ref, got = _outputs(batch)
        assert np.isfinite(got).all()
        assert row_rel_err(got, ref) <= TOL


def test_static_scratch_exactly_full():
    """A problem whose states fill the array exactly (2 requests x 8 heads x 16 nodes
    x 128 x 128 fp32 = 16 MiB): the last unit's last node writes the array's last
    bytes.  One more request is rejected before anything runs."""
    import tree_speculative_verify_tv_gb300 as tv
    b = workloads.random_batch(np.random.default_rng(63), [16, 16], 8, 128, 128,
                               decay="scalar", depth_cap=8, max_depth=8, max_nodes=16)
    d = tv.DeviceBatch(b)
    assert tv.tv_verify_serial_workspace_bytes(d.problem()) == tv.TV_SERIAL_STATIC_BYTES
    ref, got = _outputs(b)
    assert np.isfinite(got).all()
    assert row_rel_err(got, ref) <= TOL
    over = workloads.random_batch(np.random.default_rng(64), [16, 16, 1], 8, 128, 128,
                                  decay="scalar", depth_cap=8, max_depth=8, max_nodes=16)
    do = tv.DeviceBatch(over)
    rc = tv.tv_verify_serial_static(do.problem(), do.H0, do.q, do.k, do.v, do.g, do.out,
                                    do.status, check=False)
    assert rc == tv.TV_ERR_UNSUPPORTED


def test_static_scratch_takes_no_memory_per_call():
    """After a first call has loaded the library's code on the device, a call takes no
    device memory: the free memory the driver reports is the same before and after."""
    import torch
    import tree_speculative_verify_tv_gb300 as tv
    b = workloads.config2(seed=65, B=1)
    d = tv.DeviceBatch(b)
    p = d.problem()
    d.status.zero_()
    tv.tv_verify_serial_static(p, d.H0, d.q, d.k, d.v, d.g, d.out, d.status)
    torch.cuda.synchronize()
    free0 = torch.cuda.mem_get_info()[0]
    for _ in range(3):
        tv.tv_verify_serial_static(p, d.H0, d.q, d.k, d.v, d.g, d.out, d.status)
    torch.cuda.synchronize()
    assert torch.cuda.mem_get_info()[0] == free0
    assert int(d.status[0]) == 0
