"""GPU parity of tv_verify_serial, the naive node-by-node evaluator with per-node
states: against the fp64 oracle (2e-3 normwise per output row) and against the
tree closed form of tv_verify on the same inputs."""
import numpy as np
import pytest

import workloads
from gpu_util import check_verify, row_rel_err

pytestmark = pytest.mark.gpu


@pytest.fixture(scope="module", autouse=True)
def _lib():
    import torch
    if not torch.cuda.is_available():
        pytest.skip("no CUDA device")
    import tree_speculative_verify_tv_gb300 as tv
    tv.build()
    tv.load()


def serial(batch):
    import torch
    import tree_speculative_verify_tv_gb300 as tv
    d = tv.DeviceBatch(batch)
    nbytes = tv.tv_verify_serial_workspace_bytes(d.problem())
    ws = torch.empty(max(nbytes // 4, 4), dtype=torch.float32, device="cuda")
    ws.fill_(float("nan"))  # every state read must have been written first
    d.status.zero_()
    d.out.fill_(float("nan"))
    d.verify_serial(ws)
    torch.cuda.synchronize()
    out_s = d.out[:batch.T].cpu().numpy().astype(np.float64)
    st_s = int(d.status[0])
    d.status.zero_()
    d.verify()
    torch.cuda.synchronize()
    return st_s, out_s, int(d.status[0]), d.out[:batch.T].cpu().numpy().astype(np.float64)


@pytest.mark.parametrize("make", [
    lambda: workloads.config1(),
    lambda: workloads.config2(),
    lambda: workloads.config3(B=8),
    lambda: workloads.config4(B=8, H=4),
    lambda: workloads.config5(B=2, layers=1, heads=4),
], ids=["c1", "c2", "c3-B8", "c4-B8H4", "c5-B2"])
def test_serial_matches_oracle_and_closed_form(make):
    b = make()
    st, out, st2, out2 = serial(b)
    assert st == 0 and st2 == 0
    check_verify(b, out)
    assert row_rel_err(out, out2) <= 2e-3


@pytest.mark.parametrize("dk,dv,decay,dtype", [(16, 24, "scalar", "f32"), (64, 128, "diag", "bf16"),
                                               (128, 64, "scalar", "bf16"), (256, 8, "diag", "f32")])
def test_serial_ragged_shapes(dk, dv, decay, dtype):
    rng = np.random.default_rng(dk + dv)
    b = workloads.random_batch(rng, [0, 7, 1, 33, 0, 12], 3, dk, dv, decay=decay,
                               qkv_dtype=dtype, depth_cap=9, max_depth=9)
    st, out, _, _ = serial(b)
    assert st == 0
    check_verify(b, out)


def test_serial_malformed_tree_zero_rows():
    import tree_speculative_verify_tv_gb300 as tv
    rng = np.random.default_rng(4)
    b = workloads.random_batch(rng, [5, 6, 4], 2, 64, 64, decay="scalar", depth_cap=6,
                               max_depth=6)
    s1 = b.node_offsets[1]
    b.depth[s1 + 3] = 9
    st, out, _, _ = serial(b)
    assert st == tv.TV_ERR_TREE
    assert np.all(out[s1:b.node_offsets[2]] == 0.0)
    import oracle
    ref = oracle.verify(b, units=[0, 1, 4, 5])
    for u, o in ref.items():
        bb, h = divmod(u, b.H)
        assert row_rel_err(out[b.node_offsets[bb]:b.node_offsets[bb + 1], h], o) <= 2e-3
