"""The library is thread-safe: host threads that call it at the same time, each on
its own stream and buffers, get the same results as one thread alone.  The two
problems below run the one-unit tensor-core kernel with different shared-memory
sizes (16-node trees and trees of up to 128 nodes), the case where a per-call
rewrite of the kernel's shared-memory limit could let one thread's launch see the
other's smaller limit; and the fused kernel and tree attention alongside."""
import threading

import numpy as np
import pytest

import workloads

pytestmark = pytest.mark.gpu


@pytest.fixture(scope="module", autouse=True)
def _lib():
    import torch
    if not torch.cuda.is_available():
        pytest.skip("no CUDA device")
    import tree_speculative_verify_tv_gb300 as tv
    tv.build()
    tv.load()


def _once(d, variant, stream):
    import torch
    d.status.zero_()
    d.out.fill_(float("nan"))
    d.verify(stream=stream, variant=variant)
    stream.synchronize()
    return int(d.status[0]), d.out.clone()


@pytest.mark.parametrize("variants", [(2, 2), (0, 2), (3, 2)])
def test_two_host_threads_two_shapes(variants):
    import torch
    import tree_speculative_verify_tv_gb300 as tv
    small = workloads.config2(seed=71, B=4, H=6)
    big = workloads.random_batch(np.random.default_rng(72), [100, 60, 128, 7], 6, 128, 64,
                                 decay="scalar", depth_cap=10, max_depth=12, max_nodes=128)
    batches = (small, big)
    devs = [tv.DeviceBatch(b) for b in batches]
    streams = [torch.cuda.Stream() for _ in batches]
    refs = []
    for d, v, s in zip(devs, variants, streams):
        st, out = _once(d, v, s)
        assert st == 0
        refs.append(out)
    errors = []

    def worker(i):
        try:
            with torch.cuda.stream(streams[i]):
                for _ in range(40):
                    st, out = _once(devs[i], variants[i], streams[i])
                    if st != 0 or not torch.equal(out, refs[i]):
                        errors.append((i, st))
                        return
        except Exception as e:  # a TVError (for instance TV_ERR_CUDA) fails the test
            errors.append((i, repr(e)))

    threads = [threading.Thread(target=worker, args=(i,)) for i in range(2)]
    for t in threads:
        t.start()
    for t in threads:
        t.join()
    assert not errors, errors


def test_tree_attention_beside_verify_threads():
    import torch
    import tree_speculative_verify_tv_gb300 as tv
    b = workloads.config2(seed=73, B=4, H=6)
    a = workloads.attention_inputs(b, 8, 2, 128, [300] * b.B, P=384, seed=74)
    cu = lambda x: torch.from_numpy(np.ascontiguousarray(x)).cuda()
    args = [cu(b.node_offsets), cu(b.parent), cu(a["ctx_len"]), cu(a["q"]), cu(a["k_cache"]),
            cu(a["v_cache"]), cu(a["k_tree"]), cu(a["v_tree"])]
    out = torch.zeros((b.T, 8, 128), dtype=torch.float32, device="cuda")
    st = torch.zeros(1, dtype=torch.int32, device="cuda")
    s_att = torch.cuda.Stream()
    d = tv.DeviceBatch(b)
    s_ver = torch.cuda.Stream()

    def attention():
        with torch.cuda.stream(s_att):
            tv.tv_tree_attention(b.B, b.T, b.max_nodes, 8, 2, 128, 384, *args, a["scale"], out,
                                 None, 0, st, stream=s_att)
        s_att.synchronize()

    attention()
    ref = out.clone()
    ref_st, ref_v = _once(d, 0, s_ver)
    assert int(st[0]) == 0 and ref_st == 0
    errors = []

    def run_att():
        for _ in range(30):
            out.zero_()
            attention()
            if not torch.equal(out, ref) or int(st[0]) != 0:
                errors.append("attention")
                return

    def run_ver():
        for _ in range(30):
            s2, o2 = _once(d, 0, s_ver)
            if s2 != 0 or not torch.equal(o2, ref_v):
                errors.append("verify")
                return

    threads = [threading.Thread(target=run_att), threading.Thread(target=run_ver)]
    for t in threads:
        t.start()
    for t in threads:
        t.join()
    assert not errors, errors
