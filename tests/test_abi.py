"""C ABI checks that need no GPU: the library builds, loads, exports every
function include/treeverify.h declares, and rejects bad arguments on the host
(before any CUDA call)."""
import ctypes
import os
import re

import pytest

import tree_speculative_verify_tv_gb300 as tv

ROOT = os.path.dirname(os.path.dirname(os.path.abspath(__file__)))
HEADER = os.path.join(ROOT, "include", "treeverify.h")


@pytest.fixture(scope="module")
def lib():
    tv.build()
    return tv.load()


def declared_functions():
    src = open(HEADER).read()
    src = re.sub(r"/\*.*?\*/", "", src, flags=re.S)
    names = re.findall(r"^\s*(?:const\s+)?[A-Za-z_][A-Za-z0-9_]*\s*\*?\s*(tv_[a-z_]+)\s*\(",
                       src, flags=re.M)
    return sorted(set(names))


def test_header_declares_the_abi():
    names = declared_functions()
    assert {"tv_verify", "tv_verify_ex", "tv_verify_variant", "tv_accept_greedy", "tv_commit",
            "tv_accept_commit", "tv_commit_verify", "tv_accept_greedy_logits", "tv_status_string",
            "tv_version"} <= set(names)


def test_library_exports_every_declared_symbol(lib):
    for name in declared_functions():
        assert hasattr(lib, name), name
    assert set(declared_functions()) == set(tv.EXPORTED)


def test_version_and_status_strings(lib):
    assert tv.tv_version() == 1
    for code in range(9):
        s = tv.status_string(code)
        assert s.startswith("TV_"), s
    assert "unknown" in tv.status_string(99)


def test_header_constants_match_binding():
    src = open(HEADER).read()
    for name, val in (("TV_MAX_NODES", 256), ("TV_MAX_DEPTH", 32), ("TV_MAX_DIM", 256)):
        assert re.search(r"#define %s\s+%d" % (name, val), src)
    for name in ("TV_OK", "TV_ERR_NULL", "TV_ERR_SHAPE", "TV_ERR_DTYPE", "TV_ERR_ALIGN",
                 "TV_ERR_UNSUPPORTED", "TV_ERR_TREE", "TV_ERR_CUDA", "TV_ERR_TIMEOUT"):
        m = re.search(r"%s\s*=\s*(\d+)" % name, src)
        assert m and int(m.group(1)) == getattr(tv, name), name


# fake, aligned "device" addresses: every call below must fail before touching them
A = 0x10000
P = [A + 0x1000 * i for i in range(16)]


def prob(**kw):
    d = dict(B=2, H=3, dk=16, dv=16, total_nodes=5, max_nodes=4, max_depth=3,
             decay=tv.TV_DECAY_SCALAR, qkv_dtype=tv.TV_BF16, node_offsets=P[0], parent=P[1],
             depth=P[2])
    d.update(kw)
    return tv.make_problem(**d)


def verify_rc(p, **kw):
    args = dict(H0=P[3], q=P[4], k=P[5], v=P[6], g=P[7], out=P[8], dev_status=P[9])
    args.update(kw)
    return tv.tv_verify(p, args["H0"], args["q"], args["k"], args["v"], args["g"], args["out"],
                        args["dev_status"], stream=0, variant=kw.get("variant", 0), check=False)


@pytest.mark.parametrize("kw,code", [
    (dict(B=-1), tv.TV_ERR_SHAPE), (dict(H=0), tv.TV_ERR_SHAPE), (dict(dk=12), tv.TV_ERR_SHAPE),
    (dict(dv=0), tv.TV_ERR_SHAPE), (dict(dk=264), tv.TV_ERR_UNSUPPORTED),
    (dict(max_nodes=257), tv.TV_ERR_UNSUPPORTED), (dict(max_depth=33), tv.TV_ERR_UNSUPPORTED),
    (dict(max_nodes=0), tv.TV_ERR_SHAPE), (dict(decay=2), tv.TV_ERR_DTYPE),
    (dict(qkv_dtype=7), tv.TV_ERR_DTYPE), (dict(total_nodes=9), tv.TV_ERR_SHAPE),
    (dict(total_nodes=-1), tv.TV_ERR_SHAPE), (dict(node_offsets=None), tv.TV_ERR_NULL),
    (dict(parent=None), tv.TV_ERR_NULL), (dict(depth=None), tv.TV_ERR_NULL),
    (dict(node_offsets=A + 4), tv.TV_ERR_ALIGN),
])
def test_verify_rejects_bad_problem(lib, kw, code):
    assert verify_rc(prob(**kw)) == code


@pytest.mark.parametrize("field", ["H0", "q", "k", "v", "g", "out", "dev_status"])
def test_verify_rejects_null_and_misaligned_arrays(lib, field):
    assert verify_rc(prob(), **{field: None}) == tv.TV_ERR_NULL
    if field != "dev_status":
        assert verify_rc(prob(), **{field: P[10] + 8}) == tv.TV_ERR_ALIGN


def test_verify_forced_tc_on_unsupported_shape(lib):
    # fp32 q/k/v and dk=16 are outside the tensor-core kernel
    assert verify_rc(prob(qkv_dtype=tv.TV_F32), variant=tv.TV_VARIANT_TC) == tv.TV_ERR_UNSUPPORTED
    assert verify_rc(prob(), variant=9) == tv.TV_ERR_DTYPE


def test_variant_query_rejects_bad_problems(lib):
    assert tv.tv_verify_variant(prob(dk=12)) == -tv.TV_ERR_SHAPE
    assert tv.tv_verify_variant(prob(decay=5)) == -tv.TV_ERR_DTYPE
    assert tv.tv_verify_variant(prob(qkv_dtype=tv.TV_F32)) == tv.TV_VARIANT_SIMT
    assert tv.tv_verify_variant(prob(dk=96)) == tv.TV_VARIANT_SIMT


def test_support_query_matches_forced_launch_checks(lib):
    # fp32 q/k/v: only SIMT (and AUTO, which falls back to it)
    f32 = prob(qkv_dtype=tv.TV_F32)
    assert tv.tv_verify_supports(f32, tv.TV_VARIANT_SIMT) == 1
    assert tv.tv_verify_supports(f32, tv.TV_VARIANT_AUTO) == 1
    for v in (tv.TV_VARIANT_TC, tv.TV_VARIANT_TC_FUSED, tv.TV_VARIANT_TC_TILED):
        assert tv.tv_verify_supports(f32, v) == 0
        assert verify_rc(f32, variant=v) == tv.TV_ERR_UNSUPPORTED
    # the large-tree kernels take dk = dv = 128 only
    assert tv.tv_verify_supports(prob(dk=64, dv=64), tv.TV_VARIANT_TC_TILED) == 0
    assert tv.tv_verify_supports(prob(dk=12), tv.TV_VARIANT_TC) == -tv.TV_ERR_SHAPE
    assert tv.tv_verify_supports(prob(), 9) == -tv.TV_ERR_DTYPE


def test_fused_variant_limits(lib):
    # the fused kernels: bf16; scalar decay with dk and dv in {64, 128} and <= 32 nodes,
    # or per-channel decay with dk in {64, 128}, dv = 128 and <= 64 nodes, or <= 256
    # nodes of depth <= 16
    import torch
    if torch.cuda.is_available():
        # (the tensor-core kernels need the driver's tensor-map encoder)
        ok = prob(dk=128, dv=64, max_nodes=16, total_nodes=5)
        assert tv.tv_verify_supports(ok, tv.TV_VARIANT_TC_FUSED) == 1
        assert tv.tv_verify_variant(ok) == tv.TV_VARIANT_TC_FUSED
        assert tv.tv_verify_supports(prob(dk=128, dv=128, max_nodes=32),
                                     tv.TV_VARIANT_TC_FUSED) == 1
        # trees of 33..256 nodes keep the one-unit kernel
        assert tv.tv_verify_variant(prob(dk=128, dv=64, max_nodes=64)) == tv.TV_VARIANT_TC
        for dk in (64, 128):
            diag = prob(dk=dk, dv=128, max_nodes=64, decay=tv.TV_DECAY_DIAG)
            assert tv.tv_verify_supports(diag, tv.TV_VARIANT_TC_FUSED) == 1
            assert tv.tv_verify_variant(diag) == tv.TV_VARIANT_TC_FUSED
    for bad in (prob(dk=128, dv=64, max_nodes=33, total_nodes=5),
                prob(dk=128, dv=64, decay=tv.TV_DECAY_DIAG),
                prob(dk=128, dv=128, max_nodes=65, max_depth=17, decay=tv.TV_DECAY_DIAG),
                prob(dk=96, dv=64), prob(dk=128, dv=64, qkv_dtype=tv.TV_F32)):
        assert tv.tv_verify_supports(bad, tv.TV_VARIANT_TC_FUSED) == 0
        assert verify_rc(bad, variant=tv.TV_VARIANT_TC_FUSED) == tv.TV_ERR_UNSUPPORTED


def test_expire_wait_hook_only_with_the_fused_variant(lib):
    flag = tv.TV_VARIANT_TEST_EXPIRE_WAIT
    for v in (tv.TV_VARIANT_AUTO, tv.TV_VARIANT_SIMT, tv.TV_VARIANT_TC, tv.TV_VARIANT_TC_TILED):
        assert verify_rc(prob(dk=128, dv=64), variant=v | flag) == tv.TV_ERR_UNSUPPORTED
    assert verify_rc(prob(dk=128, dv=64), variant=0x200) == tv.TV_ERR_DTYPE
    src = open(HEADER).read()
    m = re.search(r"#define TV_VARIANT_TEST_EXPIRE_WAIT\s+(0x[0-9a-fA-F]+)", src)
    assert m and int(m.group(1), 16) == flag


def test_workspace_bytes_is_zero(lib):
    # every verify kernel keeps its transient data in shared and tensor memory
    for p in (prob(), prob(dk=128, dv=64, max_nodes=16), prob(dk=128, dv=128, max_nodes=256),
              prob(decay=tv.TV_DECAY_DIAG), prob(dk=12)):
        assert tv.tv_workspace_bytes(p) == 0


def test_empty_batches_are_no_ops(lib):
    assert verify_rc(prob(B=0, total_nodes=0)) == tv.TV_OK
    assert verify_rc(prob(total_nodes=0)) == tv.TV_OK
    rc = tv.tv_accept_greedy(0, 0, 4, 3, P[0], P[1], P[2], P[3], P[4], P[5], P[6], P[7], P[8],
                             stream=0, check=False)
    assert rc == tv.TV_OK


def test_accept_rejects_bad_arguments(lib):
    def rc(**kw):
        a = dict(B=2, T=5, mn=4, md=3, offs=P[0], par=P[1], dr=P[2], tg=P[3], root=P[4],
                 ln=P[5], path=P[6], bonus=P[7], st=P[8])
        a.update(kw)
        return tv.tv_accept_greedy(a["B"], a["T"], a["mn"], a["md"], a["offs"], a["par"],
                                   a["dr"], a["tg"], a["root"], a["ln"], a["path"], a["bonus"],
                                   a["st"], stream=0, check=False)
    assert rc(B=-1) == tv.TV_ERR_SHAPE
    assert rc(md=0) == tv.TV_ERR_SHAPE
    assert rc(md=40) == tv.TV_ERR_UNSUPPORTED
    assert rc(T=100) == tv.TV_ERR_SHAPE
    assert rc(root=None) == tv.TV_ERR_NULL
    assert rc(dr=None) == tv.TV_ERR_NULL
    assert rc(st=None) == tv.TV_ERR_NULL
    assert rc(path=P[6] + 4) == tv.TV_ERR_ALIGN


def test_commit_rejects_bad_arguments(lib):
    def rc(p=None, **kw):
        a = dict(H0=P[3], g=P[7], k=P[5], v=P[6], path=P[10], ln=P[11], Hn=P[12], st=P[9])
        a.update(kw)
        return tv.tv_commit(p or prob(), a["H0"], a["g"], a["k"], a["v"], a["path"], a["ln"],
                            a["Hn"], a["st"], stream=0, check=False)
    assert rc(prob(dv=7)) == tv.TV_ERR_SHAPE
    assert rc(path=None) == tv.TV_ERR_NULL
    assert rc(Hn=None) == tv.TV_ERR_NULL
    assert rc(Hn=P[3] + 16) == tv.TV_ERR_SHAPE      # overlaps H0 without being H0
    assert rc(Hn=P[12] + 4) == tv.TV_ERR_ALIGN


def test_accept_commit_rejects_bad_arguments(lib):
    def rc(p=None, **kw):
        a = dict(H0=P[3], g=P[7], k=P[5], v=P[6], dr=P[13], tg=P[14], root=P[15], ln=P[11],
                 path=P[10], bonus=P[4], Hn=P[12], st=P[9])
        a.update(kw)
        return tv.tv_accept_commit(p or prob(), a["H0"], a["g"], a["k"], a["v"], a["dr"], a["tg"],
                                   a["root"], a["ln"], a["path"], a["bonus"], a["Hn"], a["st"],
                                   stream=0, check=False)
    assert rc(prob(dk=12)) == tv.TV_ERR_SHAPE
    assert rc(dr=None) == tv.TV_ERR_NULL
    assert rc(bonus=None) == tv.TV_ERR_NULL
    assert rc(Hn=P[3] + 16) == tv.TV_ERR_SHAPE
    assert rc(root=P[15] + 4) == tv.TV_ERR_ALIGN
    assert rc(prob(B=0, total_nodes=0)) == tv.TV_OK


def pend(**kw):
    d = dict(total_nodes=5, max_nodes=4, max_depth=3, node_offsets=P[0], parent=P[1], g=P[7],
             k=P[5], v=P[6], path=P[10], accept_len=P[11])
    d.update(kw)
    return tv.make_pending(**d)


def test_commit_verify_rejects_bad_arguments(lib):
    def rc(p=None, pe="default", **kw):
        a = dict(H=P[3], q=P[4], k=P[5], v=P[6], g=P[7], out=P[8], st=P[9])
        a.update(kw)
        pe = pend() if pe == "default" else pe
        return tv.tv_commit_verify(p or prob(), pe, a["H"], a["q"], a["k"], a["v"], a["g"],
                                   a["out"], a["st"], stream=0, check=False)
    assert rc(prob(dk=12)) == tv.TV_ERR_SHAPE
    assert rc(prob(depth=None)) == tv.TV_ERR_NULL
    assert rc(H=None) == tv.TV_ERR_NULL
    assert rc(st=None) == tv.TV_ERR_NULL
    assert rc(q=None) == tv.TV_ERR_NULL
    assert rc(pe=pend(path=None)) == tv.TV_ERR_NULL
    assert rc(pe=pend(accept_len=None)) == tv.TV_ERR_NULL
    assert rc(pe=pend(k=None)) == tv.TV_ERR_NULL
    assert rc(pe=pend(max_depth=0)) == tv.TV_ERR_SHAPE
    assert rc(pe=pend(max_depth=33)) == tv.TV_ERR_UNSUPPORTED
    assert rc(pe=pend(max_nodes=300)) == tv.TV_ERR_UNSUPPORTED
    assert rc(pe=pend(total_nodes=9)) == tv.TV_ERR_SHAPE
    assert rc(pe=pend(path=P[10] + 4)) == tv.TV_ERR_ALIGN
    assert rc(pe=pend(v=P[6] + 8)) == tv.TV_ERR_ALIGN
    assert rc(H=P[3] + 4) == tv.TV_ERR_ALIGN
    assert rc(g=P[7] + 8) == tv.TV_ERR_ALIGN
    assert rc(prob(B=0, total_nodes=0), pe=pend(total_nodes=0)) == tv.TV_OK
    # without a pending commit the call is tv_verify and checks like it
    assert rc(pe=None, q=None) == tv.TV_ERR_NULL
    assert rc(prob(dv=0), pe=None) == tv.TV_ERR_SHAPE


def test_accept_logits_rejects_bad_arguments(lib):
    def rc(**kw):
        a = dict(B=2, T=5, mn=4, md=3, V=32000, offs=P[0], par=P[1], dr=P[2], rl=P[3], nl=P[4],
                 ra=P[5], ta=P[6], ln=P[7], path=P[8], bonus=P[9], st=P[10])
        a.update(kw)
        return tv.tv_accept_greedy_logits(a["B"], a["T"], a["mn"], a["md"], a["V"], a["offs"],
                                          a["par"], a["dr"], a["rl"], a["nl"], a["ra"], a["ta"],
                                          a["ln"], a["path"], a["bonus"], a["st"], stream=0,
                                          check=False)
    assert rc(V=0) == tv.TV_ERR_SHAPE
    assert rc(B=-1) == tv.TV_ERR_SHAPE
    assert rc(md=33) == tv.TV_ERR_UNSUPPORTED
    assert rc(T=9) == tv.TV_ERR_SHAPE
    assert rc(rl=None) == tv.TV_ERR_NULL
    assert rc(nl=None) == tv.TV_ERR_NULL
    assert rc(st=None) == tv.TV_ERR_NULL
    assert rc(ra=None) == tv.TV_ERR_NULL
    assert rc(ta=None) == tv.TV_ERR_NULL
    assert rc(nl=P[4] + 2) == tv.TV_ERR_ALIGN
    assert rc(ta=P[6] + 4) == tv.TV_ERR_ALIGN
    assert rc(B=0, T=0) == tv.TV_OK


def test_serial_rejects_bad_arguments(lib):
    p = prob()
    need = tv.tv_verify_serial_workspace_bytes(p)
    assert need == 2 * 3 * 4 * 16 * 16 * 4
    assert tv.tv_verify_serial_workspace_bytes(prob(dk=12)) == 0

    def rc(pp=None, ws=P[11], nbytes=None, **kw):
        a = dict(H0=P[3], q=P[4], k=P[5], v=P[6], g=P[7], out=P[8], st=P[9])
        a.update(kw)
        return tv.tv_verify_serial(pp or p, a["H0"], a["q"], a["k"], a["v"], a["g"], a["out"], ws,
                                   need if nbytes is None else nbytes, a["st"], stream=0,
                                   check=False)
    assert rc(ws=None) == tv.TV_ERR_NULL
    assert rc(nbytes=need - 1) == tv.TV_ERR_SHAPE
    assert rc(ws=P[11] + 4) == tv.TV_ERR_ALIGN
    assert rc(q=None) == tv.TV_ERR_NULL
    assert rc(prob(dv=12)) == tv.TV_ERR_SHAPE
    assert rc(prob(total_nodes=0)) == tv.TV_OK


def test_serial_static_rejects_problems_beyond_its_scratch(lib):
    # per-node states of 4 x 8 units x 256 nodes x 128 x 128 fp32 = 512 MiB > 16 MiB
    big = prob(B=4, H=8, dk=128, dv=128, total_nodes=4, max_nodes=256, max_depth=32)
    assert tv.tv_verify_serial_workspace_bytes(big) > tv.TV_SERIAL_STATIC_BYTES
    rc = tv.tv_verify_serial_static(big, P[3], P[4], P[5], P[6], P[7], P[8], P[9], stream=0,
                                    check=False)
    assert rc == tv.TV_ERR_UNSUPPORTED
    assert tv.tv_verify_serial_static(prob(dk=12), *P[3:10], stream=0,
                                      check=False) == tv.TV_ERR_SHAPE
    assert tv.tv_verify_serial_static(prob(), P[3], P[4], P[5], P[6], P[7], P[8], None,
                                      stream=0, check=False) == tv.TV_ERR_NULL


def test_accept_stochastic_rejects_bad_arguments(lib):
    def rc(**kw):
        a = dict(B=2, T=5, mn=4, md=3, V=100, offs=P[0], par=P[1], dr=P[2], rp=P[3], np_=P[4],
                 rq=P[5], nq=P[6], ua=P[7], ub=P[8], ln=P[9], path=P[10], bonus=P[11], st=P[12])
        a.update(kw)
        return tv.tv_accept_stochastic(a["B"], a["T"], a["mn"], a["md"], a["V"], a["offs"],
                                       a["par"], a["dr"], a["rp"], a["np_"], a["rq"], a["nq"],
                                       a["ua"], a["ub"], a["ln"], a["path"], a["bonus"], a["st"],
                                       stream=0, check=False)
    assert rc(V=0) == tv.TV_ERR_SHAPE
    assert rc(md=40) == tv.TV_ERR_UNSUPPORTED
    assert rc(rq=None) == tv.TV_ERR_NULL
    assert rc(ua=None) == tv.TV_ERR_NULL
    assert rc(ub=P[8] + 8) == tv.TV_ERR_ALIGN
    assert rc(B=0, T=0) == tv.TV_OK


def test_tree_attention_rejects_bad_arguments(lib):
    def rc(**kw):
        a = dict(B=2, T=5, mn=4, H=8, Hkv=2, d=128, P_=64, offs=P[0], par=P[1], ctx=P[2], q=P[3],
                 kc=P[4], vc=P[5], kt=P[6], vt=P[7], scale=0.1, out=P[8], ws=None, wsb=0,
                 st=P[9])
        a.update(kw)
        return tv.tv_tree_attention(a["B"], a["T"], a["mn"], a["H"], a["Hkv"], a["d"], a["P_"],
                                    a["offs"], a["par"], a["ctx"], a["q"], a["kc"], a["vc"],
                                    a["kt"], a["vt"], a["scale"], a["out"], a["ws"], a["wsb"],
                                    a["st"], stream=0, check=False)
    assert rc(H=6, Hkv=4) == tv.TV_ERR_SHAPE         # H not a multiple of Hkv
    assert rc(H=6, Hkv=2) == tv.TV_ERR_UNSUPPORTED   # a group of 3 query heads
    assert rc(d=96) == tv.TV_ERR_UNSUPPORTED
    assert rc(mn=300) == tv.TV_ERR_UNSUPPORTED
    assert rc(T=9) == tv.TV_ERR_SHAPE                # T > B * max_nodes
    assert rc(P_=0) == tv.TV_ERR_SHAPE
    assert rc(scale=float("nan")) == tv.TV_ERR_SHAPE
    assert rc(scale=float("inf")) == tv.TV_ERR_SHAPE
    assert rc(scale=0.0) == tv.TV_ERR_SHAPE
    assert rc(scale=-0.1) == tv.TV_ERR_SHAPE
    assert rc(q=None) == tv.TV_ERR_NULL
    assert rc(ctx=None) == tv.TV_ERR_NULL
    assert rc(kt=P[6] + 4) == tv.TV_ERR_ALIGN
    assert rc(ws=P[10] + 8, wsb=1024) == tv.TV_ERR_ALIGN
    assert rc(B=0, T=0) == tv.TV_OK
    assert rc(T=0, par=None, q=None, kt=None, vt=None, out=None) == tv.TV_OK


def test_build_tree_rejects_bad_arguments(lib):
    def rc(**kw):
        a = dict(B=2, C=8, cap=8, n=64, m=P[0], cost=None, par=P[1], tok=P[2], rho=P[3], cnt=P[4])
        a.update(kw)
        return tv.tv_build_tree(a["B"], a["C"], a["cap"], a["n"], a["m"], a["cost"], a["par"],
                                a["tok"], a["rho"], a["cnt"], stream=0, check=False)
    assert rc(C=0) == tv.TV_ERR_SHAPE
    assert rc(C=33) == tv.TV_ERR_SHAPE
    assert rc(cap=33) == tv.TV_ERR_SHAPE
    assert rc(n=257) == tv.TV_ERR_SHAPE
    assert rc(B=-1) == tv.TV_ERR_SHAPE
    assert rc(m=None) == tv.TV_ERR_NULL
    assert rc(cnt=None) == tv.TV_ERR_NULL
    assert rc(rho=P[3] + 8) == tv.TV_ERR_ALIGN
    assert rc(cost=P[5] + 8) == tv.TV_ERR_ALIGN
    assert rc(B=0) == tv.TV_OK


def test_binding_fails_loudly_without_library(tmp_path):
    with pytest.raises(RuntimeError, match="not built"):
        tv.load(str(tmp_path / "missing.so"))


def test_accept_commit_verify_rejects_bad_arguments(lib):
    def rc(p=None, pe="default", **kw):
        a = dict(dr=P[13], tg=P[14], root=P[15], ln=P[11], path=P[10], bonus=P[12], H=P[3],
                 q=P[4], k=P[5], v=P[6], g=P[7], out=P[8], st=P[9])
        a.update(kw)
        pe = pend() if pe == "default" else pe
        return tv.tv_accept_commit_verify(p or prob(), pe, a["dr"], a["tg"], a["root"], a["ln"],
                                          a["path"], a["bonus"], a["H"], a["q"], a["k"], a["v"],
                                          a["g"], a["out"], a["st"], stream=0, check=False)
    assert rc(prob(dk=12)) == tv.TV_ERR_SHAPE
    assert rc(pe=None) == tv.TV_ERR_NULL
    assert rc(dr=None) == tv.TV_ERR_NULL
    assert rc(bonus=None) == tv.TV_ERR_NULL
    assert rc(pe=pend(max_depth=40)) == tv.TV_ERR_UNSUPPORTED
    assert rc(pe=pend(total_nodes=100)) == tv.TV_ERR_SHAPE
    assert rc(path=P[10] + 4) == tv.TV_ERR_ALIGN
    assert rc(prob(B=0, total_nodes=0), pe=pend(total_nodes=0)) == tv.TV_OK
