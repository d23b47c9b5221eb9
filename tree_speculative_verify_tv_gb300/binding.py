"""Thin ctypes binding of libtreeverify (include/treeverify.h).

Same names as the C ABI; the functions only marshal arguments (tensor data
pointers, sizes, the current CUDA stream) and return or check the status.
Every computation runs in the library's CUDA kernels; there is no fallback:
if libtreeverify.so is missing or cannot be loaded, importing the binding's
calls raises.

Arguments may be torch tensors (their data_ptr() is passed) or plain integer
device addresses.
"""
from __future__ import annotations

import ctypes
import os
import threading
from typing import Optional

PKG = os.path.dirname(os.path.abspath(__file__))
LIB_PATH = os.path.join(PKG, "libtreeverify.so")

TV_OK, TV_ERR_NULL, TV_ERR_SHAPE, TV_ERR_DTYPE, TV_ERR_ALIGN = 0, 1, 2, 3, 4
TV_ERR_UNSUPPORTED, TV_ERR_TREE, TV_ERR_CUDA, TV_ERR_TIMEOUT = 5, 6, 7, 8
TV_DECAY_SCALAR, TV_DECAY_DIAG = 0, 1
TV_BF16, TV_F32 = 0, 1
TV_VARIANT_AUTO, TV_VARIANT_SIMT, TV_VARIANT_TC, TV_VARIANT_TC_FUSED = 0, 1, 2, 3
TV_VARIANT_TC_TILED = 4
TV_VARIANT_TEST_EXPIRE_WAIT = 0x100
TV_MAX_NODES, TV_MAX_DEPTH, TV_MAX_DIM = 256, 32, 256
TV_SERIAL_STATIC_BYTES = 16 << 20

EXPORTED = ("tv_verify", "tv_verify_ex", "tv_verify_variant", "tv_verify_supports",
            "tv_workspace_bytes",
            "tv_accept_greedy", "tv_commit",
            "tv_accept_commit", "tv_commit_verify", "tv_accept_commit_verify",
            "tv_accept_greedy_logits", "tv_verify_serial",
            "tv_verify_serial_workspace_bytes", "tv_verify_serial_static", "tv_build_tree",
            "tv_accept_stochastic", "tv_tree_attention", "tv_tree_attention_workspace_bytes",
            "tv_status_string", "tv_version")


class tv_problem(ctypes.Structure):
    _fields_ = [("B", ctypes.c_int32), ("H", ctypes.c_int32), ("dk", ctypes.c_int32),
                ("dv", ctypes.c_int32), ("total_nodes", ctypes.c_int32),
                ("max_nodes", ctypes.c_int32), ("max_depth", ctypes.c_int32),
                ("decay", ctypes.c_int32), ("qkv_dtype", ctypes.c_int32),
                ("node_offsets", ctypes.c_void_p), ("parent", ctypes.c_void_p),
                ("depth", ctypes.c_void_p)]


class tv_pending(ctypes.Structure):
    _fields_ = [("total_nodes", ctypes.c_int32), ("max_nodes", ctypes.c_int32),
                ("max_depth", ctypes.c_int32), ("node_offsets", ctypes.c_void_p),
                ("parent", ctypes.c_void_p), ("g", ctypes.c_void_p), ("k", ctypes.c_void_p),
                ("v", ctypes.c_void_p), ("path", ctypes.c_void_p),
                ("accept_len", ctypes.c_void_p)]


class TVError(RuntimeError):
    def __init__(self, code: int, what: str):
        self.code = code
        super().__init__("%s: %s" % (what, status_string(code)))


_lock = threading.Lock()
_lib = None


def load(path: Optional[str] = None):
    """Load libtreeverify.so (raises if it has not been built)."""
    global _lib
    with _lock:
        if _lib is not None and path is None:
            return _lib
        p = path or LIB_PATH
        if not os.path.exists(p):
            raise RuntimeError("libtreeverify.so is not built (%s); run "
                               "tree_speculative_verify_tv_gb300.build()" % p)
        L = ctypes.CDLL(p)
        vp, i32 = ctypes.c_void_p, ctypes.c_int32
        P = ctypes.POINTER(tv_problem)
        L.tv_verify.argtypes = [P, vp, vp, vp, vp, vp, vp, vp, vp]
        L.tv_verify_ex.argtypes = [P, vp, vp, vp, vp, vp, vp, vp, vp, i32]
        L.tv_accept_greedy.argtypes = [i32, i32, i32, i32, vp, vp, vp, vp, vp, vp, vp, vp, vp, vp]
        L.tv_commit.argtypes = [P, vp, vp, vp, vp, vp, vp, vp, vp, vp]
        L.tv_accept_commit.argtypes = [P, vp, vp, vp, vp, vp, vp, vp, vp, vp, vp, vp, vp, vp]
        L.tv_commit_verify.argtypes = [P, ctypes.POINTER(tv_pending), vp, vp, vp, vp, vp, vp, vp,
                                       vp]
        L.tv_accept_commit_verify.argtypes = [P, ctypes.POINTER(tv_pending)] + [vp] * 14
        L.tv_accept_greedy_logits.argtypes = [i32, i32, i32, i32, i32] + [vp] * 12
        L.tv_verify_serial.argtypes = [P] + [vp] * 7 + [ctypes.c_size_t, vp, vp]
        L.tv_verify_serial_static.argtypes = [P] + [vp] * 8
        L.tv_build_tree.argtypes = [i32] * 4 + [vp] * 7
        L.tv_accept_stochastic.argtypes = [i32] * 5 + [vp] * 14
        L.tv_tree_attention.argtypes = ([i32] * 7 + [vp] * 8 + [ctypes.c_float, vp, vp,
                                                                ctypes.c_size_t, vp, vp])
        L.tv_tree_attention_workspace_bytes.argtypes = [i32] * 7
        L.tv_tree_attention_workspace_bytes.restype = ctypes.c_size_t
        L.tv_verify_serial_workspace_bytes.argtypes = [P]
        L.tv_verify_serial_workspace_bytes.restype = ctypes.c_size_t
        L.tv_workspace_bytes.argtypes = [P]
        L.tv_workspace_bytes.restype = ctypes.c_size_t
        for f in (L.tv_verify, L.tv_verify_ex, L.tv_accept_greedy, L.tv_commit,
                  L.tv_accept_commit, L.tv_commit_verify, L.tv_accept_commit_verify,
                  L.tv_accept_greedy_logits,
                  L.tv_verify_serial, L.tv_verify_serial_static, L.tv_build_tree,
                  L.tv_accept_stochastic, L.tv_tree_attention):
            f.restype = ctypes.c_int32
        L.tv_status_string.argtypes = [i32]
        L.tv_status_string.restype = ctypes.c_char_p
        L.tv_version.argtypes = []
        L.tv_version.restype = i32
        L.tv_verify_variant.argtypes = [P]
        L.tv_verify_variant.restype = i32
        L.tv_verify_supports.argtypes = [P, i32]
        L.tv_verify_supports.restype = i32
        if path is None:
            _lib = L
        return L


def _ptr(x) -> Optional[int]:
    if x is None:
        return None
    if isinstance(x, int):
        return x
    return x.data_ptr()


def _stream(stream) -> Optional[int]:
    if stream is None:
        import torch
        return torch.cuda.current_stream().cuda_stream
    if isinstance(stream, int):
        return stream
    return stream.cuda_stream


def status_string(code: int) -> str:
    return load().tv_status_string(int(code)).decode()


tv_status_string = status_string


def tv_version() -> int:
    return load().tv_version()


def tv_verify_variant(problem: tv_problem) -> int:
    """Kernel tv_verify would choose (a TV_VARIANT_* value), or -status."""
    return load().tv_verify_variant(ctypes.byref(problem))


def tv_verify_supports(problem: tv_problem, variant: int) -> int:
    """1 if tv_verify_ex takes `variant` for this problem, 0 if it would report
    TV_ERR_UNSUPPORTED, or -status for an invalid problem or variant."""
    return load().tv_verify_supports(ctypes.byref(problem), int(variant))


def make_problem(B, H, dk, dv, total_nodes, max_nodes, max_depth, decay, qkv_dtype,
                 node_offsets, parent, depth) -> tv_problem:
    """tv_problem from sizes and (device) tree arrays; keeps no reference to tensors."""
    return tv_problem(int(B), int(H), int(dk), int(dv), int(total_nodes), int(max_nodes),
                      int(max_depth), int(decay), int(qkv_dtype), _ptr(node_offsets),
                      _ptr(parent), _ptr(depth))


def _check(code: int, what: str, check: bool) -> int:
    if check and code != TV_OK:
        raise TVError(code, what)
    return code


def tv_verify(problem: tv_problem, H0, q, k, v, g, out, dev_status, stream=None,
              variant: int = TV_VARIANT_AUTO, check: bool = True) -> int:
    rc = load().tv_verify_ex(ctypes.byref(problem), _ptr(H0), _ptr(q), _ptr(k), _ptr(v), _ptr(g),
                             _ptr(out), _ptr(dev_status), _stream(stream), int(variant))
    return _check(rc, "tv_verify", check)


def tv_workspace_bytes(problem: tv_problem) -> int:
    """Device workspace tv_verify needs: always 0 (shared and tensor memory only)."""
    return int(load().tv_workspace_bytes(ctypes.byref(problem)))


def tv_verify_serial_workspace_bytes(problem: tv_problem) -> int:
    return int(load().tv_verify_serial_workspace_bytes(ctypes.byref(problem)))


def tv_verify_serial(problem: tv_problem, H0, q, k, v, g, out, workspace, workspace_bytes,
                     dev_status, stream=None, check: bool = True) -> int:
    rc = load().tv_verify_serial(ctypes.byref(problem), _ptr(H0), _ptr(q), _ptr(k), _ptr(v),
                                 _ptr(g), _ptr(out), _ptr(workspace), int(workspace_bytes),
                                 _ptr(dev_status), _stream(stream))
    return _check(rc, "tv_verify_serial", check)


def tv_verify_serial_static(problem: tv_problem, H0, q, k, v, g, out, dev_status, stream=None,
                            check: bool = True) -> int:
    """tv_verify_serial with the library's built-in scratch array (no workspace)."""
    rc = load().tv_verify_serial_static(ctypes.byref(problem), _ptr(H0), _ptr(q), _ptr(k),
                                        _ptr(v), _ptr(g), _ptr(out), _ptr(dev_status),
                                        _stream(stream))
    return _check(rc, "tv_verify_serial_static", check)


def tv_accept_stochastic(B, total_nodes, max_nodes, max_depth, vocab, node_offsets, parent,
                         draft_tokens, root_p, node_p, root_q, node_q, u_accept, u_bonus,
                         accept_len, path, bonus, dev_status, stream=None,
                         check: bool = True) -> int:
    rc = load().tv_accept_stochastic(int(B), int(total_nodes), int(max_nodes), int(max_depth),
                                     int(vocab), _ptr(node_offsets), _ptr(parent),
                                     _ptr(draft_tokens), _ptr(root_p), _ptr(node_p), _ptr(root_q),
                                     _ptr(node_q), _ptr(u_accept), _ptr(u_bonus),
                                     _ptr(accept_len), _ptr(path), _ptr(bonus), _ptr(dev_status),
                                     _stream(stream))
    return _check(rc, "tv_accept_stochastic", check)


def tv_tree_attention_workspace_bytes(B, total_nodes, max_nodes, H, Hkv, d, P) -> int:
    return int(load().tv_tree_attention_workspace_bytes(int(B), int(total_nodes), int(max_nodes),
                                                        int(H), int(Hkv), int(d), int(P)))


def tv_tree_attention(B, total_nodes, max_nodes, H, Hkv, d, P, node_offsets, parent, ctx_len, q,
                      k_cache, v_cache, k_tree, v_tree, scale, out, workspace=None,
                      workspace_bytes=0, dev_status=None, stream=None, check: bool = True) -> int:
    rc = load().tv_tree_attention(int(B), int(total_nodes), int(max_nodes), int(H), int(Hkv),
                                  int(d), int(P), _ptr(node_offsets), _ptr(parent), _ptr(ctx_len),
                                  _ptr(q), _ptr(k_cache), _ptr(v_cache), _ptr(k_tree),
                                  _ptr(v_tree), float(scale), _ptr(out), _ptr(workspace),
                                  int(workspace_bytes), _ptr(dev_status), _stream(stream))
    return _check(rc, "tv_tree_attention", check)


def tv_build_tree(B, C, depth_cap, n, marginals, cost, parent, token, rho, count, stream=None,
                  check: bool = True) -> int:
    rc = load().tv_build_tree(int(B), int(C), int(depth_cap), int(n), _ptr(marginals), _ptr(cost),
                              _ptr(parent), _ptr(token), _ptr(rho), _ptr(count), _stream(stream))
    return _check(rc, "tv_build_tree", check)


def tv_accept_greedy(B, total_nodes, max_nodes, max_depth, node_offsets, parent, draft_tokens,
                     target_argmax, root_argmax, accept_len, path, bonus, dev_status,
                     stream=None, check: bool = True) -> int:
    rc = load().tv_accept_greedy(int(B), int(total_nodes), int(max_nodes), int(max_depth),
                                 _ptr(node_offsets), _ptr(parent), _ptr(draft_tokens),
                                 _ptr(target_argmax), _ptr(root_argmax), _ptr(accept_len),
                                 _ptr(path), _ptr(bonus), _ptr(dev_status), _stream(stream))
    return _check(rc, "tv_accept_greedy", check)


def tv_accept_greedy_logits(B, total_nodes, max_nodes, max_depth, vocab, node_offsets, parent,
                            draft_tokens, root_logits, node_logits, root_argmax, target_argmax,
                            accept_len, path, bonus, dev_status, stream=None,
                            check: bool = True) -> int:
    rc = load().tv_accept_greedy_logits(int(B), int(total_nodes), int(max_nodes), int(max_depth),
                                        int(vocab), _ptr(node_offsets), _ptr(parent),
                                        _ptr(draft_tokens), _ptr(root_logits), _ptr(node_logits),
                                        _ptr(root_argmax), _ptr(target_argmax), _ptr(accept_len),
                                        _ptr(path), _ptr(bonus), _ptr(dev_status),
                                        _stream(stream))
    return _check(rc, "tv_accept_greedy_logits", check)


def tv_commit(problem: tv_problem, H0, g, k, v, path, accept_len, H_new, dev_status, stream=None,
              check: bool = True) -> int:
    rc = load().tv_commit(ctypes.byref(problem), _ptr(H0), _ptr(g), _ptr(k), _ptr(v), _ptr(path),
                          _ptr(accept_len), _ptr(H_new), _ptr(dev_status), _stream(stream))
    return _check(rc, "tv_commit", check)


def tv_accept_commit(problem: tv_problem, H0, g, k, v, draft_tokens, target_argmax, root_argmax,
                     accept_len, path, bonus, H_new, dev_status, stream=None,
                     check: bool = True) -> int:
    rc = load().tv_accept_commit(ctypes.byref(problem), _ptr(H0), _ptr(g), _ptr(k), _ptr(v),
                                 _ptr(draft_tokens), _ptr(target_argmax), _ptr(root_argmax),
                                 _ptr(accept_len), _ptr(path), _ptr(bonus), _ptr(H_new),
                                 _ptr(dev_status), _stream(stream))
    return _check(rc, "tv_accept_commit", check)


def make_pending(total_nodes, max_nodes, max_depth, node_offsets, parent, g, k, v, path,
                 accept_len) -> tv_pending:
    """tv_pending from sizes and device arrays; keeps no reference to tensors."""
    return tv_pending(int(total_nodes), int(max_nodes), int(max_depth), _ptr(node_offsets),
                      _ptr(parent), _ptr(g), _ptr(k), _ptr(v), _ptr(path), _ptr(accept_len))


def tv_commit_verify(problem: tv_problem, pending: Optional[tv_pending], H, q, k, v, g, out,
                     dev_status, stream=None, check: bool = True) -> int:
    pp = ctypes.byref(pending) if pending is not None else None
    rc = load().tv_commit_verify(ctypes.byref(problem), pp, _ptr(H), _ptr(q), _ptr(k), _ptr(v),
                                 _ptr(g), _ptr(out), _ptr(dev_status), _stream(stream))
    return _check(rc, "tv_commit_verify", check)


def tv_accept_commit_verify(problem: tv_problem, prev: Optional[tv_pending], draft_tokens,
                            target_argmax, root_argmax, accept_len, path, bonus, H, q, k, v, g,
                            out, dev_status, stream=None, check: bool = True) -> int:
    pp = ctypes.byref(prev) if prev is not None else None
    rc = load().tv_accept_commit_verify(ctypes.byref(problem), pp,
                                        _ptr(draft_tokens), _ptr(target_argmax),
                                        _ptr(root_argmax), _ptr(accept_len), _ptr(path),
                                        _ptr(bonus), _ptr(H), _ptr(q), _ptr(k), _ptr(v), _ptr(g),
                                        _ptr(out), _ptr(dev_status), _stream(stream))
    return _check(rc, "tv_accept_commit_verify", check)


# ---------------------------------------------------------------- device batches


class DeviceBatch:
    """Device copies of one batch's inputs and output buffers (torch tensors).

    `host` is any object with the fields of a packed batch (B, H, dk, dv, decay,
    qkv_dtype, node_offsets, parent, depth, q, k, v, g, H0, draft, target,
    root_argmax, max_nodes, max_depth); bf16 arrays arrive as uint16 bit patterns.
    """

    def __init__(self, host, device="cuda", pin: bool = False):
        import numpy as np
        import torch

        def t(a, dtype=None):
            x = torch.from_numpy(np.ascontiguousarray(a))
            if dtype is not None:
                x = x.view(dtype)
            if pin:
                return x.pin_memory()
            return x.to(device)

        bf = host.qkv_dtype == "bf16"
        self.B, self.H, self.dk, self.dv = host.B, host.H, host.dk, host.dv
        self.T = int(host.node_offsets[-1])
        self.max_nodes, self.max_depth = int(host.max_nodes), int(host.max_depth)
        self.decay = TV_DECAY_DIAG if host.decay == "diag" else TV_DECAY_SCALAR
        self.qkv_dtype = TV_BF16 if bf else TV_F32
        self.node_offsets = t(host.node_offsets.astype(np.int32))
        self.parent = t(host.parent.astype(np.int32))
        self.depth = t(host.depth.astype(np.int32))
        qdt = torch.bfloat16 if bf else None
        self.q, self.k, self.v = t(host.q, qdt), t(host.k, qdt), t(host.v, qdt)
        self.g = t(host.g.astype(np.float32))
        self.H0 = t(host.H0.astype(np.float32))
        self.draft = t(host.draft.astype(np.int32))
        self.target = t(host.target.astype(np.int32))
        self.root_argmax = t(host.root_argmax.astype(np.int32))
        dev = "cpu" if pin else device
        mk = (lambda *s, dtype: torch.empty(*s, dtype=dtype, device=dev).pin_memory()) if pin \
            else (lambda *s, dtype: torch.empty(*s, dtype=dtype, device=dev))
        self.out = mk(max(self.T, 1), self.H, self.dv, dtype=torch.float32)
        self.H_new = mk(self.B, self.H, self.dk, self.dv, dtype=torch.float32)
        self.accept_len = mk(max(self.B, 1), dtype=torch.int32)
        self.path = mk(max(self.B, 1), self.max_depth, dtype=torch.int32)
        self.bonus = mk(max(self.B, 1), dtype=torch.int32)
        self.status = torch.zeros(4, dtype=torch.int32, device=dev)
        if pin:
            self.status = self.status.pin_memory()

    def variant(self) -> int:
        return tv_verify_variant(self.problem())

    def problem(self) -> tv_problem:
        return make_problem(self.B, self.H, self.dk, self.dv, self.T, self.max_nodes,
                            self.max_depth, self.decay, self.qkv_dtype, self.node_offsets,
                            self.parent, self.depth)

    # one step of the hot path: verify, greedy accept, commit
    def verify(self, stream=None, variant=TV_VARIANT_AUTO, check=True):
        return tv_verify(self.problem(), self.H0, self.q, self.k, self.v, self.g, self.out,
                         self.status, stream, variant, check)

    def verify_serial(self, workspace, stream=None, check=True):
        """tv_verify_serial into self.out; `workspace` is a device tensor of at least
        tv_verify_serial_workspace_bytes bytes."""
        return tv_verify_serial(self.problem(), self.H0, self.q, self.k, self.v, self.g,
                                self.out, workspace, workspace.numel() * workspace.element_size(),
                                self.status, stream, check)

    def accept(self, stream=None, check=True):
        return tv_accept_greedy(self.B, self.T, self.max_nodes, self.max_depth, self.node_offsets,
                                self.parent, self.draft, self.target, self.root_argmax,
                                self.accept_len, self.path, self.bonus, self.status, stream,
                                check)

    def accept_commit(self, stream=None, in_place=False, check=True):
        dst = self.H0 if in_place else self.H_new
        return tv_accept_commit(self.problem(), self.H0, self.g, self.k, self.v, self.draft,
                                self.target, self.root_argmax, self.accept_len, self.path,
                                self.bonus, dst, self.status, stream, check)

    def pending(self) -> tv_pending:
        """This batch's accepted paths and factors as the commit still to apply."""
        return make_pending(self.T, self.max_nodes, self.max_depth, self.node_offsets,
                            self.parent, self.g, self.k, self.v, self.path, self.accept_len)

    def commit_verify(self, pending: "Optional[DeviceBatch]", stream=None, check=True):
        """Apply `pending`'s accepted paths to this batch's state H0 in place, then
        verify this batch's tree against the updated state."""
        pend = pending.pending() if pending is not None else None
        return tv_commit_verify(self.problem(), pend, self.H0, self.q, self.k, self.v, self.g,
                                self.out, self.status, stream, check)

    def accept_commit_verify(self, prev: "DeviceBatch", stream=None, check=True):
        """One step of the loop: the greedy walk of `prev`'s tree, the commit of the paths
        it finds to this batch's state H0 in place, and the verification of this batch's
        tree, in one call.  The walk's results (of `prev`'s tree) go to this batch's
        accept_len, path and bonus, the step's own result buffers."""
        return tv_accept_commit_verify(self.problem(), prev.pending(), prev.draft, prev.target,
                                       prev.root_argmax, self.accept_len, self.path, self.bonus,
                                       self.H0, self.q, self.k, self.v, self.g, self.out,
                                       self.status, stream, check)

    def commit(self, stream=None, in_place=False, check=True):
        dst = self.H0 if in_place else self.H_new
        return tv_commit(self.problem(), self.H0, self.g, self.k, self.v, self.path,
                         self.accept_len, dst, self.status, stream, check)
