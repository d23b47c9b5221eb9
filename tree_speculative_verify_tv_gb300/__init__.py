"""libtreeverify: tree-speculation verification through a gated linear recurrence on GB300.

Three calls, each a CUDA kernel launch on the caller's stream (C ABI in
include/treeverify.h; this package is the ctypes binding):

* ``tv_verify``        outputs of every draft-tree node, tree closed form
* ``tv_accept_greedy`` greedy acceptance walk over each request's tree
* ``tv_commit``        state after the accepted path, rebuilt from the factors
* ``tv_accept_commit`` the two above in one launch
* ``tv_accept_greedy_logits`` the target argmax from its logits and the walk
* ``tv_build_tree``     draft trees by best-first expansion of path scores
* ``tv_accept_stochastic`` acceptance by min(1, p/q) with residual resampling
* ``tv_tree_attention`` tree-masked softmax attention over a shared-prefix KV cache
  (the attention layers of a hybrid model)
* ``tv_verify_serial``  the naive node-by-node verification with per-node states
  (a baseline for the closed form)
* ``tv_commit_verify`` the previous step's commit applied to the state in place,
  then ``tv_verify`` against it (one launch for the tensor-core shapes)
* ``tv_accept_commit_verify`` the previous tree's greedy walk, its commit and the
  verification of the current tree (one launch for the same shapes)

``build()`` compiles the CUDA sources in-tree for sm_103a.
"""
from ._build import build, LIB
from .binding import (  # noqa: F401
    DeviceBatch, TVError, load, make_pending, make_problem, status_string, tv_accept_commit,
    tv_accept_greedy, tv_accept_greedy_logits, tv_commit, tv_commit_verify, tv_pending,
    tv_accept_commit_verify,
    tv_verify_serial, tv_verify_serial_workspace_bytes, tv_verify_serial_static, tv_build_tree,
    tv_accept_stochastic, tv_tree_attention, tv_tree_attention_workspace_bytes,
    TV_SERIAL_STATIC_BYTES,
    tv_problem, tv_status_string, tv_verify, tv_verify_variant, tv_verify_supports, tv_version, EXPORTED,
    TV_OK, TV_ERR_NULL, TV_ERR_SHAPE, TV_ERR_DTYPE, TV_ERR_ALIGN, TV_ERR_UNSUPPORTED,
    TV_ERR_TREE, TV_ERR_CUDA, TV_ERR_TIMEOUT, TV_DECAY_SCALAR, TV_DECAY_DIAG, TV_BF16, TV_F32,
    TV_VARIANT_AUTO, TV_VARIANT_SIMT, TV_VARIANT_TC, TV_VARIANT_TC_FUSED, TV_VARIANT_TC_TILED,
    TV_VARIANT_TEST_EXPIRE_WAIT, tv_workspace_bytes,
    TV_MAX_NODES, TV_MAX_DEPTH, TV_MAX_DIM,
)
