// tv_api.cu -- the C ABI of libtreeverify: argument checks, kernel choice, launch.
//
// Host-checkable errors return before any CUDA call, so they can be exercised
// without a GPU.  Nothing here allocates device memory or synchronises.
#include <stdint.h>

#include <initializer_list>

#include "tv_internal.cuh"

namespace tv {
// verify_tc_big.cu: whether the staged large-tree kernel takes this problem and is
// the faster choice (per-channel decay, trees of 64 or more nodes)
bool verify_tc_staged_preferred(const VerifyArgs &a);
// verify_tc_fdiag.cu: the per-channel-decay member of TV_VARIANT_TC_FUSED (dv = 128,
// trees of up to 64 nodes)
bool verify_tc_fdiag_supported(const VerifyArgs &a);
cudaError_t launch_verify_tc_fdiag(const VerifyArgs &a, cudaStream_t s, bool expire_first_wait);
// verify_tc_fwalk.cu: its member for larger per-channel-decay trees (dv = 128, up to
// 256 nodes, depth <= 16): context product on tensor cores, tree term by fp32 walks
bool verify_tc_fwalk_supported(const VerifyArgs &a);
cudaError_t launch_verify_tc_fwalk(const VerifyArgs &a, cudaStream_t s, bool expire_first_wait);
// verify_tc_fused.cu: commit + verify with the pending path found by the greedy walk of
// p's tree in the same kernel (its results written to acc's len, path and bonus)
bool accept_commit_verify_fused_supported(const VerifyArgs &a, const PendingArgs &p);
cudaError_t launch_accept_commit_verify_fused(const VerifyArgs &a, const PendingArgs &p,
                                              const AcceptArgs &acc, float *H, cudaStream_t s);
}  // namespace tv

namespace {

inline bool aligned16(const void *p) { return (reinterpret_cast<uintptr_t>(p) & 15u) == 0; }

tv_status check_dims(const tv_problem *p) {
    if (!p) return TV_ERR_NULL;
    if (p->B < 0 || p->H < 1 || p->total_nodes < 0) return TV_ERR_SHAPE;
    if (p->dk < 8 || p->dv < 8 || (p->dk % 8) || (p->dv % 8)) return TV_ERR_SHAPE;
    if (p->max_nodes < 1 || p->max_depth < 1) return TV_ERR_SHAPE;
    if (p->dk > TV_MAX_DIM || p->dv > TV_MAX_DIM) return TV_ERR_UNSUPPORTED;
    if (p->max_nodes > TV_MAX_NODES || p->max_depth > TV_MAX_DEPTH) return TV_ERR_UNSUPPORTED;
    if (p->decay != TV_DECAY_SCALAR && p->decay != TV_DECAY_DIAG) return TV_ERR_DTYPE;
    if (p->qkv_dtype != TV_BF16 && p->qkv_dtype != TV_F32) return TV_ERR_DTYPE;
    if ((int64_t)p->total_nodes > (int64_t)p->B * p->max_nodes) return TV_ERR_SHAPE;
    if ((int64_t)p->B * p->H > 0x7fffffffLL) return TV_ERR_UNSUPPORTED;
    if (!p->node_offsets) return TV_ERR_NULL;
    if (p->total_nodes > 0 && !p->parent) return TV_ERR_NULL;
    return TV_OK;
}

tv_status check_ptrs(std::initializer_list<const void *> ptrs) {
    for (const void *q : ptrs)
        if (!q) return TV_ERR_NULL;
    for (const void *q : ptrs)
        if (!aligned16(q)) return TV_ERR_ALIGN;
    return TV_OK;
}

// TV_VARIANT_TC_FUSED: all products of a unit on tensor cores; scalar decay (trees of
// up to 32 nodes) or per-channel decay (dv = 128, trees of up to 64 nodes).
bool fused_supported(const tv::VerifyArgs &a) {
    if (a.decay != TV_DECAY_DIAG) return tv::verify_tc_fused_supported(a);
    return tv::verify_tc_fdiag_supported(a) || tv::verify_tc_fwalk_supported(a);
}

cudaError_t launch_fused(const tv::VerifyArgs &a, cudaStream_t s, bool expire) {
    if (a.decay != TV_DECAY_DIAG) return tv::launch_verify_tc_fused(a, s, expire);
    return tv::verify_tc_fdiag_supported(a) ? tv::launch_verify_tc_fdiag(a, s, expire)
                                            : tv::launch_verify_tc_fwalk(a, s, expire);
}

// The kernel TV_VARIANT_AUTO picks: the fused tensor-core kernels where they apply,
// the staged large-tree kernel for per-channel decay trees of 64 or more nodes, the
// one-unit tensor-core kernel where it applies, the large-tree tensor-core kernels for
// trees too large for it, else SIMT.
int32_t auto_variant(const tv::VerifyArgs &a) {
    if (fused_supported(a)) return TV_VARIANT_TC_FUSED;
    if (tv::verify_tc_staged_preferred(a)) return TV_VARIANT_TC_TILED;
    if (tv::verify_tc_supported(a)) return TV_VARIANT_TC;
    if (tv::verify_tc_big_supported(a)) return TV_VARIANT_TC_TILED;
    return TV_VARIANT_SIMT;
}

cudaError_t launch_verify_auto(const tv::VerifyArgs &a, cudaStream_t s) {
    switch (auto_variant(a)) {
        case TV_VARIANT_TC_FUSED: return launch_fused(a, s, false);
        case TV_VARIANT_TC: return tv::launch_verify_tc(a, s);
        case TV_VARIANT_TC_TILED: return tv::launch_verify_tc_big(a, s);
        default: return tv::launch_verify_simt(a, s);
    }
}

}  // namespace

extern "C" {

const char *tv_status_string(int32_t s) {
    switch (s) {
        case TV_OK: return "TV_OK";
        case TV_ERR_NULL: return "TV_ERR_NULL: a required pointer is NULL";
        case TV_ERR_SHAPE: return "TV_ERR_SHAPE: a size argument is out of range";
        case TV_ERR_DTYPE: return "TV_ERR_DTYPE: unknown decay kind or element type";
        case TV_ERR_ALIGN: return "TV_ERR_ALIGN: an array pointer is not 16-byte aligned";
        case TV_ERR_UNSUPPORTED: return "TV_ERR_UNSUPPORTED: a limit of the library is exceeded";
        case TV_ERR_TREE: return "TV_ERR_TREE: malformed tree, offsets or path";
        case TV_ERR_CUDA: return "TV_ERR_CUDA: a CUDA runtime call failed";
        case TV_ERR_TIMEOUT: return "TV_ERR_TIMEOUT: a bounded device wait expired";
        default: return "unknown tv_status";
    }
}

int32_t tv_version(void) { return TV_VERSION; }

int32_t tv_verify_supports(const tv_problem *p, int32_t variant) {
    tv_status st = check_dims(p);
    if (st != TV_OK) return -static_cast<int32_t>(st);
    tv::VerifyArgs a{p->B, p->H, p->dk, p->dv, p->total_nodes, p->max_nodes, p->max_depth,
                     p->decay, p->qkv_dtype, p->node_offsets, p->parent, p->depth,
                     nullptr, nullptr, nullptr, nullptr, nullptr, nullptr, nullptr};
    switch (variant) {
        case TV_VARIANT_AUTO:
        case TV_VARIANT_SIMT: return 1;
        case TV_VARIANT_TC: return tv::verify_tc_supported(a) ? 1 : 0;
        case TV_VARIANT_TC_FUSED: return fused_supported(a) ? 1 : 0;
        case TV_VARIANT_TC_TILED: return tv::verify_tc_big_supported(a) ? 1 : 0;
        default: return -static_cast<int32_t>(TV_ERR_DTYPE);
    }
}

int32_t tv_verify_variant(const tv_problem *p) {
    tv_status st = check_dims(p);
    if (st != TV_OK) return -static_cast<int32_t>(st);
    tv::VerifyArgs a{p->B, p->H, p->dk, p->dv, p->total_nodes, p->max_nodes, p->max_depth,
                     p->decay, p->qkv_dtype, p->node_offsets, p->parent, p->depth,
                     nullptr, nullptr, nullptr, nullptr, nullptr, nullptr, nullptr};
    return auto_variant(a);
}

size_t tv_workspace_bytes(const tv_problem *p) {
    (void)p;
    return 0;
}

tv_status tv_verify_ex(const tv_problem *p, const float *H0, const void *q, const void *k,
                       const void *v, const float *g, float *out, int32_t *dev_status,
                       void *stream, int32_t variant) {
    tv_status st = check_dims(p);
    if (st != TV_OK) return st;
    if (!p->depth && p->total_nodes > 0) return TV_ERR_NULL;
    const bool expire = (variant & TV_VARIANT_TEST_EXPIRE_WAIT) != 0;
    variant &= ~TV_VARIANT_TEST_EXPIRE_WAIT;
    if (variant < TV_VARIANT_AUTO || variant > TV_VARIANT_TC_TILED) return TV_ERR_DTYPE;
    if (expire && variant != TV_VARIANT_TC_FUSED) return TV_ERR_UNSUPPORTED;
    if (!dev_status) return TV_ERR_NULL;
    if (p->B == 0 || p->total_nodes == 0) return TV_OK;
    st = check_ptrs({H0, q, k, v, g, out, p->node_offsets, p->parent, p->depth, dev_status});
    if (st != TV_OK) return st;

    tv::VerifyArgs a{p->B, p->H, p->dk, p->dv, p->total_nodes, p->max_nodes, p->max_depth,
                     p->decay, p->qkv_dtype, p->node_offsets, p->parent, p->depth,
                     H0, q, k, v, g, out, dev_status};
    cudaStream_t s = static_cast<cudaStream_t>(stream);
    cudaError_t e;
    switch (variant) {
        case TV_VARIANT_SIMT: e = tv::launch_verify_simt(a, s); break;
        case TV_VARIANT_TC:
            if (!tv::verify_tc_supported(a)) return TV_ERR_UNSUPPORTED;
            e = tv::launch_verify_tc(a, s);
            break;
        case TV_VARIANT_TC_FUSED:
            if (!fused_supported(a)) return TV_ERR_UNSUPPORTED;
            e = launch_fused(a, s, expire);
            break;
        case TV_VARIANT_TC_TILED:
            if (!tv::verify_tc_big_supported(a)) return TV_ERR_UNSUPPORTED;
            e = tv::launch_verify_tc_big(a, s);
            break;
        default: e = launch_verify_auto(a, s);
    }
    return e == cudaSuccess ? TV_OK : TV_ERR_CUDA;
}

size_t tv_verify_serial_workspace_bytes(const tv_problem *p) {
    if (check_dims(p) != TV_OK) return 0;
    tv::VerifyArgs a{p->B, p->H, p->dk, p->dv, p->total_nodes, p->max_nodes, p->max_depth,
                     p->decay, p->qkv_dtype, p->node_offsets, p->parent, p->depth,
                     nullptr, nullptr, nullptr, nullptr, nullptr, nullptr, nullptr};
    return tv::verify_serial_workspace_bytes(a);
}

tv_status tv_verify_serial(const tv_problem *p, const float *H0, const void *q, const void *k,
                           const void *v, const float *g, float *out, void *workspace,
                           size_t workspace_bytes, int32_t *dev_status, void *stream) {
    tv_status st = check_dims(p);
    if (st != TV_OK) return st;
    if (!p->depth && p->total_nodes > 0) return TV_ERR_NULL;
    if (!dev_status || !workspace) return TV_ERR_NULL;
    if (p->B == 0 || p->total_nodes == 0) return TV_OK;
    st = check_ptrs({H0, q, k, v, g, out, p->node_offsets, p->parent, p->depth, dev_status,
                     workspace});
    if (st != TV_OK) return st;
    tv::VerifyArgs a{p->B, p->H, p->dk, p->dv, p->total_nodes, p->max_nodes, p->max_depth,
                     p->decay, p->qkv_dtype, p->node_offsets, p->parent, p->depth,
                     H0, q, k, v, g, out, dev_status};
    if (workspace_bytes < tv::verify_serial_workspace_bytes(a)) return TV_ERR_SHAPE;
    cudaError_t e = tv::launch_verify_serial(a, static_cast<float *>(workspace),
                                             static_cast<cudaStream_t>(stream));
    return e == cudaSuccess ? TV_OK : TV_ERR_CUDA;
}

tv_status tv_verify_serial_static(const tv_problem *p, const float *H0, const void *q,
                                  const void *k, const void *v, const float *g, float *out,
                                  int32_t *dev_status, void *stream) {
    tv_status st = check_dims(p);
    if (st != TV_OK) return st;
    if (!p->depth && p->total_nodes > 0) return TV_ERR_NULL;
    if (!dev_status) return TV_ERR_NULL;
    tv::VerifyArgs a{p->B, p->H, p->dk, p->dv, p->total_nodes, p->max_nodes, p->max_depth,
                     p->decay, p->qkv_dtype, p->node_offsets, p->parent, p->depth,
                     H0, q, k, v, g, out, dev_status};
    if (tv::verify_serial_workspace_bytes(a) > TV_SERIAL_STATIC_BYTES) return TV_ERR_UNSUPPORTED;
    if (p->B == 0 || p->total_nodes == 0) return TV_OK;
    st = check_ptrs({H0, q, k, v, g, out, p->node_offsets, p->parent, p->depth, dev_status});
    if (st != TV_OK) return st;
    cudaError_t e = tv::launch_verify_serial_static(a, static_cast<cudaStream_t>(stream));
    return e == cudaSuccess ? TV_OK : TV_ERR_CUDA;
}

tv_status tv_verify(const tv_problem *p, const float *H0, const void *q, const void *k,
                    const void *v, const float *g, float *out, int32_t *dev_status,
                    void *stream) {
    return tv_verify_ex(p, H0, q, k, v, g, out, dev_status, stream, TV_VARIANT_AUTO);
}

tv_status tv_accept_greedy(int32_t B, int32_t total_nodes, int32_t max_nodes, int32_t max_depth,
                           const int32_t *node_offsets, const int32_t *parent,
                           const int32_t *draft_tokens, const int32_t *target_argmax,
                           const int32_t *root_argmax, int32_t *accept_len, int32_t *path,
                           int32_t *bonus, int32_t *dev_status, void *stream) {
    if (B < 0 || total_nodes < 0 || max_nodes < 1 || max_depth < 1) return TV_ERR_SHAPE;
    if (max_nodes > TV_MAX_NODES || max_depth > TV_MAX_DEPTH) return TV_ERR_UNSUPPORTED;
    if ((int64_t)total_nodes > (int64_t)B * max_nodes) return TV_ERR_SHAPE;
    if (!node_offsets || !root_argmax || !accept_len || !path || !bonus || !dev_status)
        return TV_ERR_NULL;
    if (total_nodes > 0 && (!parent || !draft_tokens || !target_argmax)) return TV_ERR_NULL;
    if (B == 0) return TV_OK;
    tv_status st = check_ptrs({node_offsets, root_argmax, accept_len, path, bonus, dev_status});
    if (st != TV_OK) return st;
    if (total_nodes > 0) {
        st = check_ptrs({parent, draft_tokens, target_argmax});
        if (st != TV_OK) return st;
    }
    tv::AcceptArgs a{B, total_nodes, max_nodes, max_depth, node_offsets, parent, draft_tokens,
                     target_argmax, root_argmax, accept_len, path, bonus, dev_status};
    cudaError_t e = tv::launch_accept(a, static_cast<cudaStream_t>(stream));
    return e == cudaSuccess ? TV_OK : TV_ERR_CUDA;
}

tv_status tv_accept_greedy_logits(int32_t B, int32_t total_nodes, int32_t max_nodes,
                                  int32_t max_depth, int32_t vocab, const int32_t *node_offsets,
                                  const int32_t *parent, const int32_t *draft_tokens,
                                  const void *root_logits, const void *node_logits,
                                  int32_t *root_argmax, int32_t *target_argmax,
                                  int32_t *accept_len, int32_t *path, int32_t *bonus,
                                  int32_t *dev_status, void *stream) {
    if (B < 0 || total_nodes < 0 || max_nodes < 1 || max_depth < 1 || vocab < 1)
        return TV_ERR_SHAPE;
    if (max_nodes > TV_MAX_NODES || max_depth > TV_MAX_DEPTH) return TV_ERR_UNSUPPORTED;
    if ((int64_t)total_nodes > (int64_t)B * max_nodes) return TV_ERR_SHAPE;
    if ((int64_t)B * 8 > 0x7fffffffLL) return TV_ERR_UNSUPPORTED;
    if (!node_offsets || !root_logits || !root_argmax || !accept_len || !path || !bonus ||
        !dev_status)
        return TV_ERR_NULL;
    if (total_nodes > 0 && (!parent || !draft_tokens || !node_logits || !target_argmax))
        return TV_ERR_NULL;
    if (B == 0) return TV_OK;
    tv_status st = check_ptrs(
        {node_offsets, root_logits, root_argmax, accept_len, path, bonus, dev_status});
    if (st != TV_OK) return st;
    if (total_nodes > 0) {
        st = check_ptrs({parent, draft_tokens, node_logits, target_argmax});
        if (st != TV_OK) return st;
    }
    tv::LogitsArgs a{B, total_nodes, max_nodes, max_depth, vocab, node_offsets, parent,
                     draft_tokens, static_cast<const uint16_t *>(root_logits),
                     static_cast<const uint16_t *>(node_logits), root_argmax, target_argmax,
                     accept_len, path, bonus, dev_status};
    cudaError_t e = tv::launch_accept_logits(a, static_cast<cudaStream_t>(stream));
    return e == cudaSuccess ? TV_OK : TV_ERR_CUDA;
}

tv_status tv_accept_stochastic(int32_t B, int32_t total_nodes, int32_t max_nodes,
                               int32_t max_depth, int32_t vocab, const int32_t *node_offsets,
                               const int32_t *parent, const int32_t *draft_tokens,
                               const float *root_p, const float *node_p, const float *root_q,
                               const float *node_q, const double *u_accept,
                               const double *u_bonus, int32_t *accept_len, int32_t *path,
                               int32_t *bonus, int32_t *dev_status, void *stream) {
    if (B < 0 || total_nodes < 0 || max_nodes < 1 || max_depth < 1 || vocab < 1)
        return TV_ERR_SHAPE;
    if (max_nodes > TV_MAX_NODES || max_depth > TV_MAX_DEPTH) return TV_ERR_UNSUPPORTED;
    if ((int64_t)total_nodes > (int64_t)B * max_nodes) return TV_ERR_SHAPE;
    if (!node_offsets || !root_p || !root_q || !u_bonus || !accept_len || !path || !bonus ||
        !dev_status)
        return TV_ERR_NULL;
    if (total_nodes > 0 && (!parent || !draft_tokens || !node_p || !node_q || !u_accept))
        return TV_ERR_NULL;
    if (B == 0) return TV_OK;
    tv_status st = check_ptrs({node_offsets, root_p, root_q, u_bonus, accept_len, path, bonus,
                               dev_status});
    if (st != TV_OK) return st;
    if (total_nodes > 0) {
        st = check_ptrs({parent, draft_tokens, node_p, node_q, u_accept});
        if (st != TV_OK) return st;
    }
    tv::StochArgs a{B, total_nodes, max_nodes, max_depth, vocab, node_offsets, parent,
                    draft_tokens, root_p, node_p, root_q, node_q, u_accept, u_bonus,
                    accept_len, path, bonus, dev_status};
    cudaError_t e = tv::launch_accept_stochastic(a, static_cast<cudaStream_t>(stream));
    return e == cudaSuccess ? TV_OK : TV_ERR_CUDA;
}

}  // extern "C"

namespace {

tv_status attn_dims(int32_t B, int32_t T, int32_t max_nodes, int32_t H, int32_t Hkv, int32_t d,
                    int32_t P) {
    if (B < 0 || T < 0 || max_nodes < 1 || H < 1 || Hkv < 1 || P < 1 || d < 1) return TV_ERR_SHAPE;
    if (H % Hkv) return TV_ERR_SHAPE;
    if ((int64_t)T > (int64_t)B * max_nodes) return TV_ERR_SHAPE;
    const int32_t grp = H / Hkv;
    if (d != 64 && d != 128) return TV_ERR_UNSUPPORTED;
    if (grp > 128 || (grp & (grp - 1))) return TV_ERR_UNSUPPORTED;
    if (max_nodes > TV_MAX_NODES) return TV_ERR_UNSUPPORTED;
    if ((int64_t)B * Hkv * P > 0x7fffffffLL || (int64_t)T * H > 0x7fffffffLL)
        return TV_ERR_UNSUPPORTED;
    return TV_OK;
}

}  // namespace

extern "C" {

size_t tv_tree_attention_workspace_bytes(int32_t B, int32_t total_nodes, int32_t max_nodes,
                                         int32_t H, int32_t Hkv, int32_t d, int32_t P) {
    if (attn_dims(B, total_nodes, max_nodes, H, Hkv, d, P) != TV_OK || B == 0) return 0;
    tv::AttnArgs a{};
    a.B = B;
    a.T = total_nodes;
    a.max_nodes = max_nodes;
    a.H = H;
    a.Hkv = Hkv;
    a.d = d;
    a.P = P;
    return tv::tree_attention_workspace_bytes(a);
}

tv_status tv_tree_attention(int32_t B, int32_t total_nodes, int32_t max_nodes, int32_t H,
                            int32_t Hkv, int32_t d, int32_t P, const int32_t *node_offsets,
                            const int32_t *parent, const int32_t *ctx_len, const void *q,
                            const void *k_cache, const void *v_cache, const void *k_tree,
                            const void *v_tree, float scale, float *out, void *workspace,
                            size_t workspace_bytes, int32_t *dev_status, void *stream) {
    tv_status st = attn_dims(B, total_nodes, max_nodes, H, Hkv, d, P);
    if (st != TV_OK) return st;
    if (!(scale > 0.f) || scale > 3.0e38f) return TV_ERR_SHAPE;  // positive and finite
    if (!node_offsets || !ctx_len || !k_cache || !v_cache || !dev_status) return TV_ERR_NULL;
    if (total_nodes > 0 && (!parent || !q || !k_tree || !v_tree || !out)) return TV_ERR_NULL;
    if (B == 0 || total_nodes == 0) return TV_OK;
    st = check_ptrs({node_offsets, parent, ctx_len, q, k_cache, v_cache, k_tree, v_tree, out,
                     dev_status});
    if (st != TV_OK) return st;
    if (workspace && !aligned16(workspace)) return TV_ERR_ALIGN;
    tv::AttnArgs a{B, total_nodes, max_nodes, H, Hkv, d, P, node_offsets, parent, ctx_len,
                   q, k_cache, v_cache, k_tree, v_tree, scale, out,
                   static_cast<float *>(workspace), workspace ? workspace_bytes : 0, dev_status};
    cudaError_t e = tv::launch_tree_attention(a, static_cast<cudaStream_t>(stream));
    if (e == cudaErrorNotSupported) return TV_ERR_UNSUPPORTED;
    return e == cudaSuccess ? TV_OK : TV_ERR_CUDA;
}

tv_status tv_build_tree(int32_t B, int32_t C, int32_t depth_cap, int32_t n,
                        const double *marginals, const double *cost, int32_t *parent,
                        int32_t *token, double *rho, int32_t *count, void *stream) {
    if (B < 0 || C < 1 || C > 32 || depth_cap < 1 || depth_cap > TV_MAX_DEPTH || n < 1 ||
        n > TV_MAX_NODES)
        return TV_ERR_SHAPE;
    if (!marginals || !parent || !token || !rho || !count) return TV_ERR_NULL;
    if (B == 0) return TV_OK;
    tv_status st = check_ptrs({marginals, parent, token, rho, count});
    if (st != TV_OK) return st;
    if (cost && !aligned16(cost)) return TV_ERR_ALIGN;
    tv::BuildArgs a{B, C, depth_cap, n, marginals, cost, parent, token, count, rho};
    cudaError_t e = tv::launch_build_tree(a, static_cast<cudaStream_t>(stream));
    return e == cudaSuccess ? TV_OK : TV_ERR_CUDA;
}

tv_status tv_commit(const tv_problem *p, const float *H0, const float *g, const void *k,
                    const void *v, const int32_t *path, const int32_t *accept_len,
                    float *H_new, int32_t *dev_status, void *stream) {
    tv_status st = check_dims(p);
    if (st != TV_OK) return st;
    if (!dev_status || !H0 || !H_new || !path || !accept_len) return TV_ERR_NULL;
    if (p->total_nodes > 0 && (!g || !k || !v)) return TV_ERR_NULL;
    if (p->B == 0) return TV_OK;
    // H_new is H0 or disjoint from it
    const size_t bytes = (size_t)p->B * p->H * p->dk * p->dv * sizeof(float);
    const char *h0 = reinterpret_cast<const char *>(H0);
    const char *hn = reinterpret_cast<const char *>(H_new);
    if (hn != h0 && hn < h0 + bytes && h0 < hn + bytes) return TV_ERR_SHAPE;
    st = check_ptrs({H0, H_new, path, accept_len, p->node_offsets, dev_status});
    if (st != TV_OK) return st;
    if (p->total_nodes > 0) {
        st = check_ptrs({g, k, v, p->parent});
        if (st != TV_OK) return st;
    }
    tv::CommitArgs a{p->B, p->H, p->dk, p->dv, p->total_nodes, p->max_nodes, p->max_depth,
                     p->decay, p->qkv_dtype, p->node_offsets, p->parent, H0, g, k, v, path,
                     accept_len, H_new, dev_status, nullptr, nullptr, nullptr,
                     nullptr, nullptr, nullptr};
    cudaError_t e = tv::launch_commit(a, static_cast<cudaStream_t>(stream));
    return e == cudaSuccess ? TV_OK : TV_ERR_CUDA;
}

tv_status tv_accept_commit(const tv_problem *p, const float *H0, const float *g, const void *k,
                           const void *v, const int32_t *draft_tokens,
                           const int32_t *target_argmax, const int32_t *root_argmax,
                           int32_t *accept_len, int32_t *path, int32_t *bonus, float *H_new,
                           int32_t *dev_status, void *stream) {
    tv_status st = check_dims(p);
    if (st != TV_OK) return st;
    if (!dev_status || !H0 || !H_new || !path || !accept_len || !bonus || !root_argmax)
        return TV_ERR_NULL;
    if (p->total_nodes > 0 && (!g || !k || !v || !draft_tokens || !target_argmax))
        return TV_ERR_NULL;
    if (p->B == 0) return TV_OK;
    const size_t bytes = (size_t)p->B * p->H * p->dk * p->dv * sizeof(float);
    const char *h0 = reinterpret_cast<const char *>(H0);
    const char *hn = reinterpret_cast<const char *>(H_new);
    if (hn != h0 && hn < h0 + bytes && h0 < hn + bytes) return TV_ERR_SHAPE;
    st = check_ptrs({H0, H_new, path, accept_len, bonus, root_argmax, p->node_offsets,
                     dev_status});
    if (st != TV_OK) return st;
    if (p->total_nodes > 0) {
        st = check_ptrs({g, k, v, p->parent, draft_tokens, target_argmax});
        if (st != TV_OK) return st;
    }
    tv::CommitArgs a{p->B, p->H, p->dk, p->dv, p->total_nodes, p->max_nodes, p->max_depth,
                     p->decay, p->qkv_dtype, p->node_offsets, p->parent, H0, g, k, v, nullptr,
                     nullptr, H_new, dev_status, draft_tokens, target_argmax, root_argmax,
                     path, accept_len, bonus};
    cudaError_t e = tv::launch_accept_commit(a, static_cast<cudaStream_t>(stream));
    return e == cudaSuccess ? TV_OK : TV_ERR_CUDA;
}

tv_status tv_commit_verify(const tv_problem *p, const tv_pending *pend, float *H, const void *q,
                           const void *k, const void *v, const float *g, float *out,
                           int32_t *dev_status, void *stream) {
    if (!pend) return tv_verify(p, H, q, k, v, g, out, dev_status, stream);
    tv_status st = check_dims(p);
    if (st != TV_OK) return st;
    if (!p->depth && p->total_nodes > 0) return TV_ERR_NULL;
    if (!dev_status || !H || !pend->node_offsets || !pend->path || !pend->accept_len)
        return TV_ERR_NULL;
    if (pend->total_nodes < 0 || pend->max_nodes < 1 || pend->max_depth < 1) return TV_ERR_SHAPE;
    if (pend->max_nodes > TV_MAX_NODES || pend->max_depth > TV_MAX_DEPTH)
        return TV_ERR_UNSUPPORTED;
    if ((int64_t)pend->total_nodes > (int64_t)p->B * pend->max_nodes) return TV_ERR_SHAPE;
    if (pend->total_nodes > 0 && (!pend->parent || !pend->g || !pend->k || !pend->v))
        return TV_ERR_NULL;
    if (p->total_nodes > 0 && (!q || !k || !v || !g || !out)) return TV_ERR_NULL;
    if (p->B == 0) return TV_OK;
    st = check_ptrs({H, dev_status, p->node_offsets, pend->node_offsets, pend->path,
                     pend->accept_len});
    if (st != TV_OK) return st;
    if (pend->total_nodes > 0) {
        st = check_ptrs({pend->parent, pend->g, pend->k, pend->v});
        if (st != TV_OK) return st;
    }
    if (p->total_nodes > 0) {
        st = check_ptrs({q, k, v, g, out, p->parent, p->depth});
        if (st != TV_OK) return st;
    }

    tv::VerifyArgs a{p->B, p->H, p->dk, p->dv, p->total_nodes, p->max_nodes, p->max_depth,
                     p->decay, p->qkv_dtype, p->node_offsets, p->parent, p->depth,
                     H, q, k, v, g, out, dev_status};
    tv::PendingArgs pa{pend->total_nodes, pend->max_nodes, pend->max_depth, pend->node_offsets,
                       pend->parent, pend->g, pend->k, pend->v, pend->path, pend->accept_len};
    cudaStream_t s = static_cast<cudaStream_t>(stream);
    if (p->total_nodes > 0 && tv::commit_verify_fused_supported(a, pa)) {
        cudaError_t e = tv::launch_commit_verify_fused(a, pa, H, s);
        return e == cudaSuccess ? TV_OK : TV_ERR_CUDA;
    }
    if (p->total_nodes > 0 && tv::commit_verify_tc_supported(a, pa)) {
        cudaError_t e = tv::launch_commit_verify_tc(a, pa, H, s);
        return e == cudaSuccess ? TV_OK : TV_ERR_CUDA;
    }
    // other shapes: the commit kernel in place, then the verify kernel
    tv::CommitArgs c{p->B, p->H, p->dk, p->dv, pend->total_nodes, pend->max_nodes,
                     pend->max_depth, p->decay, p->qkv_dtype, pend->node_offsets, pend->parent,
                     H, pend->g, pend->k, pend->v, pend->path, pend->accept_len, H, dev_status,
                     nullptr, nullptr, nullptr, nullptr, nullptr, nullptr};
    cudaError_t e = tv::launch_commit(c, s);
    if (e != cudaSuccess) return TV_ERR_CUDA;
    if (p->total_nodes == 0) return TV_OK;
    e = launch_verify_auto(a, s);
    return e == cudaSuccess ? TV_OK : TV_ERR_CUDA;
}


tv_status tv_accept_commit_verify(const tv_problem *p, const tv_pending *prev,
                                  const int32_t *draft_tokens, const int32_t *target_argmax,
                                  const int32_t *root_argmax, int32_t *accept_len, int32_t *path,
                                  int32_t *bonus, float *H, const void *q, const void *k,
                                  const void *v, const float *g, float *out, int32_t *dev_status,
                                  void *stream) {
    tv_status st = check_dims(p);
    if (st != TV_OK) return st;
    if (!prev || !dev_status || !H || !prev->node_offsets || !root_argmax || !accept_len ||
        !path || !bonus)
        return TV_ERR_NULL;
    if (!p->depth && p->total_nodes > 0) return TV_ERR_NULL;
    if (prev->total_nodes < 0 || prev->max_nodes < 1 || prev->max_depth < 1) return TV_ERR_SHAPE;
    if (prev->max_nodes > TV_MAX_NODES || prev->max_depth > TV_MAX_DEPTH)
        return TV_ERR_UNSUPPORTED;
    if ((int64_t)prev->total_nodes > (int64_t)p->B * prev->max_nodes) return TV_ERR_SHAPE;
    if (prev->total_nodes > 0 &&
        (!prev->parent || !prev->g || !prev->k || !prev->v || !draft_tokens || !target_argmax))
        return TV_ERR_NULL;
    if (p->total_nodes > 0 && (!q || !k || !v || !g || !out)) return TV_ERR_NULL;
    if (p->B == 0) return TV_OK;
    st = check_ptrs({H, dev_status, p->node_offsets, prev->node_offsets, root_argmax, accept_len,
                     path, bonus});
    if (st != TV_OK) return st;
    if (prev->total_nodes > 0) {
        st = check_ptrs({prev->parent, prev->g, prev->k, prev->v, draft_tokens, target_argmax});
        if (st != TV_OK) return st;
    }
    if (p->total_nodes > 0) {
        st = check_ptrs({q, k, v, g, out, p->parent, p->depth});
        if (st != TV_OK) return st;
    }
    tv::VerifyArgs a{p->B, p->H, p->dk, p->dv, p->total_nodes, p->max_nodes, p->max_depth,
                     p->decay, p->qkv_dtype, p->node_offsets, p->parent, p->depth,
                     H, q, k, v, g, out, dev_status};
    tv::PendingArgs pa{prev->total_nodes, prev->max_nodes, prev->max_depth, prev->node_offsets,
                       prev->parent, prev->g, prev->k, prev->v, path, accept_len};
    tv::AcceptArgs acc{p->B, prev->total_nodes, prev->max_nodes, prev->max_depth,
                       prev->node_offsets, prev->parent, draft_tokens, target_argmax, root_argmax,
                       accept_len, path, bonus, dev_status};
    cudaStream_t s = static_cast<cudaStream_t>(stream);
    if (p->total_nodes > 0 && tv::accept_commit_verify_fused_supported(a, pa)) {
        cudaError_t e = tv::launch_accept_commit_verify_fused(a, pa, acc, H, s);
        return e == cudaSuccess ? TV_OK : TV_ERR_CUDA;
    }
    // other shapes: the walk, then tv_commit_verify with the paths it wrote
    cudaError_t e = tv::launch_accept(acc, s);
    if (e != cudaSuccess) return TV_ERR_CUDA;
    tv_pending pend = *prev;
    pend.path = path;
    pend.accept_len = accept_len;
    return tv_commit_verify(p, &pend, H, q, k, v, g, out, dev_status, stream);
}

}  // extern "C"
