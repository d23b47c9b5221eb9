// tv_internal.cuh -- shared declarations of libtreeverify's kernels and launchers.
#pragma once

#include <cuda_runtime.h>
#include <cuda_bf16.h>
#include <stdint.h>

#include <mutex>
#include <set>
#include <utility>

#include "treeverify.h"

namespace tv {

constexpr int kMaxNodes = TV_MAX_NODES;
constexpr int kMaxDepth = TV_MAX_DEPTH;
constexpr int kMaxDim = TV_MAX_DIM;

// Everything a verify launch needs, passed by value to the kernels.
struct VerifyArgs {
    int32_t B, H, dk, dv, T, max_nodes, max_depth, decay, qkv_dtype;
    const int32_t *node_offsets, *parent, *depth;
    const float *H0;
    const void *q, *k, *v;
    const float *g;
    float *out;
    int32_t *status;
};

struct AcceptArgs {
    int32_t B, T, max_nodes, max_depth;
    const int32_t *node_offsets, *parent, *draft, *target, *root;
    int32_t *len, *path, *bonus, *status;
};

struct CommitArgs {
    int32_t B, H, dk, dv, T, max_nodes, max_depth, decay, qkv_dtype;
    const int32_t *node_offsets, *parent;
    const float *H0, *g;
    const void *k, *v;
    const int32_t *path, *len;  // accepted paths (tv_commit)
    float *H_new;
    int32_t *status;
    // tv_accept_commit: the walk's inputs and its outputs
    const int32_t *draft, *target, *root;
    int32_t *path_out, *len_out, *bonus_out;
};

// Stochastic acceptance (tv_accept_stochastic).
struct StochArgs {
    int32_t B, T, max_nodes, max_depth, V;
    const int32_t *node_offsets, *parent, *draft;
    const float *root_p, *node_p, *root_q, *node_q;
    const double *u_accept, *u_bonus;
    int32_t *len, *path, *bonus, *status;
};
cudaError_t launch_accept_stochastic(const StochArgs &a, cudaStream_t s);

// Tree-masked softmax attention over a shared-prefix KV cache (tv_tree_attention).
struct AttnArgs {
    int32_t B, T, max_nodes, H, Hkv, d, P;
    const int32_t *node_offsets, *parent, *ctx_len;
    const void *q, *k_cache, *v_cache, *k_tree, *v_tree;  // bf16
    float scale;
    float *out;
    float *ws;        // split partials (may be null)
    size_t ws_bytes;
    int32_t *status;
};
// Workspace bytes for the context split the library would pick with room for it.
size_t tree_attention_workspace_bytes(const AttnArgs &a);
cudaError_t launch_tree_attention(const AttnArgs &a, cudaStream_t s);

// Best-first draft-tree construction (tv_build_tree).
struct BuildArgs {
    int32_t B, C, depth_cap, n;
    const double *marginals, *cost;  // cost may be null
    int32_t *parent, *token, *count;
    double *rho;
};
size_t build_tree_smem_bytes(int C, int depth_cap, int n);
cudaError_t launch_build_tree(const BuildArgs &a, cudaStream_t s);

// The naive serial baseline with per-node states in a workspace (tv_verify_serial).
size_t verify_serial_workspace_bytes(const VerifyArgs &a);
cudaError_t launch_verify_serial(const VerifyArgs &a, float *ws, cudaStream_t s);
// The same with the library's built-in scratch array (tv_verify_serial_static).
cudaError_t launch_verify_serial_static(const VerifyArgs &a, cudaStream_t s);

// Target argmax from logits + greedy walk (tv_accept_greedy_logits).
struct LogitsArgs {
    int32_t B, T, max_nodes, max_depth, V;
    const int32_t *node_offsets, *parent, *draft;
    const uint16_t *root_logits, *node_logits;  // bf16 bit patterns
    int32_t *root_out, *target_out;             // argmax of every root / node row
    int32_t *len, *path, *bonus, *status;
};
cudaError_t launch_accept_logits(const LogitsArgs &a, cudaStream_t s);

// A commit carried into the next verification (tv_commit_verify).
struct PendingArgs {
    int32_t T, max_nodes, max_depth;
    const int32_t *node_offsets, *parent;
    const float *g;
    const void *k, *v;
    const int32_t *path, *len;
};

cudaError_t launch_verify_simt(const VerifyArgs &a, cudaStream_t s);
// Returns cudaErrorNotSupported when the shape is outside the tensor-core kernel.
cudaError_t launch_verify_tc(const VerifyArgs &a, cudaStream_t s);
bool verify_tc_supported(const VerifyArgs &a);
// Node-tiled tensor-core kernel for large trees (dk = dv = 128).
bool verify_tc_big_supported(const VerifyArgs &a);
cudaError_t launch_verify_tc_big(const VerifyArgs &a, cudaStream_t s);
// Scalar-decay kernel with all three products on tensor cores (trees of <= 32
// nodes), one (request, head) per CTA.  `expire_first_wait` is the test hook of
// TV_VARIANT_TEST_EXPIRE_WAIT.
bool verify_tc_fused_supported(const VerifyArgs &a);
cudaError_t launch_verify_tc_fused(const VerifyArgs &a, cudaStream_t s,
                                   bool expire_first_wait = false);
// One-kernel commit + verify (scalar decay, tensor cores); H is read and written.
bool commit_verify_tc_supported(const VerifyArgs &a, const PendingArgs &p);
cudaError_t launch_commit_verify_tc(const VerifyArgs &a, const PendingArgs &p, float *H,
                                    cudaStream_t s);
// The same on the fused kernel (trees of <= 32 nodes).
bool commit_verify_fused_supported(const VerifyArgs &a, const PendingArgs &p);
cudaError_t launch_commit_verify_fused(const VerifyArgs &a, const PendingArgs &p, float *H,
                                       cudaStream_t s);
cudaError_t launch_accept(const AcceptArgs &a, cudaStream_t s);
cudaError_t launch_commit(const CommitArgs &a, cudaStream_t s);
cudaError_t launch_accept_commit(const CommitArgs &a, cudaStream_t s);

// ---------------------------------------------------------------- device helpers

// First error wins; later errors leave the code unchanged.
__device__ __forceinline__ void report(int32_t *status, int32_t code) {
    atomicCAS(status, 0, code);
}

__device__ __forceinline__ float to_f32(float x) { return x; }
__device__ __forceinline__ float to_f32(__nv_bfloat16 x) { return __bfloat162float(x); }

template <typename E>
__device__ __forceinline__ float ldg_f(const E *p, size_t i) {
    return to_f32(p[i]);
}

__device__ __forceinline__ float warp_sum(float x) {
#pragma unroll
    for (int o = 16; o > 0; o >>= 1) x += __shfl_xor_sync(0xffffffffu, x, o);
    return x;
}

// Request b's node range; false when node_offsets are unusable.
__device__ __forceinline__ bool request_range(const int32_t *offs, int b, int T, int max_nodes,
                                              int &off, int &n) {
    off = offs[b];
    int end = offs[b + 1];
    n = end - off;
    return off >= 0 && end >= off && end <= T && n <= max_nodes;
}

}  // namespace tv

namespace tv {

// Loads one request's parent[] and depth[] (and, when g != nullptr, the scalar
// decays g[(off+i)*H + h]) into shared memory in one memory round trip and
// checks the tree: parent[i] in [-1, i) (parents precede children, so every
// root path ends at the context) and depth[i] = depth[parent]+1 (1 for a child
// of the context) with depth <= max_depth.  Every thread of the block must call
// it; returns the same verdict in all threads.
__device__ __forceinline__ bool load_check_tree(const int32_t *parent, const int32_t *depth,
                                                int off, int n, int max_depth, int *s_par,
                                                int *s_dep, int *s_flag,
                                                const float *g = nullptr, int H = 0, int h = 0,
                                                float *s_g = nullptr) {
    if (threadIdx.x == 0) *s_flag = 0;
    __syncthreads();
    for (int i = threadIdx.x; i < n; i += blockDim.x) {
        const int p = parent[off + i];
        const int d = depth[off + i];
        float gv = 0.f;
        if (g) gv = g[(size_t)(off + i) * H + h];
        s_par[i] = p;
        s_dep[i] = d;
        if (g) s_g[i] = gv;
        if (p < -1 || p >= i) *s_flag = 1;
    }
    __syncthreads();
    if (*s_flag == 0) {
        for (int i = threadIdx.x; i < n; i += blockDim.x) {
            int p = s_par[i];
            int want = p < 0 ? 1 : s_dep[p] + 1;
            if (s_dep[i] != want || s_dep[i] > max_depth) *s_flag = 1;
        }
    }
    __syncthreads();
    return *s_flag == 0;
}

// Raises `kern`'s dynamic shared-memory limit to the most it can use beside its
// static shared memory (227 KB per CTA in all), once per (kernel, device) and under
// a lock; with `max_carveout` it also asks for the largest shared-memory carveout.
// Launches then pass only their own size, so host threads that call the library at
// the same time never rewrite the attribute under one another, and every device a
// process drives gets the setting.  (A device reset by the caller drops it; the
// library is not used across one.)
template <typename Kern>
cudaError_t configure_smem_once(Kern kern, bool max_carveout) {
    int dev = 0;
    cudaError_t e = cudaGetDevice(&dev);
    if (e != cudaSuccess) return e;
    static std::mutex mu;
    static std::set<std::pair<const void *, int>> done;
    std::lock_guard<std::mutex> lock(mu);
    const auto key = std::make_pair(reinterpret_cast<const void *>(kern), dev);
    if (done.count(key)) return cudaSuccess;
    cudaFuncAttributes fa;
    e = cudaFuncGetAttributes(&fa, kern);
    if (e != cudaSuccess) return e;
    e = cudaFuncSetAttribute(kern, cudaFuncAttributeMaxDynamicSharedMemorySize,
                             227 * 1024 - (int)fa.sharedSizeBytes);
    if (e != cudaSuccess) return e;
    if (max_carveout) {
        // without this the driver may configure a smaller shared-memory carveout and
        // fit fewer CTAs than registers and shared memory allow
        e = cudaFuncSetAttribute(kern, cudaFuncAttributePreferredSharedMemoryCarveout,
                                 cudaSharedmemCarveoutMaxShared);
        if (e != cudaSuccess) return e;
    }
    done.insert(key);
    return cudaSuccess;
}

// Programmatic dependent launch: wait for the previous kernel in the stream
// (no-op when launched without the attribute), and let the next one launch.
__device__ __forceinline__ void pdl_wait() { asm volatile("griddepcontrol.wait;" ::: "memory"); }
__device__ __forceinline__ void pdl_launch_next() {
    asm volatile("griddepcontrol.launch_dependents;" ::: "memory");
}

// Launch `kern` on `s` with programmatic stream serialization allowed.
template <typename... KArgs, typename... Args>
cudaError_t launch_pdl(void (*kern)(KArgs...), dim3 grid, dim3 block, size_t smem,
                       cudaStream_t s, Args &&...args) {
    cudaLaunchConfig_t cfg = {};
    cfg.gridDim = grid;
    cfg.blockDim = block;
    cfg.dynamicSmemBytes = smem;
    cfg.stream = s;
    cudaLaunchAttribute attr[1];
    attr[0].id = cudaLaunchAttributeProgrammaticStreamSerialization;
    attr[0].val.programmaticStreamSerializationAllowed = 1;
    cfg.attrs = attr;
    cfg.numAttrs = 1;
    cudaError_t e = cudaLaunchKernelEx(&cfg, kern, static_cast<Args &&>(args)...);
    if (e != cudaSuccess) return e;
    return cudaGetLastError();
}

}  // namespace tv
