// accept.cu -- greedy acceptance walk over each request's draft tree.
//
// LLM Primer VI ch. 9 §9.1: the longest draft prefix that agrees with the target
// is accepted and, at the first disagreement, the target's own token is kept.
// On a tree: t = root_argmax[b]; move to the lowest-index child whose draft token
// equals t, set t = target_argmax[child]; stop when no child matches; bonus = t.
//
// One warp per request.  The request's parent/draft/target arrays are first
// copied to shared memory with independent coalesced loads (one round trip to
// memory), then the walk runs on shared memory: children of node c all have
// larger indices than c, so each step scans the nodes after the current one 32
// at a time and a ballot finds the lowest matching index.  Integer-only, exact.
#include "greedy_walk.cuh"

namespace tv {
namespace {

constexpr int kWarps = 8;

__global__ void __launch_bounds__(kWarps * 32) accept_kernel(AcceptArgs a) {
    __shared__ int s_par[kWarps][kMaxNodes];
    __shared__ int s_drf[kWarps][kMaxNodes];
    __shared__ int s_tgt[kWarps][kMaxNodes];
    const int lane = threadIdx.x & 31, w = threadIdx.x >> 5;
    const int b = blockIdx.x * kWarps + w;
    pdl_wait();
    pdl_launch_next();
    if (b >= a.B) return;
    const int md = a.max_depth;
    int32_t *path = a.path + (size_t)b * md;
    int *par = s_par[w], *drf = s_drf[w], *tgt = s_tgt[w];

    int off, n;
    int L = -1;
    int32_t t = -1;
    if (request_range(a.node_offsets, b, a.T, a.max_nodes, off, n))
        L = warp_greedy_walk(a.parent, a.draft, a.target, off, n, md, a.root[b], par, drf, tgt,
                             path, &t);
    if (L < 0) {
        if (lane == 0) report(a.status, TV_ERR_TREE);
        L = 0;
        t = -1;
    }
    __syncwarp();  // order lane 0's path stores before the padding stores
    for (int m = L + lane; m < md; m += 32) path[m] = -1;
    if (lane == 0) {
        a.len[b] = L;
        a.bonus[b] = t;
    }
}

}  // namespace

cudaError_t launch_accept(const AcceptArgs &a, cudaStream_t s) {
    dim3 grid((unsigned)((a.B + kWarps - 1) / kWarps));
    return launch_pdl(accept_kernel, grid, dim3(kWarps * 32), 0, s, a);
}

}  // namespace tv
