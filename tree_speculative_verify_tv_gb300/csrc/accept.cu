// accept.cu -- greedy acceptance walk over each request's draft tree.
//
// LLM Primer VI ch. 9 §9.1: the longest draft prefix that agrees with the target
// is accepted and, at the first disagreement, the target's own token is kept.
// On a tree: t = root_argmax[b]; move to the lowest-index child whose draft token
// equals t, set t = target_argmax[child]; stop when no child matches; bonus = t.
//
// One warp per request.  Children of node c all have larger indices than c, so
// each step scans the nodes after the current one 32 at a time; a ballot finds
// the lowest matching index.  Integer-only, exact.
#include "tv_internal.cuh"

namespace tv {
namespace {

constexpr int kWarps = 8;

__global__ void __launch_bounds__(kWarps * 32) accept_kernel(AcceptArgs a) {
    const int lane = threadIdx.x & 31;
    const int b = blockIdx.x * kWarps + (threadIdx.x >> 5);
    if (b >= a.B) return;
    const int md = a.max_depth;
    int32_t *path = a.path + (size_t)b * md;

    int off, n;
    bool ok = request_range(a.node_offsets, b, a.T, a.max_nodes, off, n);
    if (ok) {
        // parents precede children: parent[i] in [-1, i)
        bool bad = false;
        for (int i = lane; i < n; i += 32) {
            int p = a.parent[off + i];
            bad |= (p < -1 || p >= i);
        }
        ok = !__any_sync(0xffffffffu, bad);
    }

    int L = 0;
    int32_t t = a.root[b];
    if (ok) {
        int cur = -1;
        for (;;) {
            int found = -1;
            for (int base = cur + 1; base < n; base += 32) {
                const int i = base + lane;
                bool hit = i < n && a.parent[off + i] == cur && a.draft[off + i] == t;
                unsigned m = __ballot_sync(0xffffffffu, hit);
                if (m) {
                    found = base + __ffs(m) - 1;
                    break;
                }
            }
            if (found < 0) break;
            if (L >= md) {  // deeper than the caller's bound: not a valid tree for it
                ok = false;
                break;
            }
            if (lane == 0) path[L] = found;
            ++L;
            t = a.target[off + found];
            cur = found;
        }
    }
    if (!ok) {
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
    accept_kernel<<<grid, kWarps * 32, 0, s>>>(a);
    return cudaGetLastError();
}

}  // namespace tv
