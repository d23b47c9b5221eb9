// greedy_walk.cuh -- the greedy acceptance walk of one request, run by one warp.
//
// LLM Primer VI ch. 9 §9.1: the longest draft prefix that agrees with the target
// is accepted and, at the first disagreement, the target's own token is kept.
// On a tree: t = root token; move to the lowest-index child whose draft token
// equals t, set t = target argmax after that child; stop when no child matches;
// the bonus is the final t.
#pragma once

#include "tv_internal.cuh"

namespace tv {

// The walk on shared memory, parents already checked to lie in [-1, i): children
// of node c all have larger indices, so each step scans the nodes after the
// current one 32 at a time and a ballot finds the lowest matching index.  Writes
// path[0..L) (lane 0) and returns L, with *bonus = final token; returns -1 for a
// walk longer than max_depth.  Every lane of the warp must call it.
__device__ __forceinline__ int warp_greedy_walk_shared(const int *par, const int *drf,
                                                       const int *tgt, int n, int max_depth,
                                                       int32_t root, int *path, int32_t *bonus) {
    const int lane = threadIdx.x & 31;
    int L = 0, cur = -1;
    int32_t t = root;
    for (;;) {
        int found = -1;
        for (int base = cur + 1; base < n; base += 32) {
            const int i = base + lane;
            const bool hit = i < n && par[i] == cur && drf[i] == t;
            const unsigned m = __ballot_sync(0xffffffffu, hit);
            if (m) {
                found = base + __ffs(m) - 1;
                break;
            }
        }
        if (found < 0) break;
        if (L >= max_depth) return -1;  // deeper than the caller's bound
        if (lane == 0) path[L] = found;
        ++L;
        t = tgt[found];
        cur = found;
    }
    *bonus = t;
    return L;
}

// Copies request rows [off, off+n) of parent/draft/target into the warp's shared
// buffers (one round trip of independent loads), checks parent[i] in [-1, i), then
// runs warp_greedy_walk_shared.  Returns -1 for a malformed tree or a walk longer
// than max_depth.  Every lane of the warp must call it.
__device__ __forceinline__ int warp_greedy_walk(const int32_t *parent, const int32_t *draft,
                                                const int32_t *target, int off, int n,
                                                int max_depth, int32_t root, int *par, int *drf,
                                                int *tgt, int *path, int32_t *bonus) {
    const int lane = threadIdx.x & 31;
    bool bad = false;
    for (int i = lane; i < n; i += 32) {
        const int p = parent[off + i];
        par[i] = p;
        drf[i] = draft[off + i];
        tgt[i] = target[off + i];
        bad |= (p < -1 || p >= i);
    }
    if (__any_sync(0xffffffffu, bad)) return -1;
    __syncwarp();
    return warp_greedy_walk_shared(par, drf, tgt, n, max_depth, root, path, bonus);
}

}  // namespace tv
