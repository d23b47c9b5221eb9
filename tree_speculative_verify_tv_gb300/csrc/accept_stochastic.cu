// accept_stochastic.cu -- stochastic acceptance of draft trees.
//
// LLM Primer VI ch. 9 §9.1: a draft token x drawn from the draft distribution q
// is accepted with probability min(1, p(x)/q(x)), p the target distribution; after
// a rejection the emitted token is drawn from the normalized residual (p - q)_+,
// which keeps the output distribution equal to sampling the target.  On a tree
// (reading): the children of the current node are tried in index order, each
// against the current residual (a rejection replaces p by (p - q)_+ / sum); the
// first accepted child becomes the current node, with its own p and q; when no
// child is accepted, the bonus token is drawn from the current residual by inverse
// CDF with the request's uniform.  The acceptance test for child c is
// u_accept[c] * q(x) < p(x).  The uniforms are inputs.
//
// One CTA per request.  Probability rows are fp32 in HBM; every quantity that
// decides a token is fp64.  The residual after k rejections at a node is not
// stored: p_k(x) = max(p_{k-1}(x) - q(x), 0) / Z_k is re-evaluated per element
// from p(x), q(x) and the normalizers Z_1..Z_k kept in shared memory (a zero Z
// leaves p unchanged), so no scratch memory is needed.
#include "tv_internal.cuh"

namespace tv {
namespace {

constexpr int kThreadsA = 256;
constexpr int kWarpsA = kThreadsA / 32;

__device__ __forceinline__ double residual(const float *P, const float *Q, int x, const double *Z,
                                           int nz) {
    double p = P[x];
    const double q = Q[x];
    for (int j = 0; j < nz; ++j)
        if (Z[j] > 0.0) p = fmax(p - q, 0.0) / Z[j];
    return p;
}

// Sum over the block, returned to every thread.
__device__ __forceinline__ double block_sum(double v, double *red) {
    const int lane = threadIdx.x & 31, warp = threadIdx.x >> 5;
#pragma unroll
    for (int o = 16; o > 0; o >>= 1) v += __shfl_xor_sync(0xffffffffu, v, o);
    if (lane == 0) red[warp] = v;
    __syncthreads();
    double t = 0.0;
#pragma unroll
    for (int w = 0; w < kWarpsA; ++w) t += red[w];
    __syncthreads();
    return t;
}

__global__ void __launch_bounds__(kThreadsA) accept_stochastic_kernel(StochArgs a) {
    __shared__ int s_par[kMaxNodes], s_drf[kMaxNodes], s_path[kMaxDepth];
    __shared__ double s_z[kMaxNodes];  // normalizers of the residual at the current node
    __shared__ double s_red[kWarpsA + 1];
    __shared__ int s_bad, s_idx;
    const int b = blockIdx.x, tid = threadIdx.x;
    const int V = a.V, md = a.max_depth;

    pdl_wait();
    pdl_launch_next();
    int off = 0, n = 0;
    const bool range = request_range(a.node_offsets, b, a.T, a.max_nodes, off, n);
    if (tid == 0) s_bad = range ? 0 : 1;
    __syncthreads();
    if (range)
        for (int i = tid; i < n; i += kThreadsA) {
            const int p = a.parent[off + i], x = a.draft[off + i];
            s_par[i] = p;
            s_drf[i] = x;
            if (p < -1 || p >= i || x < 0 || x >= V) s_bad = 1;
        }
    __syncthreads();
    int32_t *path = a.path + (size_t)b * md;
    if (s_bad) {
        if (tid == 0) {
            report(a.status, TV_ERR_TREE);
            a.len[b] = 0;
            a.bonus[b] = -1;
        }
        for (int m = tid; m < md; m += kThreadsA) path[m] = -1;
        return;
    }

    const float *P = a.root_p + (size_t)b * V;
    const float *Q = a.root_q + (size_t)b * V;
    int cur = -1, L = 0, nz = 0;
    bool too_deep = false;
    for (;;) {  // every thread takes the same branches: all values below are uniform
        bool found = false;
        for (int c = cur + 1; c < n; ++c) {
            if (s_par[c] != cur) continue;
            const int x = s_drf[c];
            const double lhs = a.u_accept[off + c] * (double)Q[x];
            const double rhs = residual(P, Q, x, s_z, nz);
            if (lhs < rhs) {
                if (L >= md) {
                    too_deep = true;
                    break;
                }
                if (tid == 0) s_path[L] = c;
                ++L;
                cur = c;
                P = a.node_p + (size_t)(off + c) * V;
                Q = a.node_q + (size_t)(off + c) * V;
                nz = 0;
                found = true;
                break;
            }
            // rejected: the residual's normalizer over the whole row
            double part = 0.0;
            for (int y = tid; y < V; y += kThreadsA)
                part += fmax(residual(P, Q, y, s_z, nz) - (double)Q[y], 0.0);
            const double z = block_sum(part, s_red);
            if (tid == 0) s_z[nz] = z;
            __syncthreads();
            ++nz;
        }
        if (!found || too_deep) break;
    }
    if (too_deep) {
        if (tid == 0) {
            report(a.status, TV_ERR_TREE);
            a.len[b] = 0;
            a.bonus[b] = -1;
        }
        for (int m = tid; m < md; m += kThreadsA) path[m] = -1;
        return;
    }

    // bonus token: the first index whose running sum of the residual exceeds
    // u_bonus * total; each thread owns a contiguous chunk of the row
    const int chunk = (V + kThreadsA - 1) / kThreadsA;
    const int x0 = min(tid * chunk, V), x1 = min(x0 + chunk, V);
    double part = 0.0;
    for (int y = x0; y < x1; ++y) part += residual(P, Q, y, s_z, nz);
    // exclusive scan of the chunk sums
    const int lane = tid & 31, warp = tid >> 5;
    double incl = part;
#pragma unroll
    for (int o = 1; o < 32; o <<= 1) {
        const double t = __shfl_up_sync(0xffffffffu, incl, o);
        if (lane >= o) incl += t;
    }
    if (lane == 31) s_red[warp] = incl;
    if (tid == 0) s_idx = 0x7fffffff;
    __syncthreads();
    double base = 0.0, total = 0.0;
    for (int w = 0; w < kWarpsA; ++w) {
        if (w < warp) base += s_red[w];
        total += s_red[w];
    }
    const double excl = base + incl - part;
    const double target = a.u_bonus[b] * total;
    if (excl <= target && target < excl + part) {
        double run = excl;
        for (int y = x0; y < x1; ++y) {
            run += residual(P, Q, y, s_z, nz);
            if (run > target) {
                atomicMin(&s_idx, y);
                break;
            }
        }
    }
    __syncthreads();
    int idx = s_idx;
    if (idx == 0x7fffffff) {
        // the target fell past the last running sum (rounding): last index with p > 0
        int last = -1;
        for (int y = x0; y < x1; ++y)
            if (residual(P, Q, y, s_z, nz) > 0.0) last = y;
        last = __reduce_max_sync(0xffffffffu, last);
        if (lane == 0) s_red[warp] = (double)last;
        __syncthreads();
        double m = -1.0;
        for (int w = 0; w < kWarpsA; ++w) m = fmax(m, s_red[w]);
        idx = (int)m;
    }
    __syncthreads();
    for (int m = tid; m < md; m += kThreadsA) path[m] = m < L ? s_path[m] : -1;
    if (tid == 0) {
        a.len[b] = L;
        a.bonus[b] = idx;
    }
}

}  // namespace

cudaError_t launch_accept_stochastic(const StochArgs &a, cudaStream_t s) {
    return launch_pdl(accept_stochastic_kernel, dim3((unsigned)a.B), dim3(kThreadsA), 0, s, a);
}

}  // namespace tv
