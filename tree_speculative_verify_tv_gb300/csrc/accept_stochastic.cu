// accept_stochastic.cu -- stochastic acceptance of draft trees.
//
// LLM Primer VI ch. 9 §9.1: a draft token x drawn from the draft distribution q
// is accepted with probability min(1, p(x)/q(x)), p the target distribution; after
// a rejection the emitted token is drawn from the normalized residual (p - q)_+,
// which keeps the output distribution equal to sampling the target.  On a tree
// (reading): the children of the current node are tried in index order, each
// against the current residual (a rejection replaces p by (p - q)_+ / sum, unchanged
// when that sum is 0); the first accepted child becomes the current node, with its
// own p and q; when no child is accepted, the bonus token is drawn from the current
// residual by inverse CDF with the request's uniform.  The acceptance test for child c
// is u_accept[c] * q(x) < p(x).  The uniforms are inputs.
//
// One CTA of 1024 threads per request.  Every sibling of a node is tested against the
// same q, so the residual after any number of rejections has a closed form:
//     p_k(y) = max(p(y) - a_k q(y), 0) / b_k,   a_0 = 0, b_0 = 1,
// and a rejection gives a_{k+1} = a_k + b_k, b_{k+1} = T = sum_y max(p(y) - a_{k+1} q(y), 0)
// (= b_k Z_{k+1}; a zero sum leaves (a, b) unchanged).  By induction: where
// p - a_k q <= 0 the next residual is 0 as well, elsewhere max(p_k - q, 0) / Z_{k+1} =
// max(p - (a_k + b_k) q, 0) / (b_k Z_{k+1}).  So a rejection costs one pass over the
// row and no scratch memory.
//
// Precision: a, b, the tested residual p_k(x) and every comparison are fp64.  The
// row sums T (and the bonus token's running sums) are formed from per-element terms
// computed in double-float arithmetic -- an fp32 pair (hi, lo) with error-free sums
// and products (Dekker, "A floating-point technique for extending the available
// precision", 1971; Knuth's two-sum) -- which keeps about 48 bits on the fp32 pipe
// (GB300's fp64 rate is a small fraction of its fp32 rate); partial sums are combined
// in double-float within a warp and in fp64 across the 32 warps.
#include "tv_internal.cuh"

namespace tv {
namespace {

constexpr int kThreadsA = 1024;
constexpr int kWarpsA = kThreadsA / 32;

struct DF {
    float hi, lo;
};

// s + e = a + b exactly (no ordering assumption).
__device__ __forceinline__ DF two_sum(float a, float b) {
    const float s = __fadd_rn(a, b);
    const float bb = __fadd_rn(s, -a);
    const float e = __fadd_rn(__fadd_rn(a, -__fadd_rn(s, -bb)), __fadd_rn(b, -bb));
    return {s, e};
}

__device__ __forceinline__ DF df_add(DF x, DF y) {
    DF s = two_sum(x.hi, y.hi);
    const float e = __fadd_rn(s.lo, __fadd_rn(x.lo, y.lo));
    return two_sum(s.hi, e);
}

// max(p - a q, 0) with a = ahi + alo (fp32 pair), p and q fp32.
__device__ __forceinline__ DF term(float p, float q, float ahi, float alo) {
    const float prod = __fmul_rn(ahi, q);
    const float perr = __fmaf_rn(ahi, q, -prod);      // ahi q = prod + perr exactly
    const float small = __fmaf_rn(alo, q, perr);      // a q ~= prod + small
    DF d = two_sum(p, -prod);
    d = two_sum(d.hi, __fadd_rn(d.lo, -small));
    if (d.hi < 0.f || (d.hi == 0.f && d.lo <= 0.f)) return {0.f, 0.f};
    return d;
}

__device__ __forceinline__ double to_double(DF x) { return (double)x.hi + (double)x.lo; }

__device__ __forceinline__ DF shfl_xor_df(DF v, int o) {
    return {__shfl_xor_sync(0xffffffffu, v.hi, o), __shfl_xor_sync(0xffffffffu, v.lo, o)};
}

__device__ __forceinline__ DF shfl_up_df(DF v, int o) {
    return {__shfl_up_sync(0xffffffffu, v.hi, o), __shfl_up_sync(0xffffffffu, v.lo, o)};
}

// Sum over the block, returned to every thread: double-float within warps, fp64
// across the 32 warp sums (one warp).
__device__ __forceinline__ double block_sum(DF v, double *red) {
    const int lane = threadIdx.x & 31, warp = threadIdx.x >> 5;
#pragma unroll
    for (int o = 16; o > 0; o >>= 1) v = df_add(v, shfl_xor_df(v, o));
    if (lane == 0) red[warp] = to_double(v);
    __syncthreads();
    if (warp == 0) {
        double t = red[lane];
#pragma unroll
        for (int o = 16; o > 0; o >>= 1) t += __shfl_xor_sync(0xffffffffu, t, o);
        if (lane == 0) red[kWarpsA] = t;
    }
    __syncthreads();
    const double t = red[kWarpsA];
    __syncthreads();  // red is reused
    return t;
}

// T = sum_y max(P[y] - a Q[y], 0) over the row.
__device__ __forceinline__ double row_sum(const float *P, const float *Q, int V, double a,
                                          double *red) {
    const float ahi = (float)a, alo = (float)(a - (double)ahi);
    DF acc = {0.f, 0.f};
    for (int y = threadIdx.x; y < V; y += kThreadsA)
        acc = df_add(acc, term(__ldg(P + y), __ldg(Q + y), ahi, alo));
    return block_sum(acc, red);
}

__device__ __forceinline__ double residual_at(const float *P, const float *Q, int x, double a,
                                              double b) {
    const double d = (double)P[x] - a * (double)Q[x];
    return d > 0.0 ? d / b : 0.0;
}

__global__ void __launch_bounds__(kThreadsA) accept_stochastic_kernel(StochArgs a) {
    __shared__ int s_par[kMaxNodes], s_drf[kMaxNodes], s_path[kMaxDepth];
    __shared__ double s_red[kWarpsA + 1], s_base[kWarpsA + 1];
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
    double ca = 0.0, cb = 1.0;  // residual coefficients at the current node
    int cur = -1, L = 0;
    bool too_deep = false;
    for (;;) {  // every thread takes the same branches: all values below are uniform
        bool found = false;
        for (int c = cur + 1; c < n; ++c) {
            if (s_par[c] != cur) continue;
            const int x = s_drf[c];
            const double lhs = a.u_accept[off + c] * (double)Q[x];
            if (lhs < residual_at(P, Q, x, ca, cb)) {
                if (L >= md) {
                    too_deep = true;
                    break;
                }
                if (tid == 0) s_path[L] = c;
                ++L;
                cur = c;
                P = a.node_p + (size_t)(off + c) * V;
                Q = a.node_q + (size_t)(off + c) * V;
                ca = 0.0;
                cb = 1.0;
                found = true;
                break;
            }
            // rejected: the next residual, unless it sums to zero
            const double na = ca + cb;
            const double t = row_sum(P, Q, V, na, s_red);
            if (t > 0.0) {
                ca = na;
                cb = t;
            }
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

    // bonus token: the first index whose running sum of the residual exceeds u_bonus
    // times the total (sums of the unnormalized terms; each thread owns a contiguous
    // chunk of the row)
    const float ahi = (float)ca, alo = (float)(ca - (double)ahi);
    const int chunk = (V + kThreadsA - 1) / kThreadsA;
    const int x0 = min(tid * chunk, V), x1 = min(x0 + chunk, V);
    DF pacc = {0.f, 0.f};
    for (int y = x0; y < x1; ++y) pacc = df_add(pacc, term(P[y], Q[y], ahi, alo));
    // exclusive scan of the chunk sums: double-float within warps, fp64 across them
    const int lane = tid & 31, warp = tid >> 5;
    DF incl = pacc;
#pragma unroll
    for (int o = 1; o < 32; o <<= 1) {
        const DF v = shfl_up_df(incl, o);
        if (lane >= o) incl = df_add(incl, v);
    }
    if (lane == 31) s_red[warp] = to_double(incl);
    if (tid == 0) s_idx = 0x7fffffff;
    __syncthreads();
    if (warp == 0) {
        const double w = s_red[lane];
        double v = w;
#pragma unroll
        for (int o = 1; o < 32; o <<= 1) {
            const double u = __shfl_up_sync(0xffffffffu, v, o);
            if (lane >= o) v += u;
        }
        s_base[lane] = v - w;
        if (lane == 31) s_base[kWarpsA] = v;
    }
    __syncthreads();
    const double part = to_double(pacc);
    const double excl = s_base[warp] + (to_double(incl) - part);
    const double total = s_base[kWarpsA];
    const double target = a.u_bonus[b] * total;
    if (excl <= target && target < excl + part) {
        double run = excl;
        for (int y = x0; y < x1; ++y) {
            run += to_double(term(P[y], Q[y], ahi, alo));
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
        for (int y = x0; y < x1; ++y) {
            const DF tv = term(P[y], Q[y], ahi, alo);
            if (tv.hi > 0.f || tv.lo > 0.f) last = y;
        }
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
