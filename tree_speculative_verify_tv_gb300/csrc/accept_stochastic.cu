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
// One cluster of 8 CTAs (256 threads each) per request; CTA r owns the r-th eighth
// of every probability row.  Every sibling of a node is tested against the
// same q, so the residual after any number of rejections has a closed form:
//     p_k(y) = max(p(y) - a_k q(y), 0) / b_k,   a_0 = 0, b_0 = 1,
// and a rejection gives a_{k+1} = a_k + b_k, b_{k+1} = T = sum_y max(p(y) - a_{k+1} q(y), 0)
// (= b_k Z_{k+1}; a zero sum leaves (a, b) unchanged).  By induction: where
// p - a_k q <= 0 the next residual is 0 as well, elsewhere max(p_k - q, 0) / Z_{k+1} =
// max(p - (a_k + b_k) q, 0) / (b_k Z_{k+1}).  So a rejection costs one pass over the
// row and no scratch memory.  A pass adds its slice in every CTA, the eight slice
// sums are exchanged through distributed shared memory, and every CTA adds them in
// rank order, so all CTAs hold bit-identical sums and take identical decisions (the
// cluster's control flow stays uniform, which the cluster barriers rely on).  When a
// node is entered, each CTA starts asynchronous copies of its slice of the node's p
// and q rows into shared memory (the passes read them there) and reads its children's
// test values p(x), q(x) and uniforms in one round trip.
//
// Precision: a, b, the tested residual p_k(x) and every comparison are fp64.  The
// row sums T (and the bonus token's running sums) are formed from per-element terms
// computed in double-float arithmetic -- an fp32 pair (hi, lo) with error-free sums
// and products (Dekker, "A floating-point technique for extending the available
// precision", 1971; Knuth's two-sum) -- which keeps about 48 bits on the fp32 pipe
// (GB300's fp64 rate is a small fraction of its fp32 rate); partial sums are combined
// in double-float within a warp and in fp64 across the 32 warps.
#include <cooperative_groups.h>

#include "tv_internal.cuh"

namespace tv {
namespace {

constexpr int kCluster = 8;     // CTAs per request
constexpr int kThreadsA = 256;
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
// across the warp sums (one warp).
__device__ __forceinline__ double block_sum(DF v, double *red) {
    const int lane = threadIdx.x & 31, warp = threadIdx.x >> 5;
#pragma unroll
    for (int o = 16; o > 0; o >>= 1) v = df_add(v, shfl_xor_df(v, o));
    if (lane == 0) red[warp] = to_double(v);
    __syncthreads();
    if (warp == 0) {
        double t = lane < kWarpsA ? red[lane] : 0.0;
#pragma unroll
        for (int o = 16; o > 0; o >>= 1) t += __shfl_xor_sync(0xffffffffu, t, o);
        if (lane == 0) red[kWarpsA] = t;
    }
    __syncthreads();
    const double t = red[kWarpsA];
    __syncthreads();  // red is reused
    return t;
}

// This CTA's part of T = sum_y max(P[y] - a Q[y], 0): elements [y0, y1), read at
// P[y - base], Q[y - base] (base = 0 for the rows in global memory, y0 for the slice
// staged in shared memory; the same elements in the same order either way).
__device__ __forceinline__ double slice_sum(const float *P, const float *Q, int base, int y0,
                                            int y1, double a, double *red) {
    const float ahi = (float)a, alo = (float)(a - (double)ahi);
    DF acc = {0.f, 0.f};
    for (int y = y0 + threadIdx.x; y < y1; y += kThreadsA)
        acc = df_add(acc, term(P[y - base], Q[y - base], ahi, alo));
    return block_sum(acc, red);
}

__device__ __forceinline__ double residual_at(float px, float qx, double a, double b) {
    const double d = (double)px - a * (double)qx;
    return d > 0.0 ? d / b : 0.0;
}

// 4-byte asynchronous copy global -> shared (no alignment beyond the element), and
// the wait for all of this thread's copies.
__device__ __forceinline__ void cp_async_f32(float *dst, const float *src) {
    asm volatile("cp.async.ca.shared.global [%0], [%1], 4;" ::"r"(
                     static_cast<uint32_t>(__cvta_generic_to_shared(dst))),
                 "l"(src)
                 : "memory");
}
__device__ __forceinline__ void cp_async_wait_all() {
    asm volatile("cp.async.wait_all;" ::: "memory");
}

// STAGED: this CTA's slice of the current node's p and q rows is copied into
// shared memory as the node is entered, so the passes over it (rejections, bonus)
// read shared memory; otherwise they read global memory.
template <bool STAGED>
__global__ void __launch_bounds__(kThreadsA) accept_stochastic_kernel(StochArgs a) {
    namespace cg = cooperative_groups;
    __shared__ int s_par[kMaxNodes], s_drf[kMaxNodes], s_path[kMaxDepth];
    __shared__ double s_red[kWarpsA + 1], s_base[kWarpsA + 1];
    __shared__ double s_slot[2];     // this CTA's slice sum of the last two passes
    __shared__ double s_tot;         // this CTA's slice total for the bonus draw
    __shared__ int s_bad, s_idx, s_last;
    __shared__ float s_px[kMaxNodes], s_qx[kMaxNodes];  // p(x_c), q(x_c) of the tested children
    __shared__ double s_uc[kMaxNodes];                  // and their uniforms
    extern __shared__ float s_slice[];                  // STAGED: p slice, then q slice
    cg::cluster_group cluster = cg::this_cluster();
    const int rank = (int)cluster.block_rank();
    const int b = blockIdx.x / kCluster, tid = threadIdx.x;
    const int V = a.V, md = a.max_depth;
    const int y0 = (int)((long long)V * rank / kCluster);
    const int y1 = (int)((long long)V * (rank + 1) / kCluster);

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
    if (s_bad) {  // the same verdict in every CTA of the cluster; nothing shared yet
        if (rank == 0) {
            if (tid == 0) {
                report(a.status, TV_ERR_TREE);
                a.len[b] = 0;
                a.bonus[b] = -1;
            }
            for (int m = tid; m < md; m += kThreadsA) path[m] = -1;
        }
        return;
    }

    // the sum over the whole row of this pass's slice sums, in rank order
    int pass = 0;
    auto cluster_sum = [&](double part) {
        const int slot = pass & 1;
        ++pass;
        if (tid == 0) s_slot[slot] = part;
        cluster.sync();  // a slot is rewritten two passes later, after the next barrier
        double t = 0.0;
        for (int r = 0; r < kCluster; ++r) t += *cluster.map_shared_rank(&s_slot[slot], r);
        return t;
    };

    const float *P = a.root_p + (size_t)b * V;
    const float *Q = a.root_q + (size_t)b * V;
    const int slice = (V + kCluster - 1) / kCluster;  // room per row in s_slice
    float *sP = s_slice, *sQ = s_slice + slice;
    // a node is entered: its slice copies start, and its children's test values are
    // read in one round trip (all threads; the copies are waited for before a pass)
    auto enter = [&](int node) {
        if (STAGED)
            for (int y = y0 + tid; y < y1; y += kThreadsA) {
                cp_async_f32(sP + (y - y0), P + y);
                cp_async_f32(sQ + (y - y0), Q + y);
            }
        for (int c = node + 1 + tid; c < n; c += kThreadsA)
            if (s_par[c] == node) {
                const int x = s_drf[c];
                s_px[c] = P[x];
                s_qx[c] = Q[x];
                s_uc[c] = a.u_accept[off + c];
            }
        __syncthreads();
    };
    bool slice_ready = !STAGED;
    auto slice_wait = [&]() {
        if (!slice_ready) {
            cp_async_wait_all();
            __syncthreads();
            slice_ready = true;
        }
    };
    const float *SP = STAGED ? sP : P, *SQ = STAGED ? sQ : Q;  // what the passes read
    const int sbase = STAGED ? y0 : 0;
    double ca = 0.0, cb = 1.0;  // residual coefficients at the current node
    int cur = -1, L = 0;
    bool too_deep = false;
    enter(-1);
    for (;;) {  // every thread of the cluster takes the same branches
        bool found = false;
        for (int c = cur + 1; c < n; ++c) {
            if (s_par[c] != cur) continue;
            const double lhs = s_uc[c] * (double)s_qx[c];
            if (lhs < residual_at(s_px[c], s_qx[c], ca, cb)) {
                if (L >= md) {
                    too_deep = true;
                    break;
                }
                if (tid == 0) s_path[L] = c;
                ++L;
                cur = c;
                P = a.node_p + (size_t)(off + c) * V;
                Q = a.node_q + (size_t)(off + c) * V;
                if (!STAGED) {
                    SP = P;
                    SQ = Q;
                }
                ca = 0.0;
                cb = 1.0;
                // the previous node's copies land and every read of its slice and test
                // values is done before the child's are requested
                cp_async_wait_all();
                __syncthreads();
                slice_ready = !STAGED;
                enter(c);
                found = true;
                break;
            }
            // rejected: the next residual, unless it sums to zero
            const double na = ca + cb;
            slice_wait();
            const double t = cluster_sum(slice_sum(SP, SQ, sbase, y0, y1, na, s_red));
            if (t > 0.0) {
                ca = na;
                cb = t;
            }
        }
        if (!found || too_deep) break;
    }

    int idx = -1;
    if (!too_deep) {
        // bonus token: the first index whose running sum of the residual exceeds
        // u_bonus times the total.  Slice totals give each CTA its base; inside a
        // slice each thread owns a contiguous chunk.
        const float ahi = (float)ca, alo = (float)(ca - (double)ahi);
        const int chunk = (y1 - y0 + kThreadsA - 1) / kThreadsA;
        const int x0 = min(y0 + tid * chunk, y1), x1 = min(x0 + chunk, y1);
        slice_wait();
        DF pacc = {0.f, 0.f};
        for (int y = x0; y < x1; ++y) pacc = df_add(pacc, term(SP[y - sbase], SQ[y - sbase], ahi, alo));
        const int lane = tid & 31, warp = tid >> 5;
        DF incl = pacc;
#pragma unroll
        for (int o = 1; o < 32; o <<= 1) {
            const DF v = shfl_up_df(incl, o);
            if (lane >= o) incl = df_add(incl, v);
        }
        if (lane == 31) s_red[warp] = to_double(incl);
        if (tid == 0) {
            s_idx = 0x7fffffff;
            s_last = -1;
        }
        __syncthreads();
        if (warp == 0) {
            const double w = lane < kWarpsA ? s_red[lane] : 0.0;
            double v = w;
#pragma unroll
            for (int o = 1; o < 32; o <<= 1) {
                const double u = __shfl_up_sync(0xffffffffu, v, o);
                if (lane >= o) v += u;
            }
            if (lane < kWarpsA) s_base[lane] = v - w;
            if (lane == kWarpsA - 1) s_tot = v;
        }
        cluster.sync();
        double base = 0.0, total = 0.0;
        for (int r = 0; r < kCluster; ++r) {
            const double tr = *cluster.map_shared_rank(&s_tot, r);
            if (r < rank) base += tr;
            total += tr;
        }
        const double part = to_double(pacc);
        const double excl = base + s_base[warp] + (to_double(incl) - part);
        const double target = a.u_bonus[b] * total;
        if (excl <= target && target < excl + part) {
            double run = excl;
            for (int y = x0; y < x1; ++y) {
                run += to_double(term(SP[y - sbase], SQ[y - sbase], ahi, alo));
                if (run > target) {
                    atomicMin(&s_idx, y);
                    break;
                }
            }
        }
        // for a target past the last running sum (rounding): the last index with p > 0
        int last = -1;
        for (int y = x0; y < x1; ++y) {
            const DF tv = term(SP[y - sbase], SQ[y - sbase], ahi, alo);
            if (tv.hi > 0.f || tv.lo > 0.f) last = y;
        }
        last = __reduce_max_sync(0xffffffffu, last);
        if (lane == 0) atomicMax(&s_last, last);
        cluster.sync();
        if (rank == 0) {
            int found = 0x7fffffff, lastc = -1;
            for (int r = 0; r < kCluster; ++r) {
                found = min(found, *cluster.map_shared_rank(&s_idx, r));
                lastc = max(lastc, *cluster.map_shared_rank(&s_last, r));
            }
            idx = found != 0x7fffffff ? found : lastc;
        }
    }
    if (rank == 0) {
        if (too_deep) {
            if (tid == 0) {
                report(a.status, TV_ERR_TREE);
                a.len[b] = 0;
                a.bonus[b] = -1;
            }
            for (int m = tid; m < md; m += kThreadsA) path[m] = -1;
        } else {
            for (int m = tid; m < md; m += kThreadsA) path[m] = m < L ? s_path[m] : -1;
            if (tid == 0) {
                a.len[b] = L;
                a.bonus[b] = idx;
            }
        }
    }
    cp_async_wait_all();  // no copy may still be landing when the CTA ends
    cluster.sync();  // no CTA leaves while another may still read its shared memory
}

}  // namespace

cudaError_t launch_accept_stochastic(const StochArgs &a, cudaStream_t s) {
    // the node's p and q slices in shared memory when they fit next to the static arrays
    const size_t slice_bytes = 2 * (size_t)((a.V + kCluster - 1) / kCluster) * sizeof(float);
    const bool staged = slice_bytes <= 160 * 1024;
    auto kern = staged ? accept_stochastic_kernel<true> : accept_stochastic_kernel<false>;
    if (staged) {
        const cudaError_t e = configure_smem_once(kern, false);
        if (e != cudaSuccess) return e;
    }
    cudaLaunchConfig_t cfg = {};
    cfg.gridDim = dim3((unsigned)a.B * kCluster);
    cfg.blockDim = dim3(kThreadsA);
    cfg.dynamicSmemBytes = staged ? slice_bytes : 0;
    cfg.stream = s;
    cudaLaunchAttribute attr[2];
    attr[0].id = cudaLaunchAttributeClusterDimension;
    attr[0].val.clusterDim.x = kCluster;
    attr[0].val.clusterDim.y = 1;
    attr[0].val.clusterDim.z = 1;
    attr[1].id = cudaLaunchAttributeProgrammaticStreamSerialization;
    attr[1].val.programmaticStreamSerializationAllowed = 1;
    cfg.attrs = attr;
    cfg.numAttrs = 2;
    cudaError_t e = cudaLaunchKernelEx(&cfg, kern, a);
    if (e != cudaSuccess) return e;
    return cudaGetLastError();
}

}  // namespace tv
