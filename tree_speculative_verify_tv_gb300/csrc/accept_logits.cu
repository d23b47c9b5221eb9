// accept_logits.cu -- the target's argmax from its logits and the greedy walk, in
// one launch.
//
// LLM Primer VI ch. 9 §9.1: greedy verification keeps the longest draft prefix
// that matches the target model's own choices and then the target's next choice.
// Here those choices are the argmax of the target's logits at the committed
// context (root row) and after every draft node (node rows); the walk is the one
// of tv_accept_greedy.
//
// Launch: one thread-block cluster of kCluster CTAs per request.  The request's
// n + 1 rows are dealt round-robin to the cluster's CTAs; a CTA reduces a row of V
// bf16 logits with 16-byte loads (eight per thread in flight) to the first index
// of its largest value and stores it into the shared memory of the cluster's
// first CTA.  After one cluster barrier that CTA runs the walk on its shared
// memory.  The logits are read once; no global scratch memory is used.
//
// Order of values: a NaN is larger than any number (the first NaN wins), -0 equals
// +0, otherwise the numeric order of the bf16 values; ties go to the lower index.
#include "greedy_walk.cuh"

namespace tv {
namespace {

constexpr int kCluster = 8;
constexpr int kThreadsL = 256;
constexpr int kUnroll = 8;

// Total-order key of a bf16 value: larger value, larger key.
__device__ __forceinline__ uint32_t order_key(uint32_t u) {
    u &= 0xFFFFu;
    if ((u & 0x7FFFu) > 0x7F80u) return 0x10000u;  // NaN
    if (u == 0x8000u) u = 0;                        // -0 -> +0
    return (u & 0x8000u) ? (~u & 0xFFFFu) : (u | 0x8000u);
}

__device__ __forceinline__ void take(uint32_t key, int idx, uint32_t &bk, int &bi) {
    if (key > bk || (key == bk && idx < bi)) {
        bk = key;
        bi = idx;
    }
}

// First index of the largest value of row[0..V); every thread of the block calls
// it and gets the result.  `red` holds two ints per warp.
__device__ int row_argmax(const uint16_t *row, int V, int *red) {
    const int tid = threadIdx.x, lane = tid & 31, warp = tid >> 5;
    uint32_t bk = 0;
    int bi = 0x7fffffff;
    if ((V & 7) == 0) {
        const uint4 *r4 = reinterpret_cast<const uint4 *>(row);
        const int n4 = V >> 3;
        for (int base = tid; base < n4; base += kThreadsL * kUnroll) {
            uint4 x[kUnroll];
#pragma unroll
            for (int u = 0; u < kUnroll; ++u) {
                const int i = base + u * kThreadsL;
                if (i < n4) x[u] = __ldg(r4 + i);
            }
#pragma unroll
            for (int u = 0; u < kUnroll; ++u) {
                const int i = base + u * kThreadsL;
                if (i < n4) {
                    const uint32_t w[4] = {x[u].x, x[u].y, x[u].z, x[u].w};
#pragma unroll
                    for (int e = 0; e < 4; ++e) {
                        take(order_key(w[e]), 8 * i + 2 * e, bk, bi);
                        take(order_key(w[e] >> 16), 8 * i + 2 * e + 1, bk, bi);
                    }
                }
            }
        }
    } else {
        for (int i = tid; i < V; i += kThreadsL) take(order_key(row[i]), i, bk, bi);
    }
    // block reduction: largest key, then the lowest index holding it
    uint32_t wk = __reduce_max_sync(0xffffffffu, bk);
    int wi = (int)__reduce_min_sync(0xffffffffu, bk == wk ? (uint32_t)bi : 0x7fffffffu);
    if (lane == 0) {
        red[2 * warp] = (int)wk;
        red[2 * warp + 1] = wi;
    }
    __syncthreads();
    if (warp == 0) {
        const bool live = lane < kThreadsL / 32;
        const uint32_t k2 = live ? (uint32_t)red[2 * lane] : 0u;
        const int i2 = live ? red[2 * lane + 1] : 0x7fffffff;
        const uint32_t mk = __reduce_max_sync(0xffffffffu, k2);
        const int mi = (int)__reduce_min_sync(0xffffffffu, k2 == mk ? (uint32_t)i2 : 0x7fffffffu);
        if (lane == 0) red[2 * (kThreadsL / 32)] = mi;
    }
    __syncthreads();
    const int r = red[2 * (kThreadsL / 32)];
    __syncthreads();  // `red` is reused by the next row
    return r;
}

__device__ __forceinline__ uint32_t cluster_rank() {
    uint32_t r;
    asm volatile("mov.u32 %0, %%cluster_ctarank;" : "=r"(r));
    return r;
}

// Store to the shared memory of CTA `rank` of this cluster at the address that
// `local` has in this CTA.
__device__ __forceinline__ void st_cluster(int *local, uint32_t rank, int v) {
    uint32_t remote;
    asm volatile("mapa.shared::cluster.u32 %0, %1, %2;"
                 : "=r"(remote)
                 : "r"(static_cast<uint32_t>(__cvta_generic_to_shared(local))), "r"(rank));
    asm volatile("st.shared::cluster.u32 [%0], %1;" ::"r"(remote), "r"(v) : "memory");
}

__device__ __forceinline__ void cluster_sync_all() {
    asm volatile("barrier.cluster.arrive.release.aligned;\n\t"
                 "barrier.cluster.wait.acquire.aligned;" ::: "memory");
}

__global__ void __launch_bounds__(kThreadsL) accept_logits_kernel(LogitsArgs a) {
    __shared__ int s_arg[kMaxNodes + 1];  // first CTA: argmax of every row, root first
    __shared__ int s_par[kMaxNodes], s_drf[kMaxNodes], s_path[kMaxDepth];
    __shared__ int s_red[2 * (kThreadsL / 32) + 1];
    const uint32_t rank = cluster_rank();
    const int b = blockIdx.x / kCluster;
    const int tid = threadIdx.x, lane = tid & 31;
    const int md = a.max_depth;

    pdl_wait();
    pdl_launch_next();
    int off = 0, n = 0;
    const bool range = request_range(a.node_offsets, b, a.T, a.max_nodes, off, n);
    if (range) {
        for (int row = (int)rank; row <= n; row += kCluster) {
            const uint16_t *src = row == 0 ? a.root_logits + (size_t)b * a.V
                                           : a.node_logits + (size_t)(off + row - 1) * a.V;
            const int am = row_argmax(src, a.V, s_red);
            if (tid == 0) {
                st_cluster(&s_arg[row], 0, am);
                if (row == 0 && a.root_out) a.root_out[b] = am;
                if (row > 0 && a.target_out) a.target_out[off + row - 1] = am;
            }
        }
    }
    cluster_sync_all();  // every row's argmax is in the first CTA's shared memory
    if (rank != 0 || tid >= 32) return;

    int32_t *path = a.path + (size_t)b * md;
    int L = -1;
    int32_t t = -1;
    if (range) {
        bool bad = false;
        for (int i = lane; i < n; i += 32) {
            const int p = a.parent[off + i];
            s_par[i] = p;
            s_drf[i] = a.draft[off + i];
            bad |= (p < -1 || p >= i);
        }
        if (!__any_sync(0xffffffffu, bad)) {
            __syncwarp();
            L = warp_greedy_walk_shared(s_par, s_drf, s_arg + 1, n, md, s_arg[0], s_path, &t);
        }
    }
    if (L < 0) {
        if (lane == 0) report(a.status, TV_ERR_TREE);
        L = 0;
        t = -1;
    }
    __syncwarp();
    for (int m = lane; m < md; m += 32) path[m] = m < L ? s_path[m] : -1;
    if (lane == 0) {
        a.len[b] = L;
        a.bonus[b] = t;
    }
}

}  // namespace

cudaError_t launch_accept_logits(const LogitsArgs &a, cudaStream_t s) {
    cudaLaunchConfig_t cfg = {};
    cfg.gridDim = dim3((unsigned)(a.B * kCluster));
    cfg.blockDim = dim3(kThreadsL);
    cfg.dynamicSmemBytes = 0;
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
    cudaError_t e = cudaLaunchKernelEx(&cfg, accept_logits_kernel, a);
    if (e != cudaSuccess) return e;
    return cudaGetLastError();
}

}  // namespace tv
