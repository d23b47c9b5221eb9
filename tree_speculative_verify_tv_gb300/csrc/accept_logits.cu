// accept_logits.cu -- the target's argmax from its logits and the greedy walk, in
// one launch.
//
// LLM Primer VI ch. 9 §9.1: greedy verification keeps the longest draft prefix
// that matches the target model's own choices and then the target's next choice.
// Here those choices are the argmax of the target's logits at the committed
// context (root row) and after every draft node (node rows); the walk is the one
// of tv_accept_greedy.
//
// Launch: one thread-block cluster of 16 CTAs per request (8 where the device
// does not allow 16).  The request's n + 1 rows are dealt round-robin to the
// cluster's CTAs; a CTA reduces a row of V bf16 logits (16-byte loads, 16 per
// thread in flight) to the first index of its largest value and stores it into
// the shared memory of the cluster's first CTA.  After one cluster barrier that
// CTA runs the walk on its shared memory.  The logits are read once; no global
// scratch memory is used.
//
// Order of values: a NaN is larger than any number (the first NaN wins), -0 equals
// +0, otherwise the numeric order of the bf16 values; ties go to the lower index.
#include "greedy_walk.cuh"

namespace tv {
namespace {

constexpr int kClusterMax = 16;  // non-portable cluster size where allowed, else 8
constexpr int kThreadsL = 256;
constexpr int kRegs = 16;         // 16-byte pieces per thread held in registers per chunk

// Total-order key of a bf16 value: larger value, larger key.
__device__ __forceinline__ uint32_t order_key(uint32_t u) {
    u &= 0xFFFFu;
    if ((u & 0x7FFFu) > 0x7F80u) return 0x10000u;  // NaN
    if (u == 0x8000u) u = 0;                        // -0 -> +0
    return (u & 0x8000u) ? (~u & 0xFFFFu) : (u | 0x8000u);
}

__device__ __forceinline__ __nv_bfloat162 as_bf2(uint32_t w) {
    return *reinterpret_cast<const __nv_bfloat162 *>(&w);
}

// Block-wide: the largest key and the lowest index holding it, in every thread.
__device__ __forceinline__ void block_best(uint32_t &bk, int &bi, int *red) {
    const int lane = threadIdx.x & 31, warp = threadIdx.x >> 5;
    const uint32_t wk = __reduce_max_sync(0xffffffffu, bk);
    const int wi = (int)__reduce_min_sync(0xffffffffu, bk == wk ? (uint32_t)bi : 0x7fffffffu);
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
        if (lane == 0) {
            red[2 * (kThreadsL / 32)] = (int)mk;
            red[2 * (kThreadsL / 32) + 1] = mi;
        }
    }
    __syncthreads();
    bk = (uint32_t)red[2 * (kThreadsL / 32)];
    bi = red[2 * (kThreadsL / 32) + 1];
    __syncthreads();  // `red` is reused
}

// First index of the largest value of row[0..V); every thread of the block calls
// it and gets the result.  V % 8 == 0: the row goes through registers in chunks of
// kRegs 16-byte pieces per thread; per chunk a packed bf16 maximum (NaN wins)
// gives the chunk's largest value, then each thread looks for the first of its
// values equal to it (a NaN when the maximum is a NaN; -0 equals +0) and the block
// keeps the lowest index.  Chunks are combined in order, an earlier chunk winning
// ties.  Other V: one value per thread at a time through the order key.
__device__ int row_argmax(const uint16_t *row, int V, int *red) {
    const int tid = threadIdx.x;
    uint32_t bk = 0;
    int bi = 0x7fffffff;
    if ((V & 7) == 0) {
        const uint4 *r4 = reinterpret_cast<const uint4 *>(row);
        const int n4 = V >> 3;
        for (int base = 0; base < n4; base += kThreadsL * kRegs) {
            uint4 x[kRegs];
#pragma unroll
            for (int u = 0; u < kRegs; ++u) {
                const int i = base + tid + u * kThreadsL;
                x[u] = i < n4 ? __ldg(r4 + i) : make_uint4(0xFF80FF80u, 0xFF80FF80u, 0xFF80FF80u,
                                                            0xFF80FF80u);  // -inf padding
            }
            __nv_bfloat162 m2 = as_bf2(0xFF80FF80u);
#pragma unroll
            for (int u = 0; u < kRegs; ++u) {
                m2 = __hmax2_nan(m2, as_bf2(x[u].x));
                m2 = __hmax2_nan(m2, as_bf2(x[u].y));
                m2 = __hmax2_nan(m2, as_bf2(x[u].z));
                m2 = __hmax2_nan(m2, as_bf2(x[u].w));
            }
            const uint32_t mw = *reinterpret_cast<const uint32_t *>(&m2);
            uint32_t ck = max(order_key(mw), order_key(mw >> 16));
            int ci = 0;
            block_best(ck, ci, red);  // chunk maximum (index unused yet)
            // first index of the chunk maximum among this thread's values
            const bool nan_max = ck == 0x10000u;
            const uint32_t mbits = ck >= 0x8000u ? (ck & 0x7FFFu) : (~ck & 0xFFFFu);
            const __nv_bfloat162 M2 = as_bf2(mbits | (mbits << 16));
            int first = 0x7fffffff;
#pragma unroll
            for (int u = 0; u < kRegs; ++u) {
                const int i = base + tid + u * kThreadsL;
                if (first == 0x7fffffff && i < n4) {
                    const uint32_t w[4] = {x[u].x, x[u].y, x[u].z, x[u].w};
#pragma unroll
                    for (int e = 3; e >= 0; --e) {
                        const __nv_bfloat162 h2 = as_bf2(w[e]);
                        bool lo, hi;
                        if (nan_max) {
                            lo = __hisnan(__low2bfloat16(h2));
                            hi = __hisnan(__high2bfloat16(h2));
                        } else {
                            lo = __heq(__low2bfloat16(h2), __low2bfloat16(M2));
                            hi = __heq(__high2bfloat16(h2), __low2bfloat16(M2));
                        }
                        if (hi) first = 8 * i + 2 * e + 1;
                        if (lo) first = 8 * i + 2 * e;
                    }
                }
            }
            uint32_t fk = ck;
            block_best(fk, first, red);
            if (ck > bk) {  // an equal maximum in a later chunk does not replace it
                bk = ck;
                bi = first;
            }
        }
        return bi;
    }
    for (int i = tid; i < V; i += kThreadsL) {
        const uint32_t key = order_key(row[i]);
        if (key > bk || (key == bk && i < bi)) {
            bk = key;
            bi = i;
        }
    }
    block_best(bk, bi, red);
    return bi;
}

__device__ __forceinline__ uint32_t cluster_rank() {
    uint32_t r;
    asm volatile("mov.u32 %0, %%cluster_ctarank;" : "=r"(r));
    return r;
}

__device__ __forceinline__ uint32_t cluster_size() {
    uint32_t r;
    asm volatile("mov.u32 %0, %%cluster_nctarank;" : "=r"(r));
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
    __shared__ int s_red[2 * (kThreadsL / 32) + 2];
    const uint32_t rank = cluster_rank(), csize = cluster_size();
    const int b = blockIdx.x / (int)csize;
    const int tid = threadIdx.x, lane = tid & 31;
    const int md = a.max_depth;

    pdl_wait();
    pdl_launch_next();
    int off = 0, n = 0;
    const bool range = request_range(a.node_offsets, b, a.T, a.max_nodes, off, n);
    if (range) {
        for (int row = (int)rank; row <= n; row += (int)csize) {
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
    // 16 CTAs per request where the device allows clusters of 16, else 8
    static const int cluster = [] {
        if (cudaFuncSetAttribute(accept_logits_kernel,
                                 cudaFuncAttributeNonPortableClusterSizeAllowed, 1) != cudaSuccess) {
            cudaGetLastError();
            return 8;
        }
        cudaLaunchConfig_t q = {};
        q.gridDim = dim3(kClusterMax);
        q.blockDim = dim3(kThreadsL);
        cudaLaunchAttribute at;
        at.id = cudaLaunchAttributeClusterDimension;
        at.val.clusterDim.x = kClusterMax;
        at.val.clusterDim.y = 1;
        at.val.clusterDim.z = 1;
        q.attrs = &at;
        q.numAttrs = 1;
        int nclusters = 0;
        if (cudaOccupancyMaxActiveClusters(&nclusters, accept_logits_kernel, &q) != cudaSuccess ||
            nclusters < 1) {
            cudaGetLastError();
            return 8;
        }
        return kClusterMax;
    }();
    const int kCluster = cluster;
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
