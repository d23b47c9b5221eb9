// accept_logits.cu -- the target's argmax from its logits, then the greedy walk.
//
// LLM Primer VI ch. 9 §9.1: greedy verification keeps the longest draft prefix
// that matches the target model's own choices and then the target's next choice.
// Here those choices are the argmax of the target's logits at the committed
// context (root row) and after every draft node (node rows); the walk is the one
// of tv_accept_greedy.
//
// Two launches on the caller's stream: one CTA per logits row reduces the row to
// the first index of its largest value and writes it to root_argmax /
// target_argmax; then the walk kernel of tv_accept_greedy reads those.  The
// logits are read once.  (A single launch with one thread-block cluster per
// request was slower: with n + 1 rows over the cluster's CTAs some CTA reduced
// two rows one after the other.)
//
// Order of values: a NaN is larger than any number (the first NaN wins), -0 equals
// +0, otherwise the numeric order of the bf16 values; ties go to the lower index.
#include "tv_internal.cuh"

namespace tv {
namespace {

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

// One CTA per row: rows 0..B-1 are the root rows, B..B+T-1 the node rows.
__global__ void __launch_bounds__(kThreadsL) argmax_rows_kernel(LogitsArgs a) {
    __shared__ int s_red[2 * (kThreadsL / 32) + 2];
    const int row = blockIdx.x;
    pdl_wait();
    pdl_launch_next();
    const uint16_t *src = row < a.B ? a.root_logits + (size_t)row * a.V
                                    : a.node_logits + (size_t)(row - a.B) * a.V;
    const int am = row_argmax(src, a.V, s_red);
    if (threadIdx.x == 0) {
        if (row < a.B)
            a.root_out[row] = am;
        else
            a.target_out[row - a.B] = am;
    }
}

}  // namespace

cudaError_t launch_accept_logits(const LogitsArgs &a, cudaStream_t s) {
    cudaError_t e = launch_pdl(argmax_rows_kernel, dim3((unsigned)(a.B + a.T)), dim3(kThreadsL), 0,
                               s, a);
    if (e != cudaSuccess) return e;
    AcceptArgs w{a.B, a.T, a.max_nodes, a.max_depth, a.node_offsets, a.parent, a.draft,
                 a.target_out, a.root_out, a.len, a.path, a.bonus, a.status};
    return launch_accept(w, s);
}

}  // namespace tv
