// commit.cu -- state after the accepted path, rebuilt from the per-token factors.
//
// Bole summary page, "Core techniques" §2: only the accepted path's state is
// restored, h_k = Chain(S_k..S_1) h_0 + accumulated updates.  With the accepted
// path p_1..p_L of request b:
//   H_new[r][c] = alpha_r H0[r][c] + sum_m a_{m,r} v_{p_m}[c]
//   alpha_r  = exp(sum_{l=1..L} g_{p_l, r})
//   a_{m,r}  = exp(sum_{l=m+1..L} g_{p_l, r}) k_{p_m, r}
// (for a scalar decay g_{p,r} = g_p).  A streaming rank-L update of H0: each
// thread reads float4s of H0, applies the update and writes the float4s of
// H_new, so H_new may be H0 itself.
//
// Launch: grid (B*H, ceil(dk/rows)), 256 threads; one CTA = 8192/dv key rows of
// one (request, head) (all 128 at dv = 64), 8 float4s per thread.  Memory round trips before the stream are kept to two: the
// H0 float4s, the request's offsets, the accepted length and path go out
// together; then the path's parents (for the root-path check) and its factor
// rows are gathered together.
#include "greedy_walk.cuh"

namespace tv {
namespace {

constexpr int kThreads = 256;
constexpr int kItems = 8;                                 // float4s per thread
constexpr int kRowsMax = kItems * kThreads * 4 / 64;      // 128 key rows at dv = 64

// Key rows per CTA: kItems float4s per thread cover 8192 / dv rows, at most kRowsMax.
__host__ __device__ inline int rows_per_cta(int dk, int dv) {
    int r = kItems * kThreads * 4 / dv;
    if (r > kRowsMax) r = kRowsMax;
    return r < dk ? r : dk;
}

// FUSED: run the greedy walk of the request in warp 0 instead of reading an
// accepted path (tv_accept_commit); the CTA of head 0 and the first row tile
// writes the request's acceptance outputs.
template <typename E, bool DIAG, bool FUSED>
__global__ void __launch_bounds__(kThreads) commit_kernel(CommitArgs a) {
    __shared__ int s_path[kMaxDepth];
    __shared__ int s_par[FUSED ? kMaxNodes : 1], s_drf[FUSED ? kMaxNodes : 1],
        s_tgt[FUSED ? kMaxNodes : 1];
    __shared__ int s_bad, s_bad2, s_L, s_off;
    if (FUSED && threadIdx.x == 0) s_bad2 = 0;
    __shared__ float s_k[kMaxDepth][kRowsMax];
    __shared__ float s_g[kMaxDepth][kRowsMax];
    __shared__ float s_alpha[kRowsMax];
    extern __shared__ float s_v[];  // [L][dv] value rows of the path

    const int unit = blockIdx.x;
    const int b = unit / a.H, h = unit % a.H;
    const int rpc = rows_per_cta(a.dk, a.dv);
    const int r0 = blockIdx.y * rpc;
    const int rows = min(rpc, a.dk - r0);
    const int tid = threadIdx.x, lane = tid & 31;
    const int dk = a.dk, dv = a.dv, H = a.H, md = a.max_depth;
    const E *k = static_cast<const E *>(a.k);
    const E *v = static_cast<const E *>(a.v);

    pdl_wait();
    pdl_launch_next();
    // round trip 1: this thread's H0 float4s, the offsets, the length and the path
    const int c4n = dv / 4;
    const int items = rows * c4n;
    const float4 *src = reinterpret_cast<const float4 *>(a.H0 + ((size_t)unit * dk + r0) * dv);
    float4 x[kItems];
#pragma unroll
    for (int t = 0; t < kItems; ++t)
        if (tid + t * kThreads < items) x[t] = src[tid + t * kThreads];
    if (tid < 32) {
        int off, n;
        const bool range = request_range(a.node_offsets, b, a.T, a.max_nodes, off, n);
        if (FUSED) {
            int L = -1;
            int32_t t = -1;
            if (range)
                L = warp_greedy_walk(a.parent, a.draft, a.target, off, n, md, a.root[b], s_par,
                                     s_drf, s_tgt, s_path, &t);
            const bool bad = L < 0;
            __syncwarp();
            if (h == 0 && blockIdx.y == 0) {  // the request's acceptance outputs, once
                for (int m = lane; m < md; m += 32)
                    a.path_out[(size_t)b * md + m] = (!bad && m < L) ? s_path[m] : -1;
                if (lane == 0) {
                    a.len_out[b] = bad ? 0 : L;
                    a.bonus_out[b] = bad ? -1 : t;
                }
            }
            if (lane == 0) {
                s_bad = bad;
                s_L = bad ? 0 : L;
                s_off = off;
            }
        } else {
            const int L = a.len[b];
            const int p = lane < md ? a.path[(size_t)b * md + lane] : -1;
            bool bad = !range || L < 0 || L > md || (lane < L && (p < 0 || p >= n));
            bad = __any_sync(0xffffffffu, bad);
            if (lane < L && !bad) s_path[lane] = p;
            if (lane == 0) {
                s_bad = bad;
                s_L = bad ? 0 : L;
                s_off = off;
            }
        }
    }
    __syncthreads();
    if (s_bad) {
        if (tid == 0 && h == 0 && blockIdx.y == 0) report(a.status, TV_ERR_TREE);
        return;
    }
    const int L = s_L, off = s_off;

    // round trip 2: root-path check (a walked path is one by construction) and the
    // path's factor rows
    if (!FUSED && tid < 32) {
        bool bad = false;
        if (lane < L) {
            const int par = a.parent[off + s_path[lane]];
            bad = par != (lane == 0 ? -1 : s_path[lane - 1]);
        }
        bad = __any_sync(0xffffffffu, bad);
        if (lane == 0) s_bad2 = bad;
    }
    for (int e = tid; e < L * dv; e += kThreads) {
        const int m = e / dv, c = e % dv;
        s_v[e] = ldg_f(v, ((size_t)(off + s_path[m]) * H + h) * dv + c);
    }
    for (int e = tid; e < L * rows; e += kThreads) {
        const int m = e / rows, r = e % rows;
        const size_t row = (size_t)(off + s_path[m]) * H + h;
        s_k[m][r] = ldg_f(k, row * dk + r0 + r);
        s_g[m][r] = DIAG ? a.g[row * dk + r0 + r] : a.g[row];
    }
    __syncthreads();
    if (s_bad2) {
        if (tid == 0 && h == 0 && blockIdx.y == 0) report(a.status, TV_ERR_TREE);
        return;
    }
    if (tid < rows) {
        float s = 0.f;  // sum of g over the path nodes after m
        for (int m = L - 1; m >= 0; --m) {
            const float gm = s_g[m][tid];
            s_k[m][tid] *= expf(s);  // a_{m,r}
            s += gm;
        }
        s_alpha[tid] = expf(s);
    }
    __syncthreads();

    float4 *dst = reinterpret_cast<float4 *>(a.H_new + ((size_t)unit * dk + r0) * dv);
#pragma unroll
    for (int t = 0; t < kItems; ++t) {
        const int item = tid + t * kThreads;
        if (item >= items) break;
        const int r = item / c4n, c = (item % c4n) * 4;
        float4 y = x[t];
        const float al = s_alpha[r];
        y.x *= al; y.y *= al; y.z *= al; y.w *= al;
        for (int m = 0; m < L; ++m) {
            const float am = s_k[m][r];
            const float4 vm = *reinterpret_cast<const float4 *>(s_v + m * dv + c);
            y.x += am * vm.x; y.y += am * vm.y; y.z += am * vm.z; y.w += am * vm.w;
        }
        dst[item] = y;
    }
}

template <typename E, bool DIAG, bool FUSED>
cudaError_t launch_typed(const CommitArgs &a, cudaStream_t s) {
    const int rpc = rows_per_cta(a.dk, a.dv);
    dim3 grid((unsigned)(a.B * a.H), (unsigned)((a.dk + rpc - 1) / rpc));
    size_t smem = (size_t)a.max_depth * a.dv * sizeof(float);
    const cudaError_t attr = configure_smem_once(commit_kernel<E, DIAG, FUSED>, false);
    if (attr != cudaSuccess) return attr;
    return launch_pdl(commit_kernel<E, DIAG, FUSED>, grid, dim3(kThreads), smem, s, a);
}

template <bool FUSED>
cudaError_t launch_any(const CommitArgs &a, cudaStream_t s) {
    const bool diag = a.decay == TV_DECAY_DIAG;
    if (a.qkv_dtype == TV_BF16)
        return diag ? launch_typed<__nv_bfloat16, true, FUSED>(a, s)
                    : launch_typed<__nv_bfloat16, false, FUSED>(a, s);
    return diag ? launch_typed<float, true, FUSED>(a, s) : launch_typed<float, false, FUSED>(a, s);
}

}  // namespace

cudaError_t launch_commit(const CommitArgs &a, cudaStream_t s) { return launch_any<false>(a, s); }

cudaError_t launch_accept_commit(const CommitArgs &a, cudaStream_t s) {
    return launch_any<true>(a, s);
}

}  // namespace tv
