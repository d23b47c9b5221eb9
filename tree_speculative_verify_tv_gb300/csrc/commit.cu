// commit.cu -- state after the accepted path, rebuilt from the per-token factors.
//
// Bole summary page, "Core techniques" §2: only the accepted path's state is
// restored, h_k = Chain(S_k..S_1) h_0 + accumulated updates.  With the accepted
// path p_1..p_L of request b:
//   H_new[r][c] = alpha_r H0[r][c] + sum_m a_{m,r} v_{p_m}[c]
//   alpha_r  = exp(sum_{l=1..L} g_{p_l, r})
//   a_{m,r}  = exp(sum_{l=m+1..L} g_{p_l, r}) k_{p_m, r}
// (for a scalar decay g_{p,r} = g_p).  A streaming rank-L update of H0: each
// thread reads a float4 of H0, applies the update and writes the float4 of
// H_new, so H_new may be H0 itself.
//
// Launch: grid (B*H, ceil(dk/32)), 256 threads; one CTA = 32 key rows of one
// (request, head).
#include "tv_internal.cuh"

namespace tv {
namespace {

constexpr int kThreads = 256;
constexpr int kRows = 32;

template <typename E, bool DIAG>
__global__ void __launch_bounds__(kThreads) commit_kernel(CommitArgs a) {
    __shared__ int s_path[kMaxDepth];
    __shared__ int s_L, s_flag;
    __shared__ float s_a[kMaxDepth][kRows];
    __shared__ float s_alpha[kRows];
    extern __shared__ float s_v[];  // [L][dv] value rows of the path

    const int unit = blockIdx.x;
    const int b = unit / a.H, h = unit % a.H;
    const int r0 = blockIdx.y * kRows;
    const int rows = min(kRows, a.dk - r0);
    const int tid = threadIdx.x;
    const int dk = a.dk, dv = a.dv, H = a.H;
    const E *k = static_cast<const E *>(a.k);
    const E *v = static_cast<const E *>(a.v);

    int off, n;
    if (!request_range(a.node_offsets, b, a.T, a.max_nodes, off, n)) {
        if (tid == 0 && h == 0 && blockIdx.y == 0) report(a.status, TV_ERR_TREE);
        return;
    }
    if (tid == 0) {
        // the path must be a root path of request b's tree, at most max_depth long
        int L = a.len[b], bad = (L < 0 || L > a.max_depth);
        int prev = -1;
        for (int m = 0; !bad && m < L; ++m) {
            int p = a.path[(size_t)b * a.max_depth + m];
            if (p < 0 || p >= n || a.parent[off + p] != prev) bad = 1;
            else s_path[m] = p;
            prev = p;
        }
        s_L = bad ? 0 : L;
        s_flag = bad;
    }
    __syncthreads();
    if (s_flag) {
        if (tid == 0 && h == 0 && blockIdx.y == 0) report(a.status, TV_ERR_TREE);
        return;
    }
    const int L = s_L;

    for (int e = tid; e < L * dv; e += kThreads) {
        int m = e / dv, c = e % dv;
        s_v[e] = ldg_f(v, ((size_t)(off + s_path[m]) * H + h) * dv + c);
    }
    if (tid < rows) {
        const int r = r0 + tid;
        float s = 0.f;  // sum of g over the path nodes after m
        for (int m = L - 1; m >= 0; --m) {
            const size_t row = (size_t)(off + s_path[m]) * H + h;
            s_a[m][tid] = expf(s) * ldg_f(k, row * dk + r);
            s += DIAG ? a.g[row * dk + r] : a.g[row];
        }
        s_alpha[tid] = expf(s);
    }
    __syncthreads();

    const int c4n = dv / 4;
    const float4 *src = reinterpret_cast<const float4 *>(a.H0 + ((size_t)unit * dk + r0) * dv);
    float4 *dst = reinterpret_cast<float4 *>(a.H_new + ((size_t)unit * dk + r0) * dv);
    for (int item = tid; item < rows * c4n; item += kThreads) {
        const int r = item / c4n, c = (item % c4n) * 4;
        float4 x = src[item];
        const float al = s_alpha[r];
        x.x *= al; x.y *= al; x.z *= al; x.w *= al;
        for (int m = 0; m < L; ++m) {
            const float am = s_a[m][r];
            const float *vm = s_v + m * dv + c;
            x.x += am * vm[0]; x.y += am * vm[1]; x.z += am * vm[2]; x.w += am * vm[3];
        }
        dst[item] = x;
    }
}

template <typename E, bool DIAG>
cudaError_t launch_typed(const CommitArgs &a, cudaStream_t s) {
    dim3 grid((unsigned)(a.B * a.H), (unsigned)((a.dk + kRows - 1) / kRows));
    size_t smem = (size_t)a.max_depth * a.dv * sizeof(float);
    commit_kernel<E, DIAG><<<grid, kThreads, smem, s>>>(a);
    return cudaGetLastError();
}

}  // namespace

cudaError_t launch_commit(const CommitArgs &a, cudaStream_t s) {
    const bool diag = a.decay == TV_DECAY_DIAG;
    if (a.qkv_dtype == TV_BF16)
        return diag ? launch_typed<__nv_bfloat16, true>(a, s) : launch_typed<__nv_bfloat16, false>(a, s);
    return diag ? launch_typed<float, true>(a, s) : launch_typed<float, false>(a, s);
}

}  // namespace tv
