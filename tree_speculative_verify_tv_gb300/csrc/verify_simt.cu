// verify_simt.cu -- CUDA-core tree verification, every supported shape.
//
// Tree closed form (Bole summary page, "Core techniques" §1): for node i with
// root path anc*(i) (i included) and G_i = sum_{j in anc*(i)} g_j,
//   o_i = H0^T (e^{G_i} * q_i) + sum_{j in anc*(i)} w_ij v_j,
//   w_ij = sum_c q_ic k_jc e^{G_ic - G_jc}.
// No per-node state is formed; only the factors (g, k, v) are read (§2).
//
// Decay factors are built as products of exp(g) along the path while walking
// from i up to the context, so e^{G_i - G_j} for every ancestor j and e^{G_i}
// itself come out of one walk, exponents never exceed 0 for g <= 0, and no
// difference of large cumulative sums is exponentiated.
//
// Launch: grid (B*H, ceil(max_nodes/32)), 256 threads; one CTA = one
// (request, head) and a tile of 32 nodes.  Warps compute the ancestor weights
// w_ij and the decayed queries; then every thread owns one value column for 8
// nodes and accumulates the context term H0^T q~ (H0 rows read coalesced) and the
// ancestor term sum_j w_ij v_j.
#include "tv_internal.cuh"

namespace tv {
namespace {

constexpr int kThreads = 256;
constexpr int kTile = 32;      // nodes per CTA
constexpr int kGroup = 8;      // nodes per output thread
constexpr int kLaneCh = kMaxDim / 32;

template <typename E, bool DIAG>
__global__ void __launch_bounds__(kThreads) verify_simt_kernel(VerifyArgs a) {
    __shared__ int s_par[kMaxNodes];
    __shared__ int s_dep[kMaxNodes];
    __shared__ int s_anc[kTile][kMaxDepth];
    __shared__ float s_w[kTile][kMaxDepth];
    __shared__ int s_d[kTile];
    __shared__ int s_flag;
    extern __shared__ float s_qt[];  // [kTile][dk] decayed queries e^{G_i} * q_i

    const int unit = blockIdx.x;
    const int b = unit / a.H, h = unit % a.H;
    const int tile0 = blockIdx.y * kTile;
    const int tid = threadIdx.x, lane = tid & 31, warp = tid >> 5;
    const int dk = a.dk, dv = a.dv, H = a.H;
    const E *q = static_cast<const E *>(a.q);
    const E *k = static_cast<const E *>(a.k);
    const E *v = static_cast<const E *>(a.v);

    pdl_wait();
    pdl_launch_next();
    int off, n;
    if (!request_range(a.node_offsets, b, a.T, a.max_nodes, off, n)) {
        if (tid == 0 && h == 0 && blockIdx.y == 0) report(a.status, TV_ERR_TREE);
        return;
    }
    if (tile0 >= n) return;
    const int nt = min(kTile, n - tile0);

    if (!load_check_tree(a.parent, a.depth, off, n, a.max_depth, s_par, s_dep, &s_flag)) {
        if (tid == 0 && h == 0 && blockIdx.y == 0) report(a.status, TV_ERR_TREE);
        for (int e = tid; e < nt * dv; e += kThreads) {
            int t = e / dv, c = e % dv;
            a.out[((size_t)(off + tile0 + t) * H + h) * dv + c] = 0.f;
        }
        return;
    }

    // Root path of each node of the tile, from the node up to the context.
    if (tid < nt) {
        int j = tile0 + tid, d = 0;
        while (j >= 0 && d < kMaxDepth) {
            s_anc[tid][d++] = j;
            j = s_par[j];
        }
        s_d[tid] = d;
    }
    __syncthreads();

    // Ancestor weights and decayed queries, one warp per node.
    for (int t = warp; t < nt; t += kThreads / 32) {
        const size_t row_i = (size_t)(off + tile0 + t) * H + h;
        float qv[kLaneCh], f[kLaneCh];
#pragma unroll
        for (int m = 0; m < kLaneCh; ++m) {
            int c = lane + 32 * m;
            qv[m] = c < dk ? ldg_f(q, row_i * dk + c) : 0.f;
            f[m] = 1.f;
        }
        const int d = s_d[t];
        for (int s = 0; s < d; ++s) {
            const int j = s_anc[t][s];
            const size_t row_j = (size_t)(off + j) * H + h;
            float part = 0.f;
#pragma unroll
            for (int m = 0; m < kLaneCh; ++m) {
                int c = lane + 32 * m;
                if (c < dk) part += qv[m] * ldg_f(k, row_j * dk + c) * f[m];
            }
            part = warp_sum(part);
            if (lane == 0) s_w[t][s] = part;
            // extend the decay product by node j: f = e^{G_i - G_parent(j)}
            if (DIAG) {
#pragma unroll
                for (int m = 0; m < kLaneCh; ++m) {
                    int c = lane + 32 * m;
                    if (c < dk) f[m] *= expf(a.g[row_j * dk + c]);
                }
            } else {
                float e = expf(a.g[row_j]);
#pragma unroll
                for (int m = 0; m < kLaneCh; ++m) f[m] *= e;
            }
        }
#pragma unroll
        for (int m = 0; m < kLaneCh; ++m) {
            int c = lane + 32 * m;
            if (c < dk) s_qt[t * dk + c] = qv[m] * f[m];
        }
    }
    __syncthreads();

    // Outputs: one value column x up to 8 nodes per item.
    const float *H0u = a.H0 + (size_t)unit * dk * dv;
    const int groups = (nt + kGroup - 1) / kGroup;
    for (int item = tid; item < groups * dv; item += kThreads) {
        const int grp = item / dv, c = item % dv;
        const int n0 = grp * kGroup, nn = min(kGroup, nt - n0);
        float acc[kGroup];
#pragma unroll
        for (int x = 0; x < kGroup; ++x) acc[x] = 0.f;
        for (int r = 0; r < dk; ++r) {
            const float hv = __ldg(H0u + (size_t)r * dv + c);
#pragma unroll
            for (int x = 0; x < kGroup; ++x)
                if (x < nn) acc[x] += s_qt[(n0 + x) * dk + r] * hv;
        }
#pragma unroll
        for (int x = 0; x < kGroup; ++x) {
            if (x >= nn) break;
            const int t = n0 + x;
            const int d = s_d[t];
            float o = acc[x];
            for (int s = 0; s < d; ++s) {
                const int j = s_anc[t][s];
                o += s_w[t][s] * ldg_f(v, ((size_t)(off + j) * H + h) * dv + c);
            }
            a.out[((size_t)(off + tile0 + t) * H + h) * dv + c] = o;
        }
    }
}

template <typename E, bool DIAG>
cudaError_t launch_typed(const VerifyArgs &a, cudaStream_t s) {
    dim3 grid((unsigned)(a.B * a.H), (unsigned)((a.max_nodes + kTile - 1) / kTile));
    size_t smem = (size_t)kTile * a.dk * sizeof(float);
    return launch_pdl(verify_simt_kernel<E, DIAG>, grid, dim3(kThreads), smem, s, a);
}

}  // namespace

cudaError_t launch_verify_simt(const VerifyArgs &a, cudaStream_t s) {
    const bool diag = a.decay == TV_DECAY_DIAG;
    if (a.qkv_dtype == TV_BF16)
        return diag ? launch_typed<__nv_bfloat16, true>(a, s) : launch_typed<__nv_bfloat16, false>(a, s);
    return diag ? launch_typed<float, true>(a, s) : launch_typed<float, false>(a, s);
}

}  // namespace tv
