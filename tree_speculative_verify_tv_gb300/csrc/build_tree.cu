// build_tree.cu -- draft trees by best-first expansion of path scores, on the GPU.
//
// BASTION page, Method §1-§3: the drafter gives, for every position k, a
// distribution q_k over C candidates; a node at depth d holding x_1..x_d has path
// score rho = prod_k q_k(x_k); the tree grows by repeatedly adding the frontier
// node with the largest rho (§2), and, with a step-cost table C(N), stops once the
// estimated speed-up sum(rho) / C(N) would drop (§3).  Node index = order of
// addition, so parents precede children and the result feeds tv_verify directly.
//
// One warp per request.  The frontier is kept lazily: one entry per node that can
// still get children (entry 0 is the context, entry i + 1 node i), holding its best
// child not yet in the tree.  Each step takes the largest entry score; equal scores
// go to the lower entry, then to the lower candidate index.  That is the order in
// which a frontier that receives all C children of a node when the node is added
// (in candidate order) would hand them out.  Scores are fp64 products computed the
// same way as in that formulation, so every choice is made on identical values.
// Comparisons run on integer keys: for non-negative doubles the order of the bit
// patterns is the numeric order (zero of either sign maps to 0, "none" to -1), so
// they stay off GB300's narrow fp64 pipe; one warp per CTA, so requests do not share
// an SM's fp64 unit for the products.
#include "tv_internal.cuh"

namespace tv {
namespace {

constexpr int kWarpsB = 1;

// Order key of a score: a non-negative double's bit pattern, -1 for "none".
__device__ __forceinline__ long long score_key(double s) {
    const long long b = __double_as_longlong(s);  // -0.0 is the most negative pattern
    return b >= 0 ? b : (b == (long long)0x8000000000000000ULL ? 0LL : -1LL);
}

struct WarpBest {
    long long k;
    int i;
};

// Largest key, then smallest i, over the lanes in `mask` (every lane of the mask
// calls with the same mask): three warp reductions, on the key's high word, on its
// low word among the lanes that tie, and on i among the lanes that tie on both.
__device__ __forceinline__ WarpBest warp_best(long long k, int i, unsigned mask = 0xffffffffu) {
    const int hi = static_cast<int>(k >> 32);
    const unsigned lo = static_cast<unsigned>(k);
    const int mh = __reduce_max_sync(mask, hi);
    const unsigned ml = __reduce_max_sync(mask, hi == mh ? lo : 0u);
    const int mi = __reduce_min_sync(mask, (hi == mh && lo == ml) ? i : 0x7fffffff);
    return {static_cast<long long>((static_cast<unsigned long long>(static_cast<unsigned>(mh)) << 32) | ml),
            mi};
}

__global__ void __launch_bounds__(kWarpsB * 32) build_tree_kernel(BuildArgs a) {
    extern __shared__ double s_dyn[];
    const int lane = threadIdx.x & 31, w = threadIdx.x >> 5;
    const int b = blockIdx.x * kWarpsB + w;
    pdl_wait();
    pdl_launch_next();
    if (b >= a.B) return;
    const int C = a.C, cap = a.depth_cap, n = a.n;
    // per warp, in doubles: q [cap][C]; per entry rho (fp64) and score key (int64),
    // best child, depth and taken mask (three 32-bit words, two doubles of room)
    const size_t per_warp = (size_t)cap * C + 4 * (size_t)(n + 1);
    double *sq = s_dyn + w * per_warp;
    double *erho = sq + cap * C;
    long long *escore = reinterpret_cast<long long *>(erho + (n + 1));
    int *ebest = reinterpret_cast<int *>(escore + (n + 1));
    int *edep = ebest + (n + 1);
    uint32_t *emask = reinterpret_cast<uint32_t *>(edep + (n + 1));

    const double *marg = a.marginals + (size_t)b * cap * C;
    for (int e = lane; e < cap * C; e += 32) sq[e] = marg[e];
    __syncwarp();

    // best child of entry e not yet in the tree: largest erho * q, lowest candidate
    auto refresh = [&](int e) {
        const uint32_t taken = emask[e];
        const int d = edep[e];
        long long k = -1;
        if (lane < C && !((taken >> lane) & 1u)) k = score_key(erho[e] * sq[d * C + lane]);
        const WarpBest bb = warp_best(k, lane < C ? lane : 0x7fffffff);
        if (lane == 0) {
            escore[e] = bb.k;
            ebest[e] = bb.i;
        }
        __syncwarp();
    };
    // the same for entries e0 and (when two) e1 side by side, one per half-warp
    // (C <= 16), from their rho, depth and taken mask as the caller holds them
    auto refresh2 = [&](int e0, double rho0, int dep0, uint32_t mask0, int e1, double rho1,
                        int dep1, bool two) {
        const int half = lane >> 4, c = lane & 15;
        const bool act = c < C && (half == 0 || two);
        const int e = half ? e1 : e0;
        long long k = -1;
        if (act && !(((half ? 0u : mask0) >> c) & 1u))
            k = score_key((half ? rho1 : rho0) * sq[(half ? dep1 : dep0) * C + c]);
        const WarpBest bb = warp_best(k, act ? c : 0x7fffffff, half ? 0xffff0000u : 0x0000ffffu);
        if (c == 0 && (half == 0 || two)) {
            escore[e] = bb.k;
            ebest[e] = bb.i;
        }
        __syncwarp();
    };

    if (lane == 0) {
        erho[0] = 1.0;
        edep[0] = 0;
        emask[0] = 0u;
    }
    __syncwarp();
    refresh(0);

    int32_t *par_out = a.parent + (size_t)b * n;
    int32_t *tok_out = a.token + (size_t)b * n;
    double *rho_out = a.rho + (size_t)b * n;
    double total = 0.0;
    double prev_ratio = 0.0;  // total / C(i), as the previous step computed it
    int count = 0;
    // entries 0..n in blocks of `per` consecutive entries per lane (per <= 9)
    const int per = (n + 1 + 31) / 32;
    for (int i = 0; i < n; ++i) {
        long long s = -1;
        int e = 0x7fffffff;
#pragma unroll
        for (int j = 0; j < 9; ++j) {  // entries 0..i exist
            const int k = lane * per + j;
            if (j < per && k <= i) {
                const long long ks = escore[k];
                if (ks > s) {  // ascending k in a lane: the first maximum is the lowest
                    s = ks;
                    e = k;
                }
            }
        }
        const WarpBest best = warp_best(s, e);
        if (best.k < 0) break;  // the frontier is empty
        const int ep = best.i;
        // the entry's score: its key is the bit pattern of the product refresh formed
        // (a zero of either sign reads back as +0)
        const double bs = __longlong_as_double(best.k);
        // the stop rule (sum rho) / C(N) would drop, tested after the frontier update
        // so that the division overlaps it (on a stop, node i is not counted and its
        // outputs are overwritten below); total / C(i) is the previous step's
        // quotient, the same correctly rounded value
        const double ratio = a.cost ? (total + bs) / a.cost[i + 1] : 0.0;
        const bool stop = a.cost && i >= 1 && ratio < prev_ratio;
        const int y = ebest[ep];
        const int d = edep[ep] + 1;
        const double rho_ep = erho[ep];
        const uint32_t mask_ep = emask[ep] | (1u << y);
        if (lane == 0) {
            par_out[i] = ep - 1;
            tok_out[i] = y;
            rho_out[i] = bs;
            emask[ep] = mask_ep;
            // entry of node i: its children join the frontier below the depth cap
            erho[i + 1] = bs;
            edep[i + 1] = d;
            emask[i + 1] = 0u;
            escore[i + 1] = -1;
        }
        __syncwarp();
        if (C <= 16) {
            refresh2(ep, rho_ep, d - 1, mask_ep, i + 1, bs, d, d < cap);
        } else {
            refresh(ep);
            if (d < cap) refresh(i + 1);
        }
        if (stop) break;
        total += bs;
        prev_ratio = ratio;
        count = i + 1;
    }
    for (int i = count + lane; i < n; i += 32) {
        par_out[i] = -1;
        tok_out[i] = -1;
        rho_out[i] = 0.0;
    }
    if (lane == 0) a.count[b] = count;
}

}  // namespace

size_t build_tree_smem_bytes(int C, int depth_cap, int n) {
    return (size_t)kWarpsB * ((size_t)depth_cap * C + 4 * (size_t)(n + 1)) * sizeof(double);
}

cudaError_t launch_build_tree(const BuildArgs &a, cudaStream_t s) {
    const size_t smem = build_tree_smem_bytes(a.C, a.depth_cap, a.n);
    cudaError_t e = configure_smem_once(build_tree_kernel, false);
    if (e != cudaSuccess) return e;
    return launch_pdl(build_tree_kernel, dim3((unsigned)((a.B + kWarpsB - 1) / kWarpsB)),
                      dim3(kWarpsB * 32), smem, s, a);
}

}  // namespace tv
