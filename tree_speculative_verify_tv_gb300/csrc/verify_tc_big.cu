// verify_tc_big.cu -- tree verification of large trees with the context term on
// tcgen05 tensor cores, one node tile after another.
//
// Tree closed form (Bole summary page, "Core techniques" §1-§2):
//   o_i = H0^T (e^{G_i} * q_i) + sum_{j in anc*(i)} w_ij v_j,
//   w_ij = sum_c q_ic k_jc e^{G_ic - G_jc}
// with anc*(i) the root path of node i including i and G_i the sum of the path's g
// (per key channel for diagonal decay, one value per node for scalar decay).  Only the
// per-token factors are read; no per-node state is formed.
//
// For dk = dv = 128 and trees whose operands do not fit the single-tile kernel's
// shared-memory plan (256-node trees).  One CTA = one (request, head), 256 threads,
// two CTAs per SM at trees of depth <= 16:
//   * H0 (64 KB fp32) streams in as four 32-key chunks and is split once, in place,
//     into bf16 hi + lo K-major A operands (value channels x keys); they stay in
//     shared memory for every tile;
//   * nodes go in tiles of 64.  One warp per node walks its root path, reading the
//     ancestors' k and g rows through the L1/L2 caches (the next four ancestors' rows
//     in flight while one is used): w_ij for every ancestor, and
//     at the end e^{G_i} * q_i, split into bf16 hi + lo B operand rows (128-byte
//     swizzled, K-major).  Decay factors are products of exp(g) along the walk, so
//     no difference of large cumulative sums is exponentiated;
//   * one thread issues D = A_hi B_hi + A_lo B_hi + A_hi B_lo (kind::f16, M = 128 value
//     channels, N = 64 nodes, fp32 accumulators in tensor memory); the dropped
//     A_lo B_lo term is below 2^-16 relative;
//   * the epilogue reads D (lane = value channel), adds sum_j w_ij v_j (v rows
//     through the caches) and writes the fp32 output rows.
// Every wait is bounded (TV_ERR_TIMEOUT); malformed trees zero their rows and set
// TV_ERR_TREE.
#include "tc_common.cuh"

namespace tv {
namespace {
using namespace tcc;

constexpr int kThreadsG = 256;
constexpr int kTileN = 64;                              // nodes per tile (MMA N)
constexpr int kDimG = 128;                              // dk = dv
constexpr uint32_t kChunkG = kChunkRows * kDimG * 4;    // 16 KB fp32 chunk -> hi + lo
constexpr uint32_t kABytes = kDimG * kDimG * 4;         // 64 KB
constexpr uint32_t kSlabG = kTileN * 128;               // 64 rows x 128 bytes
constexpr uint32_t kBBytes = 2 * kSlabG;                // one swizzled [64][128] bf16 operand
constexpr uint32_t kTmemG = 64;
constexpr int kPre = 4;                                 // ancestors in flight per walk

struct BigLayout {
    uint32_t a_off, b_off, blo_off, w_off, anc_off, par_off, dep_off, bar_off, misc_off, total;
    __host__ __device__ explicit BigLayout(int md) {
        a_off = 0;
        b_off = a_off + kABytes;
        blo_off = b_off + kBBytes;
        w_off = blo_off + kBBytes;
        anc_off = w_off + kTileN * md * 4;
        par_off = align_up(anc_off + kTileN * md * 4, 16);
        dep_off = par_off + kMaxNodes * 4;
        bar_off = align_up(dep_off + kMaxNodes * 4, 16);
        misc_off = bar_off + 8 * 8;
        total = misc_off + 16 + 1024;  // + slack for 1024-byte base alignment
    }
};

template <bool DIAG>
__global__ void __launch_bounds__(kThreadsG, 2) verify_tc_big_kernel(const VerifyArgs a) {
    extern __shared__ uint8_t smem_raw[];
    uint8_t *smem = reinterpret_cast<uint8_t *>(
        (reinterpret_cast<uintptr_t>(smem_raw) + 1023) & ~static_cast<uintptr_t>(1023));
    const int H = a.H, md = a.max_depth;
    const BigLayout L(md);
    uint8_t *sA = smem + L.a_off;
    uint8_t *sB = smem + L.b_off;
    uint8_t *sBlo = smem + L.blo_off;
    float *sW = reinterpret_cast<float *>(smem + L.w_off);
    int *sAnc = reinterpret_cast<int *>(smem + L.anc_off);
    int *sPar = reinterpret_cast<int *>(smem + L.par_off);
    int *sDep = reinterpret_cast<int *>(smem + L.dep_off);
    uint64_t *bars = reinterpret_cast<uint64_t *>(smem + L.bar_off);
    uint32_t *sTmem = reinterpret_cast<uint32_t *>(smem + L.misc_off);
    int *sFlag = reinterpret_cast<int *>(smem + L.misc_off + 4);

    const int tid = threadIdx.x, warp = tid >> 5, lane = tid & 31;
    const int unit = blockIdx.x, b = unit / H, h = unit % H;
    constexpr int nchunks = kDimG / kChunkRows;
    const uint32_t bar0 = ptx::smem_addr(&bars[0]);         // H0 chunks 0..3
    const uint32_t bar_mma = ptx::smem_addr(&bars[nchunks]);  // one completion per tile
    const __nv_bfloat16 *q = static_cast<const __nv_bfloat16 *>(a.q);
    const __nv_bfloat16 *k = static_cast<const __nv_bfloat16 *>(a.k);
    const __nv_bfloat16 *v = static_cast<const __nv_bfloat16 *>(a.v);

    // ---- prologue that touches no input: barriers, tensor memory
    if (tid == 0) {
        for (int c = 0; c <= nchunks; ++c) ptx::mbar_init(bar0 + 8 * c, 1);
        ptx::fence_mbar_init();
        *sFlag = 0;
    }
    if (warp == 0) {
        ptx::tmem_alloc(ptx::smem_addr(sTmem), kTmemG);
        ptx::tmem_relinquish();
    }
    ptx::tc_fence_before_sync();
    __syncthreads();
    ptx::tc_fence_after_sync();
    const uint32_t tmem = *sTmem;

    ptx::grid_dependency_wait();  // inputs may be written by the previous kernel
    if (tid == 0) {
        const float *src = a.H0 + (size_t)unit * kDimG * kDimG;
        for (int c = 0; c < nchunks; ++c) {
            ptx::mbar_arrive_expect_tx(bar0 + 8 * c, kChunkG);
            ptx::bulk_g2s(ptx::smem_addr(sA) + c * kChunkG, src + c * kChunkRows * kDimG, kChunkG,
                          bar0 + 8 * c);
        }
    }
    int off = 0, n = 0;
    const bool range_ok = request_range(a.node_offsets, b, a.T, a.max_nodes, off, n);
    if (!range_ok && tid == 0 && h == 0) report(a.status, TV_ERR_TREE);
    const bool have_nodes = range_ok && n > 0;
    ptx::grid_launch_dependents();

    // ---- the tree: parents precede children, depth = depth(parent) + 1 <= max_depth
    if (have_nodes)
        for (int i = tid; i < n; i += kThreadsG) {
            const int p = a.parent[off + i];
            sPar[i] = p;
            sDep[i] = a.depth[off + i];
            if (p < -1 || p >= i) *sFlag = 1;
        }
    __syncthreads();
    if (have_nodes && *sFlag == 0)
        for (int i = tid; i < n; i += kThreadsG) {
            const int p = sPar[i];
            const int want = p < 0 ? 1 : sDep[p] + 1;
            if (sDep[i] != want || sDep[i] > md) *sFlag = 1;
        }

    // ---- H0: once every chunk has landed, split it in place into bf16 hi/lo K-major
    // operand rows: per chunk (32 keys), value channels in 8-row groups of 512 bytes
    // (4 core matrices of 8 rows x 8 keys), the hi operand in the first 8 KB, lo in
    // the second
    constexpr int kPer = kDimG * (kChunkRows / 8) / kThreadsG;  // items per thread per chunk
    float hold[nchunks][kPer][8];
    bool got = true;
    if (tid == 0)
        for (int c = 0; c < nchunks; ++c) got = ptx::mbar_wait(bar0 + 8 * c, 0, kWaitLimit) && got;
    got = __syncthreads_and(got);
    const bool tree_ok = *sFlag == 0;
    if (got) {
#pragma unroll
        for (int c = 0; c < nchunks; ++c) {
            const float *f32 = reinterpret_cast<const float *>(sA + c * kChunkG);
#pragma unroll
            for (int t = 0; t < kPer; ++t) {
                const int it = tid + t * kThreadsG;
                const int ch = it % kDimG, kq = it / kDimG;
#pragma unroll
                for (int e = 0; e < 8; ++e) hold[c][t][e] = f32[(kq * 8 + e) * kDimG + ch];
            }
        }
    }
    __syncthreads();  // every H0 read is done before the in-place rewrite
    if (!got && tid == 0) report(a.status, TV_ERR_TIMEOUT);
    if (have_nodes && !tree_ok) {
        for (int e = tid; e < n * kDimG; e += kThreadsG)
            a.out[((size_t)(off + e / kDimG) * H + h) * kDimG + e % kDimG] = 0.f;
        if (tid == 0 && h == 0) report(a.status, TV_ERR_TREE);
    }
    bool run = got && have_nodes && tree_ok;
    if (run) {
#pragma unroll
        for (int c = 0; c < nchunks; ++c) {
            uint8_t *chunk = sA + c * kChunkG;
#pragma unroll
            for (int t = 0; t < kPer; ++t) {
                const int it = tid + t * kThreadsG;
                const int ch = it % kDimG, kq = it / kDimG;
                uint32_t hi[4], lo[4];
#pragma unroll
                for (int e = 0; e < 4; ++e)
                    split_pair(hold[c][t][2 * e], hold[c][t][2 * e + 1], hi[e], lo[e]);
                const uint32_t o = (ch / 8) * 512 + kq * 128 + (ch % 8) * 16;
                *reinterpret_cast<uint4 *>(chunk + o) = make_uint4(hi[0], hi[1], hi[2], hi[3]);
                *reinterpret_cast<uint4 *>(chunk + 8192 + o) = make_uint4(lo[0], lo[1], lo[2], lo[3]);
            }
        }
    }

    // ---- node tiles
    const int quad = warp & 3, half = warp >> 2;
    const uint32_t tq = tmem + (static_cast<uint32_t>(32 * quad) << 16);
    const int c0 = lane * 4;  // a walking lane's four key channels
    int tile = 0;
    for (int t0 = 0; run && t0 < n; t0 += kTileN, ++tile) {
        // walks: one warp per node of the tile.  Lane 0 lists the root path first; the
        // k and g rows of the next kPre ancestors are then always in flight while the
        // current one is used (each is a dependent trip through the caches otherwise)
        for (int il = warp; il < kTileN; il += kThreadsG / 32) {
            const int i = t0 + il;
            float qv[4] = {0.f, 0.f, 0.f, 0.f}, f[4] = {1.f, 1.f, 1.f, 1.f};
            if (i < n) {
                load_bf16x(q + ((size_t)(off + i) * H + h) * kDimG + c0, 4, qv);
                int *anc = sAnc + il * md;
                if (lane == 0)
                    for (int j = i, d = 0; j >= 0; j = sPar[j], ++d) anc[d] = j;
                __syncwarp();
                const int di = sDep[i];
                uint2 kb[kPre];
                float4 gb[kPre];
                auto fetch = [&](int d, uint2 &kr, float4 &gr) {
                    if (d < di) {
                        const size_t row = (size_t)(off + anc[d]) * H + h;
                        kr = *reinterpret_cast<const uint2 *>(k + row * kDimG + c0);
                        if (DIAG)
                            gr = *reinterpret_cast<const float4 *>(a.g + row * kDimG + c0);
                        else
                            gr.x = a.g[row];
                    }
                };
#pragma unroll
                for (int p = 0; p < kPre; ++p) fetch(p, kb[p], gb[p]);
                for (int d0 = 0; d0 < di; d0 += kPre) {
                    // kPre partial dot products (the decay product advances ancestor by
                    // ancestor), the next kPre ancestors' rows requested, then the kPre
                    // warp reductions side by side
                    float part[kPre];
#pragma unroll
                    for (int p = 0; p < kPre; ++p) {
                        part[p] = 0.f;
                        if (d0 + p < di) {
                            const __nv_bfloat162 *k2 = reinterpret_cast<const __nv_bfloat162 *>(&kb[p]);
                            const float kv[4] = {__low2float(k2[0]), __high2float(k2[0]),
                                                 __low2float(k2[1]), __high2float(k2[1])};
#pragma unroll
                            for (int m = 0; m < 4; ++m) part[p] += qv[m] * kv[m] * f[m];
                            if (DIAG) {
                                f[0] *= expf(gb[p].x);
                                f[1] *= expf(gb[p].y);
                                f[2] *= expf(gb[p].z);
                                f[3] *= expf(gb[p].w);
                            } else {
                                const float e = expf(gb[p].x);
#pragma unroll
                                for (int m = 0; m < 4; ++m) f[m] *= e;
                            }
                            fetch(d0 + p + kPre, kb[p], gb[p]);
                        }
                    }
#pragma unroll
                    for (int o = 16; o > 0; o >>= 1)
#pragma unroll
                        for (int p = 0; p < kPre; ++p) part[p] += __shfl_xor_sync(0xffffffffu, part[p], o);
                    if (lane == 0)
#pragma unroll
                        for (int p = 0; p < kPre; ++p)
                            if (d0 + p < di) sW[il * md + d0 + p] = part[p];
                }
            }
            // B row: bf16 hi/lo of e^{G_i} * q_i (zero past the last node)
            uint32_t hi[2], lo[2];
            split_pair(qv[0] * f[0], qv[1] * f[1], hi[0], lo[0]);
            split_pair(qv[2] * f[2], qv[3] * f[3], hi[1], lo[1]);
            const uint32_t o = swz_offset(il, c0, kSlabG);
            *reinterpret_cast<uint2 *>(sB + o) = make_uint2(hi[0], hi[1]);
            *reinterpret_cast<uint2 *>(sBlo + o) = make_uint2(lo[0], lo[1]);
        }
        ptx::fence_proxy_async_smem();
        ptx::tc_fence_before_sync();
        __syncthreads();
        ptx::tc_fence_after_sync();
        // D[c][i] = sum_r A[c][r] B[i][r], one thread issues
        bool mma_ok = true;
        if (tid == 0) {
            const uint32_t idesc = ptx::idesc_bf16_f32(128, kTileN);
            const uint32_t b_hi = ptx::smem_addr(sB), b_lo = ptx::smem_addr(sBlo);
            for (int c = 0; c < nchunks; ++c) {
                const uint32_t a_hi = ptx::smem_addr(sA + c * kChunkG), a_lo = a_hi + 8192;
                const uint32_t pa[3] = {a_hi, a_lo, a_hi}, pb[3] = {b_hi, b_hi, b_lo};
                for (int p = 0; p < 3; ++p) {
                    for (int s2 = 0; s2 < kChunkRows / 16; ++s2) {
                        const int kk = c * (kChunkRows / 16) + s2;  // global 16-key step
                        const uint64_t ad = ptx::desc_kmajor_noswizzle(pa[p] + s2 * 256, 128, 512);
                        const uint64_t bd =
                            ptx::desc_kmajor_sw128(pb[p] + (kk / 4) * kSlabG + (kk % 4) * 32, 1024);
                        ptx::mma_bf16(tmem, ad, bd, idesc, (c > 0 || p > 0 || s2 > 0) ? 1u : 0u);
                    }
                }
            }
            ptx::mma_commit(bar_mma);
            mma_ok = ptx::mbar_wait(bar_mma, tile & 1, kWaitLimit);
        }
        if (!__syncthreads_and(mma_ok)) {
            if (tid == 0) report(a.status, TV_ERR_TIMEOUT);
            run = false;
            break;
        }
        ptx::tc_fence_after_sync();
        // epilogue: lanes = value channels (quadrant), columns = this warp's half of the
        // tile, 8 nodes at a time; the ancestor term goes depth by depth over those 8
        // nodes, two depths per round, so up to 16 independent v gathers are in flight
        const int c = 32 * quad + lane;
        for (int col = half * (kTileN / 2); col < (half + 1) * (kTileN / 2); col += 8) {
            float acc[8];
            ptx::tmem_ld_x8(tq + col, acc);
            int dd[8], dmax = 0;
#pragma unroll
            for (int e = 0; e < 8; ++e) {
                const int i = t0 + col + e;
                dd[e] = i < n ? sDep[i] : 0;
                dmax = max(dmax, dd[e]);
            }
            for (int d = 0; d < dmax; d += 2) {
                float vv[2][8], ww[2][8];
#pragma unroll
                for (int u = 0; u < 2; ++u)
#pragma unroll
                    for (int e = 0; e < 8; ++e) {
                        const int il = col + e;
                        const bool in = d + u < dd[e];
                        const int j = in ? sAnc[il * md + d + u] : 0;
                        ww[u][e] = in ? sW[il * md + d + u] : 0.f;
                        vv[u][e] = in ? __bfloat162float(v[((size_t)(off + j) * H + h) * kDimG + c])
                                      : 0.f;
                    }
#pragma unroll
                for (int u = 0; u < 2; ++u)
#pragma unroll
                    for (int e = 0; e < 8; ++e) acc[e] += ww[u][e] * vv[u][e];
            }
#pragma unroll
            for (int e = 0; e < 8; ++e) {
                const int i = t0 + col + e;
                if (i < n) a.out[((size_t)(off + i) * H + h) * kDimG + c] = acc[e];
            }
        }
        ptx::tc_fence_before_sync();
        __syncthreads();  // D, B and the weights are rewritten by the next tile
        ptx::tc_fence_after_sync();
    }

    // after a timed-out wait, give the copies one more bounded wait before the CTA
    // (and its shared memory) goes away
    if (tid == 0 && !got)
        for (int c = 0; c < nchunks; ++c) ptx::mbar_wait(bar0 + 8 * c, 0, kWaitLimit);
    ptx::tc_fence_before_sync();
    __syncthreads();
    if (warp == 0) ptx::tmem_dealloc(tmem, kTmemG);
}

}  // namespace

bool verify_tc_big_supported(const VerifyArgs &a) {
    return a.qkv_dtype == TV_BF16 && a.dk == kDimG && a.dv == kDimG &&
           a.max_nodes <= kMaxNodes && BigLayout(a.max_depth).total <= kSmemLimit;
}

cudaError_t launch_verify_tc_big(const VerifyArgs &a, cudaStream_t s) {
    if (!verify_tc_big_supported(a)) return cudaErrorNotSupported;
    const size_t smem = BigLayout(a.max_depth).total;
    const bool diag = a.decay == TV_DECAY_DIAG;
    auto kern = diag ? verify_tc_big_kernel<true> : verify_tc_big_kernel<false>;
    cudaError_t e = cudaFuncSetAttribute(kern, cudaFuncAttributeMaxDynamicSharedMemorySize, (int)smem);
    if (e != cudaSuccess) return e;
    e = cudaFuncSetAttribute(kern, cudaFuncAttributePreferredSharedMemoryCarveout,
                             cudaSharedmemCarveoutMaxShared);
    if (e != cudaSuccess) return e;
    return launch_pdl(kern, dim3((unsigned)(a.B * a.H)), dim3(kThreadsG), smem, s, a);
}

}  // namespace tv
