// verify_tc_big.cu -- tree verification of large trees on tcgen05 tensor cores
// (dk = dv = 128, up to 256 nodes).  Two kernels: the staged kernel (second below)
// for trees whose k, decay and v rows fit shared memory, and the node-tiled kernel
// (first) for deeper trees.  The staged kernel also serves per-channel-decay trees
// of 64 or more nodes, where it beats the one-unit kernel.
//
// Tree closed form (Bole summary page, "Core techniques" §1-§2):
//   o_i = H0^T (e^{G_i} * q_i) + sum_{j in anc*(i)} w_ij v_j,
//   w_ij = sum_c q_ic k_jc e^{G_ic - G_jc}
// with anc*(i) the root path of node i including i and G_i the sum of the path's g
// (per key channel for diagonal decay, one value per node for scalar decay).  Only the
// per-token factors are read; no per-node state is formed.
//
// Node-tiled kernel.  One CTA = one (request, head), 256 threads, two CTAs per SM
// at trees of depth <= 16:
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

// ============================================================================
// Staged variant: the whole request's rows in shared memory, both terms on the
// tensor cores.
//
// Persistent: one CTA of 512 threads per SM takes the (request, head) units
// blockIdx.x, + gridDim.x, ... in turn.  The same closed form, reorganised so that
// no ancestor row is fetched through the caches more than once per unit:
//   start    g (n x 128 fp32) and H0 are requested by TMA while the previous unit
//            finishes; H0 is split into bf16 hi + lo and stored transposed in
//            tensor memory (lane = value channel, keys along the columns) as the A
//            operand of the H0 term.
//   phase 0  E = e^g in place, one exponential per node and channel.  In tiles of
//            128 nodes, each node's e^{G_i} * q_i is the product of its root path's
//            E rows (shared memory only) and becomes a bf16 hi/lo B operand row;
//            one thread issues D[:, tile] = H0^T (e^{G} * q) (three products, A from
//            tensor memory) while the next tile's first walks run.
//   phase 1  k (n x 128 bf16) lands by TMA where the B tile was.  The walks:
//            w_ij = q_i . (k_j * e^{G_i - G_j}), eight lanes per node and four nodes
//            per warp (nodes bucketed by depth), four ancestors per round with one
//            transposed reduction.
//   phase 2  v lands by TMA (128-byte swizzled, MN-major: node rows of 64 channels)
//            where E was, then the next unit's H0 (into k's place) and q rows.
//            Per tile of 64 nodes the weights are scattered into a dense bf16
//            hi/lo K-major B operand W[i][j] (zero off the root paths) and one
//            thread issues D[:, tile] += V^T W^T (K = ancestors j < the tile's
//            end); while a tile's MMAs run, the previous tile's columns of D go
//            from tensor memory to the rows of out.  Once the last MMAs are done
//            the next unit's g is requested where E was.
// Shared memory at 256 nodes and depth 16: 128 KB (E, then v + the W tile), 64 KB
// (H0, the B tile, then k), 16 KB w, 8 KB root paths, parents and depths.
// ============================================================================

constexpr int kThreadsS = 512;
constexpr int kWarpsS = kThreadsS / 32;
constexpr int kTile2 = 64;      // nodes per walk round (an H0-term tile is two rounds)
constexpr int kTileW = 64;      // nodes per tree-term tile (MMA N)
constexpr int kBoxRows = 32;    // node rows per TMA box
constexpr uint32_t kA0 = 256;   // tensor-memory column of H0^T (hi; lo 64 columns on)

struct StagedLayout {
    uint32_t npad, r1_off, r2_off, r3_off, anc_off, par_off, dep_off, ord_off, cnt_off, bar_off, misc_off,
        total;
    __host__ __device__ StagedLayout(int max_nodes, int md) {
        npad = align_up(max_nodes > 0 ? max_nodes : 1, kTile2);
        r1_off = 0;                                       // E fp32 rows; then v + W
        r2_off = npad * kDimG * 4;                        // two B tiles (64 KB); then k rows
        r3_off = r2_off + kABytes;                        // w
        anc_off = r3_off + npad * md * 4;
        par_off = align_up(anc_off + npad * md * 2, 16);  // int16 root paths
        dep_off = par_off + npad * 2;
        ord_off = dep_off + npad * 2;                     // walk order (by depth)
        cnt_off = align_up(ord_off + npad * 2, 16);       // per-depth counts
        bar_off = align_up(cnt_off + (md + 1) * 4, 16);
        misc_off = bar_off + 8 * 8;
        total = misc_off + 16 + 1024;
    }
};

template <bool DIAG>
__global__ void __launch_bounds__(kThreadsS, 1)
    verify_tc_staged_kernel(const __grid_constant__ CUtensorMap tm_g,
                            const __grid_constant__ CUtensorMap tm_k,
                            const __grid_constant__ CUtensorMap tm_v, const VerifyArgs a) {
    extern __shared__ uint8_t smem_raw[];
    uint8_t *smem = reinterpret_cast<uint8_t *>(
        (reinterpret_cast<uintptr_t>(smem_raw) + 1023) & ~static_cast<uintptr_t>(1023));
    const int H = a.H, md = a.max_depth;
    const StagedLayout L(a.max_nodes, md);
    const int npad = static_cast<int>(L.npad);
    uint8_t *R1 = smem + L.r1_off;
    uint8_t *R2 = smem + L.r2_off;
    uint8_t *R3 = smem + L.r3_off;
    float *sE = reinterpret_cast<float *>(R1);
    const __nv_bfloat16 *sK = reinterpret_cast<const __nv_bfloat16 *>(R2);
    float *sW = reinterpret_cast<float *>(R3);
    int16_t *sAnc = reinterpret_cast<int16_t *>(smem + L.anc_off);
    int16_t *sPar = reinterpret_cast<int16_t *>(smem + L.par_off);
    int16_t *sDep = reinterpret_cast<int16_t *>(smem + L.dep_off);
    int16_t *sOrd = reinterpret_cast<int16_t *>(smem + L.ord_off);
    int *sCnt = reinterpret_cast<int *>(smem + L.cnt_off);
    uint64_t *bars = reinterpret_cast<uint64_t *>(smem + L.bar_off);
    uint32_t *sTmem = reinterpret_cast<uint32_t *>(smem + L.misc_off);
    int *sFlag = reinterpret_cast<int *>(smem + L.misc_off + 4);

    const int tid = threadIdx.x, warp = tid >> 5, lane = tid & 31;
    const int nunits = a.B * a.H;
    enum { kBarG = 0, kBarH0, kBarK, kBarV, kBarMma0, kBarMma1, kBarMma2, kBars };
    auto bar = [&](int i) { return ptx::smem_addr(&bars[i]); };
    constexpr uint32_t ncols = 512;  // D: columns 0..255; H0^T hi/lo: kA0 .. kA0 + 127
    const __nv_bfloat16 *q = static_cast<const __nv_bfloat16 *>(a.q);

    if (tid == 0) {
        for (int i = 0; i < kBars; ++i) ptx::mbar_init(bar(i), 1);
        ptx::fence_mbar_init();
        if (DIAG) ptx::prefetch_tensormap(&tm_g);
        ptx::prefetch_tensormap(&tm_k);
        ptx::prefetch_tensormap(&tm_v);
    }
    if (warp == 0) {
        ptx::tmem_alloc(ptx::smem_addr(sTmem), ncols);
        ptx::tmem_relinquish();
    }
    ptx::tc_fence_before_sync();
    __syncthreads();
    ptx::tc_fence_after_sync();
    const uint32_t tmem = *sTmem;

    // Every barrier completes once per use; its count of completions consumed so
    // far (the same in every thread) gives the parity of the next one.  The copies
    // in flight are tracked by thread 0 for the bounded waits at the end.
    uint32_t nG = 0, nH0 = 0, nK = 0, nV = 0, nM0 = 0, nM1 = 0, nM2 = 0;
    bool pend_g = false, pend_h0 = false, pend_k = false, pend_v = false;
    // thread 0 waits on a barrier, everyone learns the outcome
    auto wait_all = [&](int i, uint32_t &count) {
        bool ok = true;
        if (tid == 0) ok = ptx::mbar_wait(bar(i), count & 1u, kWaitLimit);
        ok = __syncthreads_and(ok);
        if (ok) ++count;
        else if (tid == 0) report(a.status, TV_ERR_TIMEOUT);
        return ok;
    };

    struct Unit {
        int b, h, off, n;
        bool ok;
    };
    auto unit_at = [&](int u) {
        Unit x;
        x.b = u / H;
        x.h = u % H;
        x.ok = request_range(a.node_offsets, x.b, a.T, a.max_nodes, x.off, x.n);
        return x;
    };
    // a unit's H0 (64 KB, where the phase-0 operand goes later) and g rows, by thread 0
    auto issue_h0 = [&](int u) {
        const float *src = a.H0 + (size_t)u * kDimG * kDimG;
        ptx::mbar_arrive_expect_tx(bar(kBarH0), kABytes);
        for (int c = 0; c < 4; ++c)
            ptx::bulk_g2s(ptx::smem_addr(R2) + c * kChunkG, src + c * kChunkRows * kDimG, kChunkG,
                          bar(kBarH0));
        pend_h0 = true;
    };
    auto issue_g = [&](const Unit &x) {
        const int nb = (x.n + kBoxRows - 1) / kBoxRows;
        ptx::mbar_arrive_expect_tx(bar(kBarG), nb * kBoxRows * kDimG * 4);
        for (int r = 0; r < nb; ++r)
            ptx::tma_load_3d(ptx::smem_addr(R1) + r * kBoxRows * kDimG * 4, &tm_g, 0, x.h,
                             x.off + r * kBoxRows, bar(kBarG));
        pend_g = true;
    };

    // Walks use eight lanes per node, four nodes per warp (node 4 * warp + group of
    // each 64-node round); lane l of a group holds channels 32 t + 4 l + m (t, m < 4),
    // so that a group's loads of one row cover whole 128-byte lines.
    const int grp = lane >> 3, l8 = lane & 7;
    auto qrow = [&](const Unit &x, int i, uint2 (&r)[4]) {
#pragma unroll
        for (int t = 0; t < 4; ++t)
            r[t] = i < x.n ? *reinterpret_cast<const uint2 *>(
                                 q + ((size_t)(x.off + i) * H + x.h) * kDimG + 32 * t + 4 * l8)
                           : make_uint2(0u, 0u);
    };
    auto unpack_q = [&](const uint2 (&r)[4], float (&x)[16]) {
#pragma unroll
        for (int t = 0; t < 4; ++t) {
            const __nv_bfloat162 *q2 = reinterpret_cast<const __nv_bfloat162 *>(&r[t]);
            x[4 * t] = __low2float(q2[0]);
            x[4 * t + 1] = __high2float(q2[0]);
            x[4 * t + 2] = __low2float(q2[1]);
            x[4 * t + 3] = __high2float(q2[1]);
        }
    };
    auto group_max = [&](int x) {
        x = max(x, __shfl_xor_sync(0xffffffffu, x, 8));
        return max(x, __shfl_xor_sync(0xffffffffu, x, 16));
    };

    ptx::grid_dependency_wait();  // inputs may be written by the previous kernel
    ptx::grid_launch_dependents();

    // The CTA takes units blockIdx.x, + gridDim.x, ...  A unit's H0, g and phase-0 q
    // rows are requested while the previous unit finishes (for the first one, here).
    int u = blockIdx.x;
    Unit cur = unit_at(u < nunits ? u : 0);
    uint2 q0[4][4];  // phase-0 rounds (n <= 256: at most four)
    if (u < nunits && cur.ok && cur.n > 0) {
        if (tid == 0) {
            issue_h0(u);
            if (DIAG) issue_g(cur);
        }
#pragma unroll
        for (int t = 0; t < 4; ++t) qrow(cur, t * kTile2 + 4 * warp + grp, q0[t]);
    }
    bool alive = true;  // false after a timed-out wait: the CTA stops
    for (; alive && u < nunits; u += gridDim.x) {
        const int h = cur.h, off = cur.off, n = cur.n;
        const bool have_nodes = cur.ok && n > 0;
        if (!cur.ok && tid == 0 && h == 0) report(a.status, TV_ERR_TREE);
        const int nbox = (n + kBoxRows - 1) / kBoxRows;
        const int un = u + gridDim.x;
        const Unit nxt = unit_at(un < nunits ? un : 0);
        const bool have_next = un < nunits && nxt.ok && nxt.n > 0;

        // ---- the tree: parents precede children, depth = depth(parent) + 1 <=
        // max_depth; then every node's root path (node first), and for scalar decay
        // E = e^g
        if (tid == 0) *sFlag = 0;
        __syncthreads();
        if (have_nodes)
            for (int i = tid; i < n; i += kThreadsS) {
                const int p = a.parent[off + i];
                const int d = a.depth[off + i];
                const bool ok = p >= -1 && p < i && d >= 1 && d <= md;
                sPar[i] = static_cast<int16_t>(ok ? p : -1);
                sDep[i] = static_cast<int16_t>(ok ? d : 1);
                if (!ok) *sFlag = 1;
                if (!DIAG) sE[i] = expf(a.g[(size_t)(off + i) * H + h]);
            }
        __syncthreads();
        if (have_nodes && *sFlag == 0)
            for (int i = tid; i < n; i += kThreadsS) {
                const int p = sPar[i];
                if (sDep[i] != (p < 0 ? 1 : sDep[p] + 1)) *sFlag = 1;
            }
        __syncthreads();
        const bool tree_ok = *sFlag == 0;
        if (have_nodes && tree_ok)
            for (int i = tid; i < n; i += kThreadsS) {
                int j = i;
                const int di = sDep[i];
                for (int d = 0; d < di; ++d) {
                    sAnc[i * md + d] = static_cast<int16_t>(j);
                    j = sPar[j];
                }
            }
        if (have_nodes && !tree_ok) {
            for (int e = tid; e < n * kDimG; e += kThreadsS)
                a.out[((size_t)(off + e / kDimG) * H + h) * kDimG + e % kDimG] = 0.f;
            if (tid == 0 && h == 0) report(a.status, TV_ERR_TREE);
        }
        bool run = have_nodes && tree_ok;

        // the walks' order: nodes bucketed by depth (a warp's four walks then take
        // similar numbers of steps, and siblings read the same ancestor rows together)
        if (run) {
            if (tid <= md) sCnt[tid] = 0;
            __syncthreads();
            int slot = 0;
            if (tid < n) slot = atomicAdd(&sCnt[sDep[tid]], 1);
            __syncthreads();
            if (tid == 0)
                for (int d = 0, acc = 0; d <= md; ++d) {
                    const int c = sCnt[d];
                    sCnt[d] = acc;
                    acc += c;
                }
            __syncthreads();
            if (tid < n) sOrd[sCnt[sDep[tid]] + slot] = static_cast<int16_t>(tid);
        }

        // ---- H0^T as the A operand of the H0 term, in tensor memory: lane = value
        // channel c, two keys per 32-bit column (the even key in the low half), hi in
        // columns kA0 .. kA0 + 63 and lo in the next 64.  Each warp writes its lane
        // quadrant's channels for 32 keys, from H0's rows in shared memory.  (H0 and g
        // were requested for every unit with nodes, so they are consumed even when
        // its tree is malformed.)
        if (have_nodes) {
            alive = wait_all(kBarH0, nH0);
            if (tid == 0 && alive) pend_h0 = false;
            run = run && alive;
        }
        if (run) {
            const int qd = warp & 3, cb = warp >> 2;
            const float *h0 = reinterpret_cast<const float *>(R2) + (32 * cb) * kDimG + 32 * qd + lane;
            float x0[32];
#pragma unroll
            for (int e = 0; e < 32; ++e) x0[e] = h0[e * kDimG];
            uint32_t hi[2][8], lo[2][8];
#pragma unroll
            for (int e = 0; e < 16; ++e) split_pair(x0[2 * e], x0[2 * e + 1], hi[e / 8][e % 8], lo[e / 8][e % 8]);
            const uint32_t ta = tmem + (static_cast<uint32_t>(32 * qd) << 16) + kA0 + 16 * cb;
            ptx::tmem_st_x8(ta, hi[0]);
            ptx::tmem_st_x8(ta + 8, hi[1]);
            ptx::tmem_st_x8(ta + 64, lo[0]);
            ptx::tmem_st_x8(ta + 72, lo[1]);
            ptx::tmem_wait_st();
        }

        // ---- phase 0: E = e^g in place
        if (have_nodes && DIAG && alive) {
            alive = wait_all(kBarG, nG);
            if (tid == 0 && alive) pend_g = false;
            run = run && alive;
            if (run)
                for (int e = tid; e < n * (kDimG / 4); e += kThreadsS) {
                    float4 *p = reinterpret_cast<float4 *>(sE) + e;
                    float4 x = *p;
                    x.x = __expf(x.x); x.y = __expf(x.y); x.z = __expf(x.z); x.w = __expf(x.w);
                    *p = x;
                }
        }
        __syncthreads();  // E is complete; H0 has been read out of R2

        // ---- phase 0: H0 term in tiles of 128 nodes (two 64-node rounds of walks
        // each), the B operand where H0 was: per node the product of its root path's
        // E rows times q, split into bf16 hi/lo rows; D[:, tile] = A_hi B_hi +
        // A_lo B_hi + A_hi B_lo (A from tensor memory)
        const int nround0 = (n + kTile2 - 1) / kTile2;
        const int ntile0 = (n + 2 * kTile2 - 1) / (2 * kTile2);
#pragma unroll
        for (int r = 0; r < 4; ++r) {
            if (!run || r >= nround0) break;
            const int il = 4 * warp + grp, i = r * kTile2 + il;
            float qf[16], f[16];
            unpack_q(q0[r], qf);
            const int di = i < n ? sDep[i] : 0;
            const int dmax = group_max(di);
            const int16_t *anc = sAnc + (i < n ? i : 0) * md;
#pragma unroll
            for (int m = 0; m < 16; ++m) f[m] = 1.f;
            for (int d0 = 0; d0 < dmax; d0 += 4) {
#pragma unroll
                for (int p = 0; p < 4; ++p)
                    if (d0 + p < di) {
                        const int j = anc[d0 + p];
                        if (DIAG) {
#pragma unroll
                            for (int c = 0; c < 4; ++c) {
                                const float4 e = *reinterpret_cast<const float4 *>(sE + j * kDimG + 32 * c + 4 * l8);
                                f[4 * c] *= e.x; f[4 * c + 1] *= e.y; f[4 * c + 2] *= e.z; f[4 * c + 3] *= e.w;
                            }
                        } else {
                            const float e = sE[j];
#pragma unroll
                            for (int m = 0; m < 16; ++m) f[m] *= e;
                        }
                    }
            }
            uint32_t hi[8], lo[8];
#pragma unroll
            for (int e = 0; e < 8; ++e) split_pair(qf[2 * e] * f[2 * e], qf[2 * e + 1] * f[2 * e + 1], hi[e], lo[e]);
            if (r == 2) {  // tile 0's MMAs still read the operand
                alive = wait_all(kBarMma0, nM0);
                run = run && alive;
                if (!run) break;
            }
            const int row = (r & 1) * kTile2 + il;
#pragma unroll
            for (int c = 0; c < 4; ++c) {
                const uint32_t o = swz_offset(row, 32 * c + 4 * l8, 2 * kTile2 * 128);
                *reinterpret_cast<uint2 *>(R2 + o) = make_uint2(hi[2 * c], hi[2 * c + 1]);
                *reinterpret_cast<uint2 *>(R2 + 32768 + o) = make_uint2(lo[2 * c], lo[2 * c + 1]);
            }
            if ((r & 1) == 0 && r + 1 < nround0) continue;  // the tile's second round follows
            // rows of a tile's missing second round are stale: their columns (nodes
            // past n) are never stored
            ptx::fence_proxy_async_smem();
            ptx::tc_fence_before_sync();
            __syncthreads();
            ptx::tc_fence_after_sync();
            if (tid == 0) {
                // descriptors step by adding 16-byte units to the start-address field
                constexpr uint32_t idesc = ptx::idesc_bf16_f32(128, 2 * kTile2);
                const uint64_t bh = ptx::desc_kmajor_sw128(ptx::smem_addr(R2), 1024);
                const uint64_t bl = bh + (32768 >> 4);
#pragma unroll 1
                for (int p = 0; p < 3; ++p)
#pragma unroll
                    for (int kk = 0; kk < 8; ++kk)  // 16-key steps
                        ptx::mma_bf16_ts(tmem + (r >> 1) * 2 * kTile2, tmem + kA0 + (p == 1 ? 64 : 0) + kk * 8,
                                         (p == 2 ? bl : bh) +
                                             (((kk / 4) * (2 * kTile2 * 128) + (kk % 4) * 32) >> 4),
                                         idesc, (p > 0 || kk > 0) ? 1u : 0u);
                ptx::mma_commit(bar(kBarMma0 + (r >> 1)));
            }
        }
        if (run && ntile0 > 0) {
            alive = ntile0 == 1 ? wait_all(kBarMma0, nM0) : wait_all(kBarMma1, nM1);
            run = alive;
        }

        // ---- phase 1: k rows where the B operand was; the walks (the first round's
        // q rows requested while k lands, the others one round ahead)
        auto walk_node = [&](int pos) { return pos < n ? static_cast<int>(sOrd[pos]) : n; };
        uint2 qn[4];
        if (run) qrow(cur, walk_node(4 * warp + grp), qn);
        if (run) {
            if (tid == 0) {
                ptx::mbar_arrive_expect_tx(bar(kBarK), nbox * kBoxRows * kDimG * 2);
                for (int r = 0; r < nbox; ++r)
                    ptx::tma_load_3d(ptx::smem_addr(R2) + r * kBoxRows * kDimG * 2, &tm_k, 0, h,
                                     off + r * kBoxRows, bar(kBarK));
                pend_k = true;
            }
            alive = wait_all(kBarK, nK);
            if (tid == 0 && alive) pend_k = false;
            run = alive;
        }
        if (run) {
            // four nodes per warp in rounds of 64, in the depth order
            for (int base = 4 * warp; base < n; base += 4 * kWarpsS) {
                const int i = walk_node(base + grp);
                float qf[16];
                unpack_q(qn, qf);
                qrow(cur, walk_node(base + grp + 4 * kWarpsS), qn);
                const int di = i < n ? sDep[i] : 0;
                const int dmax = group_max(di);
                const int16_t *anc = sAnc + (i < n ? i : 0) * md;
                for (int d0 = 0; d0 < dmax; d0 += 4) {
                    // partial dot products of four ancestors (the decay advancing
                    // ancestor by ancestor), then one reduction over the group for all four
                    float part[4];
#pragma unroll
                    for (int p = 0; p < 4; ++p) {
                        part[p] = 0.f;
                        if (d0 + p < di) {
                            const int j = anc[d0 + p];
                            const __nv_bfloat16 *kr = sK + j * kDimG + 4 * l8;
                            const float *er = sE + j * kDimG + 4 * l8;
                            const float es = DIAG ? 0.f : sE[j];
#pragma unroll
                            for (int t = 0; t < 4; ++t) {
                                const uint2 kraw = *reinterpret_cast<const uint2 *>(kr + 32 * t);
                                const __nv_bfloat162 *k2 = reinterpret_cast<const __nv_bfloat162 *>(&kraw);
                                part[p] += qf[4 * t] * __low2float(k2[0]) + qf[4 * t + 1] * __high2float(k2[0]) +
                                           qf[4 * t + 2] * __low2float(k2[1]) + qf[4 * t + 3] * __high2float(k2[1]);
                                if (DIAG) {
                                    const float4 e = *reinterpret_cast<const float4 *>(er + 32 * t);
                                    qf[4 * t] *= e.x; qf[4 * t + 1] *= e.y;
                                    qf[4 * t + 2] *= e.z; qf[4 * t + 3] *= e.w;
                                } else {
#pragma unroll
                                    for (int m = 0; m < 4; ++m) qf[4 * t + m] *= es;
                                }
                            }
                        }
                    }
                    // lanes with bit 2 clear keep ancestors 0,1 and the others 2,3;
                    // then bit 1 picks one of the two; bit 0 completes the sum
                    const bool b2 = l8 & 4, b1 = l8 & 2;
                    float x0 = b2 ? part[2] : part[0], x1 = b2 ? part[3] : part[1];
                    const float y0 = b2 ? part[0] : part[2], y1 = b2 ? part[1] : part[3];
                    x0 += __shfl_xor_sync(0xffffffffu, y0, 4);
                    x1 += __shfl_xor_sync(0xffffffffu, y1, 4);
                    float z = b1 ? x1 : x0;
                    z += __shfl_xor_sync(0xffffffffu, b1 ? x0 : x1, 2);
                    z += __shfl_xor_sync(0xffffffffu, z, 1);
                    const int which = (b2 ? 2 : 0) + (b1 ? 1 : 0);  // ancestor d0 + which
                    if ((l8 & 1) == 0 && d0 + which < di) sW[i * md + d0 + which] = z;
                }
            }
        }
        __syncthreads();  // every walk is done: E, k and w are final

        // ---- phase 2: v where E was; dense weight tiles of 64 nodes in the rest of
        // E's space; D += V^T W^T
        const uint32_t slab_v = static_cast<uint32_t>(npad) * 128;  // one 64-channel block of v
        constexpr uint32_t wslab = kTileW * 128;                     // 64 rows x 64 keys
        const uint32_t w_half = static_cast<uint32_t>(npad / 64) * wslab;  // hi (or lo) of a tile
        uint8_t *Wt = R1 + 2 * slab_v;
        if (run && tid == 0) {
            ptx::mbar_arrive_expect_tx(bar(kBarV), 2 * nbox * kBoxRows * 128);
            for (int s = 0; s < 2; ++s)
                for (int r = 0; r < nbox; ++r)
                    ptx::tma_load_3d(ptx::smem_addr(R1) + s * slab_v + r * kBoxRows * 128, &tm_v,
                                     64 * s, h, off + r * kBoxRows, bar(kBarV));
            pend_v = true;
        }
        // R2 (k) is free until the end of the unit: the next unit's H0, after v; and
        // the next unit's phase-0 q rows
        if (alive && have_next) {
            if (tid == 0) issue_h0(un);
#pragma unroll
            for (int t = 0; t < 4; ++t) qrow(nxt, t * kTile2 + 4 * warp + grp, q0[t]);
        }
        // a finished tile's D columns to the rows of out: lanes = value channels of
        // the warp's quadrant, 16 columns per warp
        auto store_tile = [&](int tt) {
            const int quad = warp & 3, col = tt * kTileW + 16 * (warp >> 2);
            if (col >= n) return;
            const int c = 32 * quad + lane;
            const uint32_t tq = tmem + (static_cast<uint32_t>(32 * quad) << 16) + col;
            uint32_t r0[8], r1[8];
            ptx::tmem_ld_x8_nowait(tq, r0);
            ptx::tmem_ld_x8_nowait(tq + 8, r1);
            ptx::tmem_wait_ld();
#pragma unroll
            for (int e = 0; e < 16; ++e) {
                const int i = col + e;
                if (i < n)
                    a.out[((size_t)(off + i) * H + h) * kDimG + c] = __uint_as_float(e < 8 ? r0[e] : r1[e - 8]);
            }
        };
        const int ntile2 = (n + kTileW - 1) / kTileW;
        const int n16 = (n + 15) & ~15;
        for (int t = 0; run && t < ntile2; ++t) {
            const int kt = min(n16, (t + 1) * kTileW);  // keys j < kt can be ancestors
            const int nslab = (kt + 63) / 64;
            if (t >= 1) {  // tile t - 1's MMAs still read W
                alive = wait_all(kBarMma2, nM2);
                run = alive;
                if (!run) break;
                ptx::tc_fence_after_sync();
            }
            for (int e = tid; e < nslab * (wslab / 16); e += kThreadsS) {  // 16-byte pieces
                *reinterpret_cast<uint4 *>(Wt + e * 16) = make_uint4(0u, 0u, 0u, 0u);
                *reinterpret_cast<uint4 *>(Wt + w_half + e * 16) = make_uint4(0u, 0u, 0u, 0u);
            }
            __syncthreads();
            for (int e = tid; e < kTileW * md; e += kThreadsS) {
                const int il = e / md, d = e % md, i = t * kTileW + il;
                if (i < n && d < sDep[i]) {
                    const float w = sW[i * md + d];
                    const int j = sAnc[i * md + d];
                    const uint32_t bits = __float_as_uint(w);
                    const float whi = __uint_as_float(bits & 0xFFFF0000u);
                    const uint32_t o = swz_offset(il, j, wslab);
                    *reinterpret_cast<uint16_t *>(Wt + o) = static_cast<uint16_t>(bits >> 16);
                    *reinterpret_cast<__nv_bfloat16 *>(Wt + w_half + o) = __float2bfloat16_rn(w - whi);
                }
            }
            if (t == 0) {
                alive = wait_all(kBarV, nV);
                run = alive;
                if (!run) break;
                if (tid == 0) pend_v = false;
                // rows n .. n16-1 of v (another request's, or zero past the end) meet
                // zero weights; clear them so that no non-finite value gets in
                for (int e = tid; e < (n16 - n) * 2 * 8; e += kThreadsS) {
                    const int row = n + e / 16, s = (e / 8) & 1, piece = e & 7;
                    *reinterpret_cast<uint4 *>(R1 + s * slab_v + row * 128 + piece * 16) =
                        make_uint4(0u, 0u, 0u, 0u);
                }
            }
            ptx::fence_proxy_async_smem();
            ptx::tc_fence_before_sync();
            __syncthreads();
            ptx::tc_fence_after_sync();
            if (tid == 0) {
                constexpr uint32_t idesc = ptx::idesc_bf16_f32(128, kTileW) | (1u << 15);  // A MN-major
                const uint64_t a0 = ptx::desc_mnmajor_sw128(ptx::smem_addr(R1), slab_v, 1024);
                const uint64_t wh = ptx::desc_kmajor_sw128(ptx::smem_addr(Wt), 1024), wl = wh + (w_half >> 4);
#pragma unroll 4
                for (int kk = 0; kk < kt / 16; ++kk) {
                    const uint64_t ad = a0 + ((kk * 2048) >> 4);
                    const uint32_t wo = ((kk / 4) * wslab + (kk % 4) * 32) >> 4;
                    ptx::mma_bf16(tmem + t * kTileW, ad, wh + wo, idesc, 1u);
                    ptx::mma_bf16(tmem + t * kTileW, ad, wl + wo, idesc, 1u);
                }
                ptx::mma_commit(bar(kBarMma2));
            }
            if (t >= 1) store_tile(t - 1);  // while tile t's MMAs run
        }
        if (run && ntile2 > 0) {
            alive = wait_all(kBarMma2, nM2);
            run = alive;
        }
        ptx::tc_fence_after_sync();

        // R1 is free (the tree MMAs are done): the next unit's g, while the last tile
        // is stored
        if (alive && have_next && tid == 0 && DIAG) issue_g(nxt);
        if (run && ntile2 > 0) store_tile(ntile2 - 1);
        // shared and tensor memory are rewritten by the next unit
        ptx::tc_fence_before_sync();
        __syncthreads();
        ptx::tc_fence_after_sync();
        cur = nxt;
    }

    // copies still in flight after a failed wait: one more bounded wait each before
    // the CTA (and its shared memory) goes away
    if (tid == 0) {
        if (pend_g) ptx::mbar_wait(bar(kBarG), nG & 1u, kWaitLimit);
        if (pend_h0) ptx::mbar_wait(bar(kBarH0), nH0 & 1u, kWaitLimit);
        if (pend_k) ptx::mbar_wait(bar(kBarK), nK & 1u, kWaitLimit);
        if (pend_v) ptx::mbar_wait(bar(kBarV), nV & 1u, kWaitLimit);
    }
    ptx::tc_fence_before_sync();
    __syncthreads();
    if (warp == 0) ptx::tmem_dealloc(tmem, ncols);
}

bool encode_staged_map(CUtensorMap *tm, const void *base, CUtensorMapDataType dt, int esize,
                       int H, int T, int box_w, CUtensorMapSwizzle swz) {
    // rows of 128 elements per (node, head): dims (128, H, T), one head and 32 nodes per box
    const cuuint64_t dims[3] = {(cuuint64_t)kDimG, (cuuint64_t)H, (cuuint64_t)T};
    const cuuint64_t strides[2] = {(cuuint64_t)kDimG * esize, (cuuint64_t)kDimG * esize * H};
    const cuuint32_t box[3] = {(cuuint32_t)box_w, 1, (cuuint32_t)kBoxRows};
    const cuuint32_t estr[3] = {1, 1, 1};
    return encode_fn()(tm, dt, 3, const_cast<void *>(base), dims, strides, box, estr,
                       CU_TENSOR_MAP_INTERLEAVE_NONE, swz, CU_TENSOR_MAP_L2_PROMOTION_L2_256B,
                       CU_TENSOR_MAP_FLOAT_OOB_FILL_NONE) == CUDA_SUCCESS;
}

bool staged_fits(const VerifyArgs &a) {
    return a.max_nodes <= 256 && StagedLayout(a.max_nodes, a.max_depth).total <= kSmemLimit &&
           encode_fn() != nullptr;
}

cudaError_t launch_verify_tc_staged(const VerifyArgs &a, cudaStream_t s) {
    const size_t smem = StagedLayout(a.max_nodes, a.max_depth).total;
    const bool diag = a.decay == TV_DECAY_DIAG;
    CUtensorMap tg, tk, tv_;
    constexpr CUtensorMapDataType BF = CU_TENSOR_MAP_DATA_TYPE_BFLOAT16;
    // scalar decay reads g directly; its map is a placeholder over k
    const bool ok = encode_staged_map(&tk, a.k, BF, 2, a.H, a.T, kDimG, CU_TENSOR_MAP_SWIZZLE_NONE) &&
                    encode_staged_map(&tv_, a.v, BF, 2, a.H, a.T, 64, CU_TENSOR_MAP_SWIZZLE_128B) &&
                    (diag ? encode_staged_map(&tg, a.g, CU_TENSOR_MAP_DATA_TYPE_FLOAT32, 4, a.H, a.T,
                                              kDimG, CU_TENSOR_MAP_SWIZZLE_NONE)
                          : encode_staged_map(&tg, a.k, BF, 2, a.H, a.T, kDimG,
                                              CU_TENSOR_MAP_SWIZZLE_NONE));
    if (!ok) return cudaErrorInvalidValue;
    auto kern = diag ? verify_tc_staged_kernel<true> : verify_tc_staged_kernel<false>;
    cudaError_t e = configure_smem_once(kern, true);
    if (e != cudaSuccess) return e;
    // persistent: one CTA per SM, each taking every gridDim-th (request, head) unit
    int dev = 0, sms = 0;
    e = cudaGetDevice(&dev);
    if (e != cudaSuccess) return e;
    e = cudaDeviceGetAttribute(&sms, cudaDevAttrMultiProcessorCount, dev);
    if (e != cudaSuccess) return e;
    const long long units = (long long)a.B * a.H;
    const unsigned grid = (unsigned)(units < sms ? units : sms);
    return launch_pdl(kern, dim3(grid), dim3(kThreadsS), smem, s, tg, tk, tv_, a);
}

}  // namespace

bool verify_tc_big_supported(const VerifyArgs &a) {
    return a.qkv_dtype == TV_BF16 && a.dk == kDimG && a.dv == kDimG &&
           a.max_nodes <= kMaxNodes &&
           (staged_fits(a) || BigLayout(a.max_depth).total <= kSmemLimit);
}

bool verify_tc_staged_preferred(const VerifyArgs &a) {
    return a.decay == TV_DECAY_DIAG && a.max_nodes >= 64 && verify_tc_big_supported(a) &&
           staged_fits(a);
}

cudaError_t launch_verify_tc_big(const VerifyArgs &a, cudaStream_t s) {
    if (!verify_tc_big_supported(a)) return cudaErrorNotSupported;
    if (staged_fits(a)) return launch_verify_tc_staged(a, s);
    const size_t smem = BigLayout(a.max_depth).total;
    const bool diag = a.decay == TV_DECAY_DIAG;
    auto kern = diag ? verify_tc_big_kernel<true> : verify_tc_big_kernel<false>;
    cudaError_t e = configure_smem_once(kern, true);
    if (e != cudaSuccess) return e;
    return launch_pdl(kern, dim3((unsigned)(a.B * a.H)), dim3(kThreadsG), smem, s, a);
}

}  // namespace tv
