// verify_tc_fdiag.cu -- per-channel-decay tree verification with all three products of
// a (request, head) unit on tcgen05 tensor cores, one unit per CTA, trees of up to 64
// nodes, dv = 128.
//
// Tree closed form (Bole summary page, "Core techniques" §1), per-channel decay:
//   o_i = H0^T (e^{G_i} * q_i) + sum_{j in anc*(i)} w_ij v_j,
//   w_ij = sum_c q_ic k_jc e^{G_ic - G_jc}
// with anc*(i) the root path of node i including i and G_i the sum of g over it.
// The decay of a pair factors channel by channel, e^{G_ic - G_jc} = e^{G_ic} e^{-G_jc},
// so with the scaled factors
//   q~_i = e^{G_i} * q_i,   k~_j = e^{-G_j} * k_j
// the weights are plain dot products w_ij = q~_i . k~_j on root paths, and
//   o_i = H0^T q~_i + sum_j [j in anc*(i)] (q~_i . k~_j) v_j
// -- three dense products with no decay factor left:
//   D  = H0^T Q~^T            (A = the state rows, MN-major; B = q~)
//   S  = Q~ K~^T              (A = q~ read as M = 128 rows; B = k~)
//   D += V^T W^T, W = S on root paths, 0 elsewhere
// q~, k~ and W are not bf16 values: each is split into bf16 hi + lo parts (hi = the
// upper 16 bits, exact; lo = bf16 of the rest, |x - hi - lo| <= 2^-16 |x|) and each
// product takes the passes hi.hi, lo.hi and hi.lo (lo.lo, below 2^-16 relative, is
// dropped); the fp32 state is split the same way.
//
// Range.  The scaled factors stay finite with normal lo parts while |G_ic| <= 69
// (e^{±69} is about 2^{±100}).  A unit whose path sums leave that range anywhere takes
// its weights from a walk instead (a warp per node from the node up to the context,
// the pair decays formed as products of e^{g} along the path, as the CUDA-core kernel
// does); its context product keeps q~, whose entries then underflow only where
// e^{G_ic} is below fp32's range.
//
// Memory.  The key channels are taken in groups of 64.  The state streams through four
// 8 KB chunk slots (16 key rows each): a chunk's rows are split into bf16 hi / lo parts
// in tensor memory -- the A operand of the context product, lane = value channel -- and
// its slot takes the next group's chunk at once.  A factor slot holds a group's g, q
// and k columns (g: 64 fp32 per node, q and k: 64 bf16 per node, all 128-byte
// swizzled), rewritten in place as the q~ / k~ hi and lo tiles; the next group's
// columns are copied in once the products reading them are done.  About 82 KB of shared
// memory and 256 tensor-memory columns at 64 nodes, so two CTAs share an SM, and one
// CTA's products and copies overlap the other's rewrites.
//
// Roles (416 threads):
//   warps 0-3   state chunks: a thread per value channel reads its 16 key rows of a
//               chunk, splits them and stores the parts to its tensor-memory lane
//   warps 4-11  factors: path sums G of the group's channels (4 or 8 threads per node),
//               range check, q~ hi / lo (then the context products may start), k~ hi /
//               lo; after the last group the weight tiles (the four warps on the score
//               rows' lane quadrants, half the columns each), the walk for out-of-range
//               units, and the v rows past the tree cleared
//   warp 12     copies, offsets, tree checks and ancestor masks (pointer doubling in
//               shared memory), tensor memory; one thread issues the products and
//               refills the factor slot once the score products are done
//   warps 0-7   epilogue: one value channel per lane, half the nodes per warp
// Every wait is bounded (TV_ERR_TIMEOUT); every copy and product in flight is waited
// for (bounded) before tensor memory is freed.  Malformed trees zero their rows and set
// TV_ERR_TREE.
#include "tc_common.cuh"

namespace tv {
namespace {
using namespace tcc;

constexpr int kConvWarps = 4;                           // warps 0-3: state chunks
constexpr int kFacWarps = 8;                            // warps 4-11: factors, weights
constexpr int kCtlWarp = kConvWarps + kFacWarps;        // warp 12: copies, tree, products
constexpr int kThreadsD = (kCtlWarp + 1) * 32;          // 416
constexpr int kDvD = 128;                               // value channels
constexpr int kGrpCh = 64;                              // key channels per group
constexpr int kMaxGroups = 2;                           // dk <= 128
constexpr int kChunkValsD = 2048;                       // state values per chunk
constexpr uint32_t kChunkBytesD = kChunkValsD * 4;      // 8 KB
constexpr int kChunkRowsD = kChunkValsD / kDvD;         // 16 key rows
constexpr int kChunksPerGrp = kGrpCh / kChunkRowsD;     // 4
constexpr int kMaxChunksD = kMaxGroups * kChunksPerGrp; // 8
constexpr int kRing = 3;                                // state chunk slots
constexpr float kLog2eD = 1.4426950408889634f;
constexpr float kGLimit = 69.f;  // |G| bound of the scaled factors

// Shared-memory plan, identical on host and device.  The factor blocks come first, one
// per key-channel group: q | g slab 0 (later q~ lo) | k | g slab 1 (later k~ lo), each
// np rows of 128 B.  Read as M = 128 operands, the q~ hi and lo tiles span 16 KB from
// their starts, inside the plan for every tree size.  After the products the first
// block holds the weight tiles (hi, lo) and, for the walk, the fp32 weights.
struct DiagLayout {
    uint32_t f_off, h_off, v_off, anc_off, par_off, jmp_off, meta_off, bar_off, misc_off, total;
    __host__ __device__ DiagLayout(int np, int ng) {
        f_off = 0;
        h_off = align_up(f_off + ng * 4 * np * 128, 1024);    // the state chunk ring
        v_off = align_up(h_off + kRing * kChunkBytesD, 1024);  // v, two 64-channel blocks
        anc_off = align_up(v_off + 2 * np * 128, 16);
        par_off = anc_off + np * 8;
        jmp_off = par_off + np * 4;
        meta_off = jmp_off + np * 4;
        bar_off = align_up(meta_off + 64, 16);
        misc_off = bar_off + 24 * 8;
        total = misc_off + 32 + 1024;  // + slack for 1024-byte base alignment
    }
};

enum { kMN = 0, kMOff, kMRun, kMZero, kMWalk, kMHave };

struct DiagParams {
    VerifyArgs a;
    int tmem_cols;
    int expire_first_wait;  // test hook: the first wait for a state chunk gives up at once
};

__device__ __forceinline__ float ex2f(float x) {
    float y;
    asm("ex2.approx.ftz.f32 %0, %1;" : "=f"(y) : "f"(x));
    return y;
}

template <int N>
__device__ __forceinline__ void tmem_ld_n(uint32_t taddr, uint32_t (&r)[N]) {
    if constexpr (N == 8)
        ptx::tmem_ld_x8_nowait(taddr, r);
    else if constexpr (N == 16)
        ptx::tmem_ld_x16_nowait(taddr, r);
    else
        ptx::tmem_ld_x32_nowait(taddr, r);
}

__device__ __forceinline__ void bf16x8(const uint4 &raw, float (&x)[8]) {
    const __nv_bfloat162 *p = reinterpret_cast<const __nv_bfloat162 *>(&raw);
#pragma unroll
    for (int e = 0; e < 4; ++e) {
        x[2 * e] = __low2float(p[e]);
        x[2 * e + 1] = __high2float(p[e]);
    }
}

template <int NP>
__global__ void __launch_bounds__(kThreadsD, 2)
    verify_tc_fdiag_kernel(const __grid_constant__ CUtensorMap tm_q,
                           const __grid_constant__ CUtensorMap tm_k,
                           const __grid_constant__ CUtensorMap tm_v,
                           const __grid_constant__ CUtensorMap tm_g, const DiagParams P) {
    constexpr uint32_t kTile = NP * 128;        // one factor tile: NP rows of 128 B
    constexpr uint32_t kBlock = 4 * kTile;      // one group's factor block
    constexpr uint32_t kSboW = (NP / 8) * 128;  // weight tiles: 8-row group step
    constexpr int kTpn = NP >= 64 ? 4 : 8;      // factor threads per node
    constexpr int kPpt = 8 / kTpn;              // 8-channel pieces per factor thread
    const VerifyArgs &a = P.a;
    extern __shared__ uint8_t smem_raw[];
    uint8_t *smem = reinterpret_cast<uint8_t *>(
        (reinterpret_cast<uintptr_t>(smem_raw) + 1023) & ~static_cast<uintptr_t>(1023));
    const int dk = a.dk, H = a.H, ng = dk / kGrpCh, nch = ng * kChunksPerGrp;
    const DiagLayout L(NP, ng);
    uint8_t *sF = smem + L.f_off;
    uint8_t *sH = smem + L.h_off;
    uint64_t *sAnc = reinterpret_cast<uint64_t *>(smem + L.anc_off);
    int *sPar = reinterpret_cast<int *>(smem + L.par_off);
    int *sJmp = reinterpret_cast<int *>(smem + L.jmp_off);
    int *meta = reinterpret_cast<int *>(smem + L.meta_off);
    uint32_t *sTmem = reinterpret_cast<uint32_t *>(smem + L.misc_off);
    int *sLate = reinterpret_cast<int *>(smem + L.misc_off + 4);     // a wait gave up
    int *sIssued = reinterpret_cast<int *>(smem + L.misc_off + 16);  // last chunk per slot
    // Every barrier but the ring's completes one phase per launch, so no waiter can miss
    // a phase however far a producer runs ahead; the ring slots' single waiter issues
    // each refill itself.
    const uint32_t bar0 = ptx::smem_addr(smem + L.bar_off);
    auto b_slot = [&](int s) { return bar0 + 8u * s; };                   // a chunk landed
    auto b_conv = [&](int q) { return bar0 + 8u * (kRing + q); };         // its parts stored
    auto b_fin = [&](int kg) { return bar0 + 8u * (11 + kg); };           // factor columns
    auto b_facq = [&](int kg) { return bar0 + 8u * (13 + kg); };          // q~ written
    auto b_fac = [&](int kg) { return bar0 + 8u * (15 + kg); };           // k~ written
    const uint32_t b_v = bar0 + 8u * 17, b_tree = bar0 + 8u * 18, b_sfull = bar0 + 8u * 19,
                   b_wready = bar0 + 8u * 20, b_dfull = bar0 + 8u * 21;
    const uint32_t fA = ptx::smem_addr(sF);
    const uint32_t hA = ptx::smem_addr(sH);
    const uint32_t vA = ptx::smem_addr(smem + L.v_off);
    auto late_now = [&]() { return *reinterpret_cast<volatile int *>(sLate) != 0; };

    const int tid = threadIdx.x, warp = tid >> 5, lane = tid & 31;
    const int unit = blockIdx.x, b = unit / H, h = unit % H;
    const float *h0 = a.H0 + (size_t)unit * dk * kDvD;  // chunk q: key rows 16q .. 16q + 15

    // ---- prologue that touches no input: barriers, tensor memory
    if (tid == 0) {
        ptx::prefetch_tensormap(&tm_q);
        ptx::prefetch_tensormap(&tm_k);
        ptx::prefetch_tensormap(&tm_v);
        ptx::prefetch_tensormap(&tm_g);
        for (int s = 0; s < kRing; ++s) ptx::mbar_init(b_slot(s), 1);
        for (int q = 0; q < kMaxChunksD; ++q) ptx::mbar_init(b_conv(q), kConvWarps);
        for (int kg = 0; kg < kMaxGroups; ++kg) {
            ptx::mbar_init(b_fin(kg), 1);
            ptx::mbar_init(b_facq(kg), kFacWarps);
            ptx::mbar_init(b_fac(kg), kFacWarps);
        }
        ptx::mbar_init(b_v, 1);
        ptx::mbar_init(b_tree, 1);
        ptx::mbar_init(b_sfull, 1);
        ptx::mbar_init(b_wready, kFacWarps);
        ptx::mbar_init(b_dfull, 1);
        ptx::fence_mbar_init();
        *sLate = 0;
        for (int s = 0; s < kRing; ++s) sIssued[s] = s;
    }
    if (warp == kCtlWarp) {
        ptx::tmem_alloc(ptx::smem_addr(sTmem), P.tmem_cols);
        ptx::tmem_relinquish();
    }
    ptx::tc_fence_before_sync();
    __syncthreads();
    ptx::tc_fence_after_sync();
    const uint32_t tmem = *sTmem;
    const uint32_t tD = tmem;       // H0^T Q~^T + V^T W^T: lane = value channel, column = node
    const uint32_t tS = tmem + NP;  // Q~ K~^T: lane = node, column = ancestor
    // the state's hi / lo parts: lane = value channel, 16 columns per chunk (8 hi, 8 lo)
    const uint32_t tA = tmem + 2 * NP;

    ptx::grid_dependency_wait();  // inputs may be written by the previous kernel

    if (warp == kCtlWarp) {
        // ================= copies, tree, products
        if (lane == 0)
            for (int s = 0; s < kRing && s < nch; ++s) {  // the first chunks need no offsets
                ptx::mbar_arrive_expect_tx(b_slot(s), kChunkBytesD);
                ptx::bulk_g2s(hA + s * kChunkBytesD, h0 + (size_t)s * kChunkValsD, kChunkBytesD,
                              b_slot(s));
            }
        ptx::grid_launch_dependents();
        int off = 0, n = 0;
        const bool range_ok = request_range(a.node_offsets, b, a.T, a.max_nodes, off, n);
        if (!range_ok) n = 0;
        const int npad = (n + 15) & ~15;
        if (lane == 0) {
            // every group's q, k and g columns, and v
            for (int kg = 0; kg < ng; ++kg) {
                if (n == 0) {
                    ptx::mbar_arrive(b_fin(kg));
                    continue;
                }
                const uint32_t fb = fA + kg * kBlock;
                ptx::mbar_arrive_expect_tx(b_fin(kg), npad * (kGrpCh * 4 + 2 * 128));
                for (int r = 0; r < npad; r += 16) {
                    ptx::tma_load_3d(fb + r * 128, &tm_q, kg * kGrpCh, h, off + r, b_fin(kg));
                    ptx::tma_load_3d(fb + 2 * kTile + r * 128, &tm_k, kg * kGrpCh, h, off + r,
                                     b_fin(kg));
#pragma unroll
                    for (int sl = 0; sl < 2; ++sl)  // g: two 128-byte-swizzled slabs of 32 channels
                        ptx::tma_load_3d(fb + (1 + 2 * sl) * kTile + r * 128, &tm_g,
                                         kg * kGrpCh + 32 * sl, h, off + r, b_fin(kg));
                }
            }
            if (n == 0) {
                ptx::mbar_arrive(b_v);
            } else {
                ptx::mbar_arrive_expect_tx(b_v, npad * 2 * 128);
                for (int r = 0; r < npad; r += 16)
#pragma unroll
                    for (int mb = 0; mb < 2; ++mb)
                        ptx::tma_load_3d(vA + mb * kTile + r * 128, &tm_v, mb * 64, h, off + r, b_v);
            }
        }

        // tree rows (nodes lane and lane + 32), checks, ancestor masks
        int par[2], dep[2];
        bool bad = false;
#pragma unroll
        for (int s = 0; s < 2; ++s) {
            const int i = lane + 32 * s;
            par[s] = -1;
            dep[s] = 0;
            if (i < n) {
                par[s] = a.parent[off + i];
                dep[s] = a.depth[off + i];
                bad = bad || par[s] < -1 || par[s] >= i;
                sPar[i] = par[s];
                sJmp[i] = dep[s];  // depths first, for the parent lookups below
            }
        }
        __syncwarp();
#pragma unroll
        for (int s = 0; s < 2; ++s) {
            const int i = lane + 32 * s;
            if (i < n && par[s] >= -1 && par[s] < i) {
                const int want = par[s] < 0 ? 1 : sJmp[par[s]] + 1;
                bad = bad || dep[s] != want || dep[s] > a.max_depth;
            }
        }
        const bool tree_bad = __any_sync(0xffffffffu, bad);
        const bool run = n > 0 && !tree_bad;
        uint64_t anc[2];
        int jmp[2];
#pragma unroll
        for (int s = 0; s < 2; ++s) {
            const int i = lane + 32 * s;
            anc[s] = i < n ? (1ull << i) : 0ull;
            jmp[s] = (i < n && run) ? par[s] : -1;
        }
        __syncwarp();
#pragma unroll
        for (int s = 0; s < 2; ++s) {
            const int i = lane + 32 * s;
            if (i < NP) {
                sAnc[i] = anc[s];
                sJmp[i] = jmp[s];
            }
        }
        __syncwarp();
        // pointer doubling: after round r a node's mask covers 2^{r+1} nodes of its path
        for (int r = 0; r < 6 && __any_sync(0xffffffffu, jmp[0] >= 0 || jmp[1] >= 0); ++r) {
            uint64_t na[2];
            int nj[2];
#pragma unroll
            for (int s = 0; s < 2; ++s) {
                na[s] = anc[s];
                nj[s] = jmp[s];
                if (jmp[s] >= 0) {
                    na[s] |= sAnc[jmp[s]];
                    nj[s] = sJmp[jmp[s]];
                }
            }
            __syncwarp();
#pragma unroll
            for (int s = 0; s < 2; ++s) {
                const int i = lane + 32 * s;
                anc[s] = na[s];
                jmp[s] = nj[s];
                if (i < NP) {
                    sAnc[i] = anc[s];
                    sJmp[i] = jmp[s];
                }
            }
            __syncwarp();
        }
        if (lane == 0) {
            if (!range_ok && h == 0) report(a.status, TV_ERR_TREE);
            if (n > 0 && tree_bad && h == 0) report(a.status, TV_ERR_TREE);
            meta[kMN] = n;
            meta[kMOff] = off;
            meta[kMRun] = run ? 1 : 0;
            meta[kMZero] = (n > 0 && tree_bad) ? 1 : 0;
            meta[kMWalk] = 0;
            meta[kMHave] = 0;
        }
        __syncwarp();
        if (lane == 0) ptx::mbar_arrive(b_tree);

        if (lane == 0) {
            // ---- products (one thread).  A role that gave up (its bit in sLate) released
            // its barriers unwritten: nothing more is issued then.
            bool ok = run;
            const uint32_t idn = (ptx::idesc_bf16_f32(128, 16) & ~(0x3Fu << 17)) |
                                 (static_cast<uint32_t>(npad >> 3) << 17);
            const uint32_t idm = idn | (1u << 15);  // A MN-major
            auto wait_ok = [&](uint32_t bar) {
                if (!ptx::mbar_wait(bar, 0, kWaitLimit)) atomicOr(sLate, 16);
                return !late_now();
            };
            for (int kg = 0; kg < ng && ok; ++kg) {
                const uint32_t fb = fA + kg * kBlock;
                const uint32_t qh = fb, ql = fb + kTile, kh = fb + 2 * kTile, kl = fb + 3 * kTile;
                if (!wait_ok(b_facq(kg))) {
                    ok = false;
                    break;
                }
                // D += H0^T Q~^T, one 16-row chunk (16 key channels) at a time: A = the state
                // parts in tensor memory, passes hi.hi, hi.lo, lo.hi
                for (int ch = 0; ch < kChunksPerGrp; ++ch) {
                    const int q = kg * kChunksPerGrp + ch;
                    if (!wait_ok(b_conv(q))) {
                        ok = false;
                        break;
                    }
                    ptx::tc_fence_after_sync();
                    const uint32_t ta = tA + q * 16u, o = ch * 32;
                    ptx::mma_bf16_ts(tD, ta, ptx::desc_kmajor_sw128(qh + o, 1024), idn,
                                     q > 0 ? 1u : 0u);
                    ptx::mma_bf16_ts(tD, ta, ptx::desc_kmajor_sw128(ql + o, 1024), idn, 1u);
                    ptx::mma_bf16_ts(tD, ta + 8u, ptx::desc_kmajor_sw128(qh + o, 1024), idn, 1u);
                }
                if (!ok) break;
                if (!wait_ok(b_fac(kg))) {
                    ok = false;
                    break;
                }
                ptx::tc_fence_after_sync();
                // S += Q~ K~^T over the group's 64 channels, passes hi.hi, lo.hi, hi.lo
#pragma unroll
                for (int ks = 0; ks < 4; ++ks) {
                    const uint32_t o = ks * 32;
                    ptx::mma_bf16(tS, ptx::desc_kmajor_sw128(qh + o, 1024),
                                  ptx::desc_kmajor_sw128(kh + o, 1024), idn,
                                  (kg > 0 || ks > 0) ? 1u : 0u);
                    ptx::mma_bf16(tS, ptx::desc_kmajor_sw128(ql + o, 1024),
                                  ptx::desc_kmajor_sw128(kh + o, 1024), idn, 1u);
                    ptx::mma_bf16(tS, ptx::desc_kmajor_sw128(qh + o, 1024),
                                  ptx::desc_kmajor_sw128(kl + o, 1024), idn, 1u);
                }
            }
            ptx::mma_commit(b_sfull);  // every product issued so far, or none
            if (ok && !wait_ok(b_wready)) ok = false;
            if (ok) {
                ptx::tc_fence_after_sync();
                // D += V^T W^T: A = v (both 64-channel blocks), B = W hi, then W lo
                const uint32_t wh = fA, wl = fA + NP * NP * 2;
                for (int ks = 0; ks < npad / 16; ++ks) {
                    const uint64_t ad = ptx::desc_mnmajor_sw128(vA + ks * 2048u, kTile, 1024);
                    ptx::mma_bf16(tD, ad, ptx::desc_kmajor_noswizzle(wh + ks * 256u, 128, kSboW),
                                  idm, 1u);
                    ptx::mma_bf16(tD, ad, ptx::desc_kmajor_noswizzle(wl + ks * 256u, 128, kSboW),
                                  idm, 1u);
                }
            }
            ptx::mma_commit(b_dfull);
            // products in flight complete before the epilogue or the exit reads on
            if (!ptx::mbar_wait(b_dfull, 0, kWaitLimit)) atomicOr(sLate, 64);
            meta[kMHave] = ok ? 1 : 0;
        }
    } else if (warp < kConvWarps) {
        // ================= state chunks -> hi / lo parts in tensor memory
        // thread = value channel c (its lane of the warp's quadrant); per chunk it reads the
        // 16 key rows of its channel (a warp reads 128 contiguous bytes per row), the slot
        // takes the chunk three further on, and the rows are split into bf16 hi / lo pairs
        // along the key rows -- the layout of an A operand in tensor memory -- and stored
        const int c = tid;
        if (tid == 0 && !ptx::mbar_wait(b_tree, 0, kWaitLimit)) atomicOr(sLate, 2);
        named_barrier(1, kConvWarps * 32);
        const bool go = !(*sLate & 2) && meta[kMRun] != 0;
        int q = 0;
        for (; q < nch && go; ++q) {
            const int slot = q % kRing;
            if (tid == 0) {
                // stop when another role gave up, or when this chunk does not land
                const bool ok = !late_now() &&
                                ((q == 0 && P.expire_first_wait)
                                     ? false  // test hook: treated as expired
                                     : ptx::mbar_wait(b_slot(slot), (q / kRing) & 1, kWaitLimit));
                if (!ok) atomicOr(sLate, 2);
            }
            named_barrier(1, kConvWarps * 32);
            if (*sLate & 2) break;  // the chunk did not land: stop converting
            const float *cp = reinterpret_cast<const float *>(sH + slot * kChunkBytesD);
            float x[kChunkRowsD];
#pragma unroll
            for (int r = 0; r < kChunkRowsD; ++r) x[r] = cp[r * kDvD + c];
            if (q + kRing < nch) {
                named_barrier(1, kConvWarps * 32);  // every thread has read the chunk
                if (tid == 0) {
                    ptx::fence_proxy_async_smem();
                    ptx::mbar_arrive_expect_tx(b_slot(slot), kChunkBytesD);
                    ptx::bulk_g2s(hA + slot * kChunkBytesD, h0 + (size_t)(q + kRing) * kChunkValsD,
                                  kChunkBytesD, b_slot(slot));
                    sIssued[slot] = q + kRing;
                }
            }
            uint32_t hi[kChunkRowsD / 2], lo[kChunkRowsD / 2];
#pragma unroll
            for (int m = 0; m < kChunkRowsD / 2; ++m) split_pair(x[2 * m], x[2 * m + 1], hi[m], lo[m]);
            const uint32_t ta = tA + q * 16u + (static_cast<uint32_t>(32 * warp) << 16);
            ptx::tmem_st_x8(ta, hi);
            ptx::tmem_st_x8(ta + 8u, lo);
            ptx::tmem_wait_st();
            ptx::tc_fence_before_sync();
            __syncwarp();
            if (lane == 0) ptx::mbar_arrive(b_conv(q));
        }
        // after a failed wait the remaining chunks are released unconverted (the outputs
        // are not written then)
        __syncwarp();
        if (lane == 0 && go)
            for (; q < nch; ++q) ptx::mbar_arrive(b_conv(q));
    } else {
        // ================= factors, weights (warps kConvWarps .. kCtlWarp - 1)
        const int t = tid - kConvWarps * 32, fw = warp - kConvWarps;
        constexpr int kFT = kFacWarps * 32;
        if (t == 0 && !ptx::mbar_wait(b_tree, 0, kWaitLimit)) atomicOr(sLate, 4);
        named_barrier(2, kFT);
        bool go = !(*sLate & 4) && meta[kMRun] != 0;
        const int n = meta[kMN], off = meta[kMOff];
        // node i = t / kTpn takes pieces kPpt * sub .. of a group's 64 channels
        const int i = t / kTpn, sub = t % kTpn;
        const bool mine = i < n;
        float gmax = 0.f;  // largest |G| seen: the factor range check
        for (int kg = 0; kg < ng && go; ++kg) {
            uint8_t *fb = sF + kg * kBlock;
            if (t == 0 && !(!late_now() && ptx::mbar_wait(b_fin(kg), 0, kWaitLimit)))
                atomicOr(sLate, 4);  // another role gave up, or the columns did not land
            named_barrier(2, kFT);
            if (*sLate & 4) {
                if (lane == 0) {  // release the product thread
                    ptx::mbar_arrive(b_facq(kg));
                    ptx::mbar_arrive(b_fac(kg));
                }
                go = false;
                break;
            }
            // path sums of g over this thread's channels: per ancestor, in index order
            // (depth order on a root path), 2 * kPpt independent 16-byte loads.  The g
            // slabs are 128-byte swizzled, so the rows of different ancestors spread over
            // the banks.
            float G[kPpt * 8];
#pragma unroll
            for (int e = 0; e < kPpt * 8; ++e) G[e] = 0.f;
            if (mine) {
                uint64_t m = sAnc[i];
                while (m) {
                    const int j = __ffsll(static_cast<long long>(m)) - 1;
                    m &= m - 1;
#pragma unroll
                    for (int x = 0; x < 2 * kPpt; ++x) {
                        const int cx = 2 * kPpt * sub + x;  // 4-channel chunk of the 64
                        const float4 gv = *reinterpret_cast<const float4 *>(
                            fb + (1 + 2 * (cx >> 3)) * kTile + j * 128 + (((cx & 7) ^ (j & 7)) << 4));
                        G[4 * x] += gv.x; G[4 * x + 1] += gv.y;
                        G[4 * x + 2] += gv.z; G[4 * x + 3] += gv.w;
                    }
                }
#pragma unroll
                for (int e = 0; e < kPpt * 8; ++e) {
                    gmax = fmaxf(gmax, fabsf(G[e]));
                    G[e] *= kLog2eD;  // exponents in base 2 from here on
                }
            }
            named_barrier(2, kFT);  // every path sum is read before the g slabs are rewritten
            // q~ = e^{G} q first (the context products need only q~), then k~ = e^{-G} k;
            // hi parts over q and k, lo parts over the g slabs
#pragma unroll
            for (int side = 0; side < 2; ++side) {
#pragma unroll
                for (int y = 0; y < kPpt; ++y) {
                    const int p = kPpt * sub + y;  // 8-channel piece
                    const uint32_t sw = static_cast<uint32_t>(i * 128 + ((p ^ (i & 7)) << 4));
                    uint32_t hi[4] = {0u, 0u, 0u, 0u}, lo[4] = {0u, 0u, 0u, 0u};
                    if (mine) {
                        float xv[8];
                        bf16x8(*reinterpret_cast<const uint4 *>(fb + 2 * side * kTile + sw), xv);
#pragma unroll
                        for (int e = 0; e < 8; e += 2) {
                            const float e0 = ex2f(side ? -G[8 * y + e] : G[8 * y + e]);
                            const float e1 = ex2f(side ? -G[8 * y + e + 1] : G[8 * y + e + 1]);
                            split_pair(xv[e] * e0, xv[e + 1] * e1, hi[e / 2], lo[e / 2]);
                        }
                    }
                    if (i < NP) {
                        *reinterpret_cast<uint4 *>(fb + 2 * side * kTile + sw) =
                            make_uint4(hi[0], hi[1], hi[2], hi[3]);
                        *reinterpret_cast<uint4 *>(fb + (2 * side + 1) * kTile + sw) =
                            make_uint4(lo[0], lo[1], lo[2], lo[3]);
                    }
                }
                ptx::fence_proxy_async_smem();
                __syncwarp();
                if (lane == 0) ptx::mbar_arrive(side == 0 ? b_facq(kg) : b_fac(kg));
            }
        }
        if (!(gmax <= kGLimit)) atomicOr(&meta[kMWalk], 1);

        // ---- weights, once every product of the groups is done
        if (t == 0 && !(!late_now() && ptx::mbar_wait(b_sfull, 0, kWaitLimit)))
            atomicOr(sLate, 4);
        named_barrier(2, kFT);
        go = go && !(*sLate & 4);
        const bool walk = go && meta[kMWalk] != 0;
        // fp32 weights of the walk after the weight tiles; the factor blocks are free now
        float *W32 = reinterpret_cast<float *>(sF + 2 * NP * NP * 2);
        if (walk) {
            // out-of-range path sums: w_ij by a walk from i to the context, the pair
            // decay e^{G_i - G_j} a running product of e^{g} (global rows, through L2)
            for (int e = t; e < NP * NP; e += kFT) W32[e] = 0.f;
            named_barrier(2, kFT);
            const __nv_bfloat16 *qg = static_cast<const __nv_bfloat16 *>(a.q);
            const __nv_bfloat16 *kgl = static_cast<const __nv_bfloat16 *>(a.k);
            const int lch = dk / 32;
            for (int wi = fw; wi < n; wi += kFacWarps) {
                const size_t ri = ((size_t)(off + wi) * H + h) * dk;
                float qv[4], f[4];
#pragma unroll
                for (int m = 0; m < 4; ++m) {
                    qv[m] = m < lch ? __bfloat162float(qg[ri + lane + 32 * m]) : 0.f;
                    f[m] = 1.f;
                }
                int j = wi;  // the checked tree's parents precede their children
                while (j >= 0) {
                    const size_t rj = ((size_t)(off + j) * H + h) * dk;
                    float part = 0.f;
#pragma unroll
                    for (int m = 0; m < 4; ++m)
                        if (m < lch) part += qv[m] * __bfloat162float(kgl[rj + lane + 32 * m]) * f[m];
                    part = warp_sum(part);
                    if (lane == 0) W32[wi * NP + j] = part;
#pragma unroll
                    for (int m = 0; m < 4; ++m)
                        if (m < lch) f[m] *= expf(a.g[rj + lane + 32 * m]);
                    j = sPar[j];
                }
            }
            named_barrier(2, kFT);
        }
        const int qd = warp & 3;  // tensor-memory lane quadrant of this warp
        if (go && qd >= 2) {
            // rows npad > j >= n of v (another request's, or zero past the end) meet zero
            // weights; clear them so that no non-finite value gets in
            const int vz = (fw >> 2) * 2 + (qd - 2);  // 0..3 over the four such warps
            bool vok = true;
            if (lane == 0) vok = ptx::mbar_wait(b_v, 0, kWaitLimit);
            vok = __shfl_sync(0xffffffffu, vok ? 1 : 0, 0) != 0;
            if (!vok) {
                if (lane == 0) atomicOr(sLate, 8);
            } else {
                const int npad = (n + 15) & ~15;
                for (int e = vz * 32 + lane; e < (npad - n) * 16; e += 128) {
                    const int jr = n + e / 16, mb = (e / 8) % 2, piece = e % 8;
                    *reinterpret_cast<uint4 *>(smem + L.v_off + mb * kTile + jr * 128 + piece * 16) =
                        make_uint4(0u, 0u, 0u, 0u);
                }
            }
        }
        if (go && qd < 2 && 32 * qd < NP) {
            // weight tiles: row i = node (thread), columns = ancestors, K-major without
            // swizzle (8-row x 16-byte core matrices), hi at the start of the first factor
            // block, lo after it; the two warps of a lane quadrant take half the columns each
            constexpr int CW = NP / 2;
            const int wr = 32 * qd + lane, cb = (fw >> 2) * CW;
            const uint64_t m = wr < NP ? sAnc[wr] : 0ull;
            uint32_t sr[CW];
            if (!walk) {
                ptx::tc_fence_after_sync();
                tmem_ld_n<CW>(tS + (static_cast<uint32_t>(32 * qd) << 16) + cb, sr);
                ptx::tmem_wait_ld();
            } else {
#pragma unroll
                for (int jj = 0; jj < CW; ++jj)
                    sr[jj] = wr < NP ? __float_as_uint(W32[wr * NP + cb + jj]) : 0u;
            }
            uint32_t whi[CW / 2], wlo[CW / 2];
#pragma unroll
            for (int jj = 0; jj < CW; jj += 2) {
                const float wa = ((m >> (cb + jj)) & 1ull) ? __uint_as_float(sr[jj]) : 0.f;
                const float wb = ((m >> (cb + jj + 1)) & 1ull) ? __uint_as_float(sr[jj + 1]) : 0.f;
                split_pair(wa, wb, whi[jj / 2], wlo[jj / 2]);
            }
            if (wr < NP) {
                uint8_t *wh = sF + (wr / 8) * kSboW + (wr % 8) * 16 + (cb / 8) * 128;
                uint8_t *wl = wh + NP * NP * 2;
#pragma unroll
                for (int cc = 0; cc < CW / 8; ++cc) {
                    *reinterpret_cast<uint4 *>(wh + cc * 128) =
                        make_uint4(whi[4 * cc], whi[4 * cc + 1], whi[4 * cc + 2], whi[4 * cc + 3]);
                    *reinterpret_cast<uint4 *>(wl + cc * 128) =
                        make_uint4(wlo[4 * cc], wlo[4 * cc + 1], wlo[4 * cc + 2], wlo[4 * cc + 3]);
                }
            }
        }
        ptx::fence_proxy_async_smem();
        ptx::tc_fence_before_sync();
        __syncwarp();
        if (lane == 0) ptx::mbar_arrive(b_wready);
    }

    // ================= join, then the epilogue (warps 0-7)
    ptx::tc_fence_before_sync();
    __syncthreads();
    ptx::tc_fence_after_sync();
    const int late = *sLate;
    const int n = meta[kMN], off = meta[kMOff];
    const bool ok = meta[kMRun] != 0 && meta[kMHave] != 0 && late == 0;
    if (tid == 0 && late) report(a.status, TV_ERR_TIMEOUT);
    if (meta[kMZero])
        for (int e = tid; e < n * kDvD; e += kThreadsD)
            a.out[((size_t)(off + e / kDvD) * H + h) * kDvD + e % kDvD] = 0.f;
    if (ok && warp < 8) {
        // warp w: lane quadrant w % 4 (value channels), node half w / 4
        constexpr int HALF = NP / 2;
        const int qd = warp & 3, hf = warp >> 2;
        uint32_t dv[HALF];
        tmem_ld_n<HALF>(tD + (static_cast<uint32_t>(32 * qd) << 16) + hf * HALF, dv);
        ptx::tmem_wait_ld();
        float *o = a.out + ((size_t)(off + hf * HALF) * H + h) * kDvD + 32 * qd + lane;
#pragma unroll
        for (int i = 0; i < HALF; ++i)
            if (hf * HALF + i < n) o[(size_t)i * H * kDvD] = __uint_as_float(dv[i]);
    }
    if (warp == kCtlWarp && lane == 0) {
        // every copy issued lands before the CTA's memory can go away
        bool drained = true;
        for (int s = 0; s < kRing && s < nch; ++s)
            drained = ptx::mbar_wait(b_slot(s), (sIssued[s] / kRing) & 1, kWaitLimit) && drained;
        for (int kg = 0; kg < ng; ++kg) drained = ptx::mbar_wait(b_fin(kg), 0, kWaitLimit) && drained;
        drained = ptx::mbar_wait(b_v, 0, kWaitLimit) && drained;
        if (!drained) report(a.status, TV_ERR_TIMEOUT);
    }
    ptx::tc_fence_before_sync();
    __syncthreads();
    if (warp == kCtlWarp) ptx::tmem_dealloc(tmem, P.tmem_cols);
}

// ---------------------------------------------------------------- host side

int fdiag_np(const VerifyArgs &a) { return a.max_nodes <= 16 ? 16 : a.max_nodes <= 32 ? 32 : 64; }

template <int NP>
cudaError_t launch_fdiag_t(const VerifyArgs &a, bool expire, cudaStream_t s) {
    const auto BF = CU_TENSOR_MAP_DATA_TYPE_BFLOAT16;
    CUtensorMap tq, tk, tv_, tg;
    // q, k: 64-channel K-major operand boxes; v: MN-major blocks of 64 channels; g: 32
    // fp32 channels per box, 128-byte swizzled
    if (!(encode_rows(&tq, a.q, BF, 2, a.dk, a.H, a.T, 64, CU_TENSOR_MAP_SWIZZLE_128B) &&
          encode_rows(&tk, a.k, BF, 2, a.dk, a.H, a.T, 64, CU_TENSOR_MAP_SWIZZLE_128B) &&
          encode_rows(&tv_, a.v, BF, 2, kDvD, a.H, a.T, 64, CU_TENSOR_MAP_SWIZZLE_128B) &&
          encode_rows(&tg, a.g, CU_TENSOR_MAP_DATA_TYPE_FLOAT32, 4, a.dk, a.H, a.T, 32,
                      CU_TENSOR_MAP_SWIZZLE_128B)))
        return cudaErrorInvalidValue;
    DiagParams P;
    P.a = a;
    P.tmem_cols = tmem_columns(2 * NP + 64 * (a.dk / kGrpCh));
    P.expire_first_wait = expire ? 1 : 0;
    auto kern = verify_tc_fdiag_kernel<NP>;
    cudaError_t e = configure_smem_once(kern, true);
    if (e != cudaSuccess) return e;
    const size_t smem = DiagLayout(NP, a.dk / kGrpCh).total;
    return launch_pdl(kern, dim3((unsigned)(a.B * a.H)), dim3(kThreadsD), smem, s, tq, tk, tv_, tg,
                      P);
}

}  // namespace

bool verify_tc_fdiag_supported(const VerifyArgs &a) {
    return a.decay == TV_DECAY_DIAG && a.qkv_dtype == TV_BF16 && (a.dk == 64 || a.dk == 128) &&
           a.dv == kDvD && a.max_nodes >= 1 && a.max_nodes <= 64 && encode_fn() != nullptr &&
           DiagLayout(fdiag_np(a), a.dk / kGrpCh).total <= kSmemLimit;
}

cudaError_t launch_verify_tc_fdiag(const VerifyArgs &a, cudaStream_t s, bool expire_first_wait) {
    if (!verify_tc_fdiag_supported(a)) return cudaErrorNotSupported;
    switch (fdiag_np(a)) {
        case 16: return launch_fdiag_t<16>(a, expire_first_wait, s);
        case 32: return launch_fdiag_t<32>(a, expire_first_wait, s);
        default: return launch_fdiag_t<64>(a, expire_first_wait, s);
    }
}

}  // namespace tv
