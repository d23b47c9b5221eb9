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
// Memory.  The key channels are taken in groups of 64.  The state streams through a ring
// of three 8 KB chunk slots (16 key rows each): a chunk's rows are split into bf16 hi / lo
// parts in tensor memory -- the A operand of the context product, lane = value channel --
// and its slot takes the chunk three further on at once.  A factor block per group holds
// the group's g, q and k columns (g: 64 fp32 per node, q and k: 64 bf16 per node, all
// 128-byte swizzled), rewritten in place as the q~ / k~ hi and lo tiles.  About 108 KB of
// shared memory and 256 tensor-memory columns at 64 nodes: two CTAs per SM.
//
// Persistent CTAs: one per resident slot, each taking every grid-th (request, head) unit,
// so that a unit's loads overlap the previous unit's tail.  The ring streams across unit
// boundaries (the next unit's first chunks arrive while this unit's last ones are
// converted); the factor blocks but the last take the next unit's columns once this
// unit's context and score products are done, the last block (which meanwhile holds the
// weight tiles) and v once all its products are; the next unit's tree is checked ahead
// into the second copy of the tree arrays.  Barriers other than the ring's come in an
// even and an odd copy, so a unit waits for phase unit / 2 of its copy.
//
// Roles (448 threads):
//   warps 0-3   state chunks: a thread per value channel reads its 16 key rows of a
//               chunk, splits them and stores the parts to its tensor-memory lane; before
//               a unit's chunks, the previous unit's outputs (one channel per thread)
//   warps 4-11  factors: path sums G of the group's channels (4 or 8 threads per node),
//               range check, q~ hi / lo (then the context products may start), k~ hi /
//               lo; after the products, the weight tiles (the four warps on the score
//               rows' lane quadrants, half the columns each), the walk for out-of-range
//               units, and the v rows past the tree cleared
//   warp 12     tensor memory; one thread issues the products
//   warp 13     the ring's first chunks; per unit the tree checks and ancestor masks
//               (pointer doubling in shared memory) and the factor and v copies
// Every wait is bounded (TV_ERR_TIMEOUT); every copy and product in flight is waited
// for (bounded) before tensor memory is freed.  Malformed trees zero their rows and set
// TV_ERR_TREE.
#include "tc_common.cuh"

namespace tv {
namespace {
using namespace tcc;

constexpr int kConvWarps = 4;                           // warps 0-3: state chunks, epilogue
constexpr int kFacWarps = 8;                            // warps 4-11: factors, weights
constexpr int kMmaWarp = kConvWarps + kFacWarps;        // warp 12: products (one thread)
constexpr int kLoadWarp = kMmaWarp + 1;                 // warp 13: trees, factor copies
constexpr int kThreadsD = (kLoadWarp + 1) * 32;         // 448
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

// Barriers.  The ring's three slots stream state chunks across units (one phase per use
// of a slot).  Every other barrier is per unit and comes in two copies, one for even and
// one for odd units, so that a unit's phase is phase (unit >> 1) of its copy: no
// producer can run a whole two units ahead of a waiter, since each unit's products wait
// on the resources the unit before released.
enum {
    kBarSlot = 0,                                   // [kRing]: a chunk landed
    kBarConv = kBarSlot + kRing,                    // [2][kMaxChunksD]: its parts stored
    kBarFin = kBarConv + 2 * kMaxChunksD,           // [2][kMaxGroups]: factor columns landed
    kBarFacq = kBarFin + 2 * kMaxGroups,            // [2][kMaxGroups]: q~ written
    kBarFac = kBarFacq + 2 * kMaxGroups,            // [2][kMaxGroups]: k~ written
    kBarV = kBarFac + 2 * kMaxGroups,               // [2]: v landed
    kBarTree = kBarV + 2,                           // [2]: tree checked, masks ready
    kBarSfull = kBarTree + 2,                       // [2]: context and score products done
    kBarWready = kBarSfull + 2,                     // [2]: weight tiles written
    kBarDfull = kBarWready + 2,                     // [2]: every product done
    kBarDfree = kBarDfull + 2,                      // [2]: the outputs read from D
    kNumBars = kBarDfree + 2
};

enum { kMN = 0, kMOff, kMRun, kMZero, kMWalk, kMetaWords = 16 };

// Shared-memory plan, identical on host and device.  The factor blocks come first, one
// per key-channel group: q | g slab 0 (later q~ lo) | k | g slab 1 (later k~ lo), each
// np rows of 128 B.  Read as M = 128 operands, the q~ hi and lo tiles span 16 KB from
// their starts, inside the plan for every tree size.  After a unit's products the last
// block holds its weight tiles (hi, lo) and, for the walk, the fp32 weights.  Tree
// arrays and metadata come in two copies (even and odd units).
struct DiagLayout {
    uint32_t f_off, h_off, v_off, tree_off, tree_bytes, meta_off, bar_off, misc_off, total;
    __host__ __device__ DiagLayout(int np, int ng) {
        f_off = 0;
        h_off = align_up(f_off + ng * 4 * np * 128, 1024);    // the state chunk ring
        v_off = align_up(h_off + kRing * kChunkBytesD, 1024);  // v, two 64-channel blocks
        tree_off = align_up(v_off + 2 * np * 128, 16);
        tree_bytes = np * (8 + 4 + 4);                         // masks, parents, jumps
        meta_off = tree_off + 2 * tree_bytes;
        bar_off = align_up(meta_off + 2 * kMetaWords * 4, 16);
        misc_off = bar_off + kNumBars * 8;
        total = misc_off + 32 + 1024;  // + slack for 1024-byte base alignment
    }
};

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
    const int units = a.B * H, G = gridDim.x;
    const int nu = (units - (int)blockIdx.x + G - 1) / G;  // units of this CTA
    auto unit_of = [&](int it) { return (int)blockIdx.x + it * G; };
    const DiagLayout L(NP, ng);
    uint8_t *sF = smem + L.f_off;
    uint8_t *sH = smem + L.h_off;
    // per-parity tree arrays and metadata
    auto sAnc = [&](int it) { return reinterpret_cast<uint64_t *>(smem + L.tree_off + (it & 1) * L.tree_bytes); };
    auto sPar = [&](int it) {
        return reinterpret_cast<int *>(smem + L.tree_off + (it & 1) * L.tree_bytes + NP * 8);
    };
    auto sJmp = [&](int it) {
        return reinterpret_cast<int *>(smem + L.tree_off + (it & 1) * L.tree_bytes + NP * 12);
    };
    auto meta = [&](int it) { return reinterpret_cast<int *>(smem + L.meta_off) + (it & 1) * kMetaWords; };
    uint32_t *sTmem = reinterpret_cast<uint32_t *>(smem + L.misc_off);
    int *sLate = reinterpret_cast<int *>(smem + L.misc_off + 4);     // a wait gave up
    int *sIssued = reinterpret_cast<int *>(smem + L.misc_off + 16);  // last chunk per slot
    const uint32_t bar0 = ptx::smem_addr(smem + L.bar_off);
    auto bar = [&](int idx) { return bar0 + 8u * idx; };
    auto b_slot = [&](int s) { return bar(kBarSlot + s); };
    auto b_conv = [&](int it, int q) { return bar(kBarConv + (it & 1) * kMaxChunksD + q); };
    auto b_fin = [&](int it, int kg) { return bar(kBarFin + (it & 1) * kMaxGroups + kg); };
    auto b_facq = [&](int it, int kg) { return bar(kBarFacq + (it & 1) * kMaxGroups + kg); };
    auto b_fac = [&](int it, int kg) { return bar(kBarFac + (it & 1) * kMaxGroups + kg); };
    auto b_v = [&](int it) { return bar(kBarV + (it & 1)); };
    auto b_tree = [&](int it) { return bar(kBarTree + (it & 1)); };
    auto b_sfull = [&](int it) { return bar(kBarSfull + (it & 1)); };
    auto b_wready = [&](int it) { return bar(kBarWready + (it & 1)); };
    auto b_dfull = [&](int it) { return bar(kBarDfull + (it & 1)); };
    auto b_dfree = [&](int it) { return bar(kBarDfree + (it & 1)); };
    auto ph = [](int it) { return static_cast<uint32_t>((it >> 1) & 1); };  // phase parity
    const uint32_t fA = ptx::smem_addr(sF);
    const uint32_t hA = ptx::smem_addr(sH);
    const uint32_t vA = ptx::smem_addr(smem + L.v_off);
    const uint32_t wA = fA + (ng - 1) * kBlock;  // weight tiles: the last factor block
    auto late_now = [&]() { return *reinterpret_cast<volatile int *>(sLate) != 0; };
    auto chunk_src = [&](int gq) {  // global chunk gq = unit index * nch + chunk
        return a.H0 + (size_t)unit_of(gq / nch) * dk * kDvD + (size_t)(gq % nch) * kChunkValsD;
    };

    const int tid = threadIdx.x, warp = tid >> 5, lane = tid & 31;

    // ---- prologue that touches no input: barriers, tensor memory
    if (tid == 0) {
        ptx::prefetch_tensormap(&tm_q);
        ptx::prefetch_tensormap(&tm_k);
        ptx::prefetch_tensormap(&tm_v);
        ptx::prefetch_tensormap(&tm_g);
        for (int s = 0; s < kRing; ++s) ptx::mbar_init(b_slot(s), 1);
        for (int p = 0; p < 2; ++p) {
            for (int q = 0; q < kMaxChunksD; ++q) ptx::mbar_init(b_conv(p, q), kConvWarps);
            for (int kg = 0; kg < kMaxGroups; ++kg) {
                ptx::mbar_init(b_fin(p, kg), 1);
                ptx::mbar_init(b_facq(p, kg), kFacWarps);
                ptx::mbar_init(b_fac(p, kg), kFacWarps);
            }
            ptx::mbar_init(b_v(p), 1);
            ptx::mbar_init(b_tree(p), 1);
            ptx::mbar_init(b_sfull(p), 1);
            ptx::mbar_init(b_wready(p), kFacWarps);
            ptx::mbar_init(b_dfull(p), 1);
            ptx::mbar_init(b_dfree(p), kConvWarps);
        }
        ptx::fence_mbar_init();
        *sLate = 0;
        for (int s = 0; s < kRing; ++s) sIssued[s] = -1;
    }
    if (warp == kMmaWarp) {
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

    if (warp == kLoadWarp) {
        // ================= trees and copies: the ring's first chunks, then per unit the
        // tree checks and masks, and the factor columns and v once their space is free
        if (lane == 0)
            for (int s = 0; s < kRing && s < nu * nch; ++s) {  // the first chunks need no offsets
                ptx::mbar_arrive_expect_tx(b_slot(s), kChunkBytesD);
                ptx::bulk_g2s(hA + s * kChunkBytesD, chunk_src(s), kChunkBytesD, b_slot(s));
                sIssued[s] = s;
            }
        ptx::grid_launch_dependents();
        int last_f = -1;  // the last unit whose factor columns and v were requested
        for (int it = 0; it < nu; ++it) {
            // the tree arrays of this parity were last read by unit it - 2's epilogue
            bool ok = true;
            if (it >= 2 && lane == 0)
                ok = !late_now() && ptx::mbar_wait(b_dfree(it - 2), ph(it - 2), kWaitLimit);
            ok = __shfl_sync(0xffffffffu, ok ? 1 : 0, 0) != 0;
            if (!ok) {
                if (lane == 0) atomicOr(sLate, 32);
                break;
            }
            const int u = unit_of(it), b = u / H, h = u % H;
            int off = 0, n = 0;
            const bool range_ok = request_range(a.node_offsets, b, a.T, a.max_nodes, off, n);
            if (!range_ok) n = 0;
            uint64_t *anc_s = sAnc(it);
            int *par_s = sPar(it), *jmp_s = sJmp(it), *mt = meta(it);
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
                    par_s[i] = par[s];
                    jmp_s[i] = dep[s];  // depths first, for the parent lookups below
                }
            }
            __syncwarp();
#pragma unroll
            for (int s = 0; s < 2; ++s) {
                const int i = lane + 32 * s;
                if (i < n && par[s] >= -1 && par[s] < i) {
                    const int want = par[s] < 0 ? 1 : jmp_s[par[s]] + 1;
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
                    anc_s[i] = anc[s];
                    jmp_s[i] = jmp[s];
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
                        na[s] |= anc_s[jmp[s]];
                        nj[s] = jmp_s[jmp[s]];
                    }
                }
                __syncwarp();
#pragma unroll
                for (int s = 0; s < 2; ++s) {
                    const int i = lane + 32 * s;
                    anc[s] = na[s];
                    jmp[s] = nj[s];
                    if (i < NP) {
                        anc_s[i] = anc[s];
                        jmp_s[i] = jmp[s];
                    }
                }
                __syncwarp();
            }
            if (lane == 0) {
                if (!range_ok && h == 0) report(a.status, TV_ERR_TREE);
                if (n > 0 && tree_bad && h == 0) report(a.status, TV_ERR_TREE);
                mt[kMN] = n;
                mt[kMOff] = off;
                mt[kMRun] = run ? 1 : 0;
                mt[kMZero] = (n > 0 && tree_bad) ? 1 : 0;
                mt[kMWalk] = 0;
            }
            __syncwarp();
            if (lane == 0) ptx::mbar_arrive(b_tree(it));

            if (lane == 0) {
                // factor columns: the blocks but the last once unit it - 1's context and
                // score products are done, the last (which held its weight tiles) and v
                // once all its products are
                const int npad = (n + 15) & ~15;
                auto issue_block = [&](int kg) {
                    if (n == 0) {
                        ptx::mbar_arrive(b_fin(it, kg));
                        return;
                    }
                    const uint32_t fb = fA + kg * kBlock;
                    ptx::mbar_arrive_expect_tx(b_fin(it, kg), npad * (kGrpCh * 4 + 2 * 128));
                    for (int r = 0; r < npad; r += 16) {
                        ptx::tma_load_3d(fb + r * 128, &tm_q, kg * kGrpCh, h, off + r, b_fin(it, kg));
                        ptx::tma_load_3d(fb + 2 * kTile + r * 128, &tm_k, kg * kGrpCh, h, off + r,
                                         b_fin(it, kg));
#pragma unroll
                        for (int sl = 0; sl < 2; ++sl)  // g: two 128-byte-swizzled slabs
                            ptx::tma_load_3d(fb + (1 + 2 * sl) * kTile + r * 128, &tm_g,
                                             kg * kGrpCh + 32 * sl, h, off + r, b_fin(it, kg));
                    }
                };
                // (the previous unit's own copies into a block have landed too, even where
                // no role waited for them: a unit with a malformed tree)
                bool lok = true;
                if (it >= 1)
                    lok = !late_now() && ptx::mbar_wait(b_sfull(it - 1), ph(it - 1), kWaitLimit);
                for (int kg = 0; kg + 1 < ng && lok; ++kg) {
                    if (it >= 1) lok = ptx::mbar_wait(b_fin(it - 1, kg), ph(it - 1), kWaitLimit);
                    if (lok) issue_block(kg);
                }
                if (lok && it >= 1)
                    lok = !late_now() && ptx::mbar_wait(b_dfull(it - 1), ph(it - 1), kWaitLimit) &&
                          ptx::mbar_wait(b_fin(it - 1, ng - 1), ph(it - 1), kWaitLimit) &&
                          ptx::mbar_wait(b_v(it - 1), ph(it - 1), kWaitLimit);
                if (lok) {
                    issue_block(ng - 1);
                    if (n == 0) {
                        ptx::mbar_arrive(b_v(it));
                    } else {
                        ptx::mbar_arrive_expect_tx(b_v(it), npad * 2 * 128);
                        for (int r = 0; r < npad; r += 16)
#pragma unroll
                            for (int mb = 0; mb < 2; ++mb)
                                ptx::tma_load_3d(vA + mb * kTile + r * 128, &tm_v, mb * 64, h, off + r,
                                                 b_v(it));
                    }
                    last_f = it;
                } else {
                    atomicOr(sLate, 32);
                }
            }
            if (__shfl_sync(0xffffffffu, last_f, 0) != it) break;
        }
        if (lane == 0 && last_f >= 0) {
            // every factor and v copy requested lands before the CTA's memory can go away
            // (a unit's blocks but the last were requested together with its last block)
            bool drained = true;
            for (int kg = 0; kg < ng; ++kg)
                drained = ptx::mbar_wait(b_fin(last_f, kg), ph(last_f), kWaitLimit) && drained;
            drained = ptx::mbar_wait(b_v(last_f), ph(last_f), kWaitLimit) && drained;
            if (!drained) atomicOr(sLate, 128);
        }
    } else if (warp == kMmaWarp) {
        if (lane == 0) {
            // ================= products (one thread).  A role that gave up (its bit in
            // sLate) released its barriers unwritten: nothing more is issued then.
            auto wait_ok = [&](uint32_t b, uint32_t parity) {
                if (late_now()) return false;
                if (!ptx::mbar_wait(b, parity, kWaitLimit)) atomicOr(sLate, 16);
                return !late_now();
            };
            for (int it = 0; it < nu; ++it) {
                if (!wait_ok(b_tree(it), ph(it))) break;
                int *mt = meta(it);
                const int n = mt[kMN];
                const int npad = (n + 15) & ~15;
                bool ok = mt[kMRun] != 0;
                const uint32_t idn = (ptx::idesc_bf16_f32(128, 16) & ~(0x3Fu << 17)) |
                                     (static_cast<uint32_t>(npad >> 3) << 17);
                const uint32_t idm = idn | (1u << 15);  // A MN-major
                // D is free once unit it - 1's outputs were read
                if (ok && it >= 1 && !wait_ok(b_dfree(it - 1), ph(it - 1))) ok = false;
                for (int kg = 0; kg < ng && ok; ++kg) {
                    const uint32_t fb = fA + kg * kBlock;
                    const uint32_t qh = fb, ql = fb + kTile, kh = fb + 2 * kTile, kl = fb + 3 * kTile;
                    if (!wait_ok(b_facq(it, kg), ph(it))) {
                        ok = false;
                        break;
                    }
                    // D += H0^T Q~^T, one 16-row chunk (16 key channels) at a time: A = the
                    // state parts in tensor memory, passes hi.hi, hi.lo, lo.hi
                    for (int ch = 0; ch < kChunksPerGrp; ++ch) {
                        const int q = kg * kChunksPerGrp + ch;
                        if (!wait_ok(b_conv(it, q), ph(it))) {
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
                    if (!wait_ok(b_fac(it, kg), ph(it))) {
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
                ptx::mma_commit(b_sfull(it));  // every product issued so far, or none
                if (ok && !wait_ok(b_wready(it), ph(it))) ok = false;
                if (ok) {
                    ptx::tc_fence_after_sync();
                    // D += V^T W^T: A = v (both 64-channel blocks), B = W hi, then W lo
                    const uint32_t wh = wA, wl = wA + NP * NP * 2;
                    for (int ks = 0; ks < npad / 16; ++ks) {
                        const uint64_t ad = ptx::desc_mnmajor_sw128(vA + ks * 2048u, kTile, 1024);
                        ptx::mma_bf16(tD, ad, ptx::desc_kmajor_noswizzle(wh + ks * 256u, 128, kSboW),
                                      idm, 1u);
                        ptx::mma_bf16(tD, ad, ptx::desc_kmajor_noswizzle(wl + ks * 256u, 128, kSboW),
                                      idm, 1u);
                    }
                }
                ptx::mma_commit(b_dfull(it));
                // the products complete before this unit's outputs are read or the next
                // unit's columns overwrite the operands
                if (!ptx::mbar_wait(b_dfull(it), ph(it), kWaitLimit)) atomicOr(sLate, 64);
                if (late_now()) break;
            }
        }
    } else if (warp < kConvWarps) {
        // ================= state chunks -> hi / lo parts in tensor memory; epilogues
        // thread = value channel c (its lane of the warp's quadrant).  Per chunk it reads
        // the 16 key rows of its channel (a warp reads 128 contiguous bytes per row), the
        // slot takes the chunk three further on (the next unit's, past this unit's last),
        // and the rows are split into bf16 hi / lo pairs along the key rows -- the layout
        // of an A operand in tensor memory -- and stored.  Before converting a unit the
        // warps read the previous unit's outputs from D (which frees D and the parts).
        const int c = tid;
        auto epilogue = [&](int it) {
            // lane quadrant = warp: value channel c, every node; after all of unit it's
            // products.  Returns false when a wait gave up.
            // (one decision for the four warps: they meet at named barriers)
            bool ok = true;
            if (tid == 0) {
                ok = !late_now() && ptx::mbar_wait(b_dfull(it), ph(it), kWaitLimit);
                if (!ok) atomicOr(sLate, 2);
            }
            if (!named_barrier_and(1, kConvWarps * 32, ok)) return false;
            ptx::tc_fence_after_sync();
            const int *mt = meta(it);
            const int n = mt[kMN], off = mt[kMOff];
            const int u = unit_of(it), h = u % H;
            if (mt[kMZero])
                for (int i = 0; i < n; ++i) a.out[((size_t)(off + i) * H + h) * kDvD + c] = 0.f;
            if (mt[kMRun]) {  // the products are done (verdict above): D holds the outputs
                constexpr int CW = NP < 32 ? NP : 32;
#pragma unroll
                for (int cb = 0; cb < NP; cb += CW) {
                    uint32_t dv[CW];
                    tmem_ld_n<CW>(tD + (static_cast<uint32_t>(32 * warp) << 16) + cb, dv);
                    ptx::tmem_wait_ld();
                    float *o = a.out + ((size_t)(off + cb) * H + h) * kDvD + c;
#pragma unroll
                    for (int i = 0; i < CW; ++i)
                        if (cb + i < n) o[(size_t)i * H * kDvD] = __uint_as_float(dv[i]);
                }
            }
            ptx::tc_fence_before_sync();
            __syncwarp();
            if (lane == 0) ptx::mbar_arrive(b_dfree(it));
            return true;
        };
        bool go = true;
        int it = 0;
        for (; it < nu && go; ++it) {
            if (it >= 1 && !epilogue(it - 1)) {
                go = false;
                break;
            }
            bool tok = true;
            if (tid == 0) {
                tok = !late_now() && ptx::mbar_wait(b_tree(it), ph(it), kWaitLimit);
                if (!tok) atomicOr(sLate, 2);
            }
            if (!named_barrier_and(1, kConvWarps * 32, tok)) {
                go = false;
                break;
            }
            const bool run = meta(it)[kMRun] != 0;
            int q = 0;
            for (; q < nch; ++q) {
                const int gq = it * nch + q, slot = gq % kRing;
                bool cok = true;
                if (tid == 0) {
                    // stop when another role gave up, or when this chunk does not land
                    cok = !late_now() &&
                          ((gq == 0 && P.expire_first_wait)
                               ? false  // test hook: treated as expired
                               : ptx::mbar_wait(b_slot(slot), (gq / kRing) & 1, kWaitLimit));
                    if (!cok) atomicOr(sLate, 2);
                }
                // (the verdict travels with the barrier: a flag read after it could already
                // hold thread 0's verdict on the next chunk)
                if (!named_barrier_and(1, kConvWarps * 32, cok)) break;  // stop converting
                const float *cp = reinterpret_cast<const float *>(sH + slot * kChunkBytesD);
                float x[kChunkRowsD];
#pragma unroll
                for (int r = 0; r < kChunkRowsD; ++r) x[r] = cp[r * kDvD + c];
                if (gq + kRing < nu * nch) {
                    named_barrier(1, kConvWarps * 32);  // every thread has read the chunk
                    if (tid == 0) {
                        ptx::fence_proxy_async_smem();
                        ptx::mbar_arrive_expect_tx(b_slot(slot), kChunkBytesD);
                        ptx::bulk_g2s(hA + slot * kChunkBytesD, chunk_src(gq + kRing), kChunkBytesD,
                                      b_slot(slot));
                        sIssued[slot] = gq + kRing;
                    }
                }
                if (run) {
                    uint32_t hi[kChunkRowsD / 2], lo[kChunkRowsD / 2];
#pragma unroll
                    for (int m = 0; m < kChunkRowsD / 2; ++m)
                        split_pair(x[2 * m], x[2 * m + 1], hi[m], lo[m]);
                    const uint32_t ta = tA + q * 16u + (static_cast<uint32_t>(32 * warp) << 16);
                    ptx::tmem_st_x8(ta, hi);
                    ptx::tmem_st_x8(ta + 8u, lo);
                    ptx::tmem_wait_st();
                    ptx::tc_fence_before_sync();
                }
                __syncwarp();
                if (lane == 0) ptx::mbar_arrive(b_conv(it, q));
            }
            if (q < nch) {
                // after a failed wait the unit's remaining chunks are released unconverted
                // (the outputs are not written then)
                __syncwarp();
                if (lane == 0)
                    for (; q < nch; ++q) ptx::mbar_arrive(b_conv(it, q));
                go = false;
            }
        }
        if (go && nu > 0) epilogue(nu - 1);
        // every state chunk requested lands before the CTA's memory can go away
        if (tid == 0)
            for (int s = 0; s < kRing; ++s)
                if (sIssued[s] >= 0 && !ptx::mbar_wait(b_slot(s), (sIssued[s] / kRing) & 1, kWaitLimit))
                    atomicOr(sLate, 128);
    } else {
        // ================= factors, weights (warps kConvWarps .. kMmaWarp - 1)
        const int t = tid - kConvWarps * 32, fw = warp - kConvWarps;
        constexpr int kFT = kFacWarps * 32;
        // node i = t / kTpn takes pieces kPpt * sub .. of a group's 64 channels
        const int i = t / kTpn, sub = t % kTpn;
        for (int it = 0; it < nu; ++it) {
            bool tok = true;
            if (t == 0) {
                tok = !late_now() && ptx::mbar_wait(b_tree(it), ph(it), kWaitLimit);
                if (!tok) atomicOr(sLate, 4);
            }
            if (!named_barrier_and(2, kFT, tok)) break;
            int *mt = meta(it);
            bool go = mt[kMRun] != 0;
            const int n = mt[kMN], off = mt[kMOff];
            const int u = unit_of(it), h = u % H;
            const uint64_t *anc_s = sAnc(it);
            const int *par_s = sPar(it);
            const bool mine = i < n;
            float gmax = 0.f;  // largest |G| seen: the factor range check
            for (int kg = 0; kg < ng && go; ++kg) {
                uint8_t *fb = sF + kg * kBlock;
                bool fok = true;
                if (t == 0) {
                    fok = !late_now() && ptx::mbar_wait(b_fin(it, kg), ph(it), kWaitLimit);
                    if (!fok) atomicOr(sLate, 4);  // another role gave up, or the columns did not land
                }
                if (!named_barrier_and(2, kFT, fok)) {
                    if (lane == 0) {  // release the product thread
                        ptx::mbar_arrive(b_facq(it, kg));
                        ptx::mbar_arrive(b_fac(it, kg));
                    }
                    go = false;
                    break;
                }
                // path sums of g over this thread's channels: per ancestor, in index order
                // (depth order on a root path), 2 * kPpt independent 16-byte loads.  The g
                // slabs are 128-byte swizzled, so the rows of different ancestors spread
                // over the banks.
                float G[kPpt * 8];
#pragma unroll
                for (int e = 0; e < kPpt * 8; ++e) G[e] = 0.f;
                if (mine) {
                    uint64_t m = anc_s[i];
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
                    if (lane == 0) ptx::mbar_arrive(side == 0 ? b_facq(it, kg) : b_fac(it, kg));
                }
            }
            if (!(gmax <= kGLimit)) atomicOr(&mt[kMWalk], 1);

            // ---- weights, once the unit's context and score products are done
            bool sok = true;
            if (t == 0) {
                sok = !late_now() && ptx::mbar_wait(b_sfull(it), ph(it), kWaitLimit);
                if (!sok) atomicOr(sLate, 4);
            }
            go = named_barrier_and(2, kFT, sok) && go;
            const bool walk = go && mt[kMWalk] != 0;
            uint8_t *wS = sF + (ng - 1) * kBlock;  // the last factor block is free now
            // fp32 weights of the walk after the weight tiles
            float *W32 = reinterpret_cast<float *>(wS + 2 * NP * NP * 2);
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
                        j = par_s[j];
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
                if (lane == 0) vok = ptx::mbar_wait(b_v(it), ph(it), kWaitLimit);
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
                // swizzle (8-row x 16-byte core matrices), hi at the start of the last factor
                // block, lo after it; the two warps of a lane quadrant take half the columns
                constexpr int CW = NP / 2;
                const int wr = 32 * qd + lane, cb = (fw >> 2) * CW;
                const uint64_t m = wr < NP ? anc_s[wr] : 0ull;
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
                    uint8_t *wh = wS + (wr / 8) * kSboW + (wr % 8) * 16 + (cb / 8) * 128;
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
            if (lane == 0) ptx::mbar_arrive(b_wready(it));
        }
    }

    // ================= all roles done: report, free tensor memory
    ptx::tc_fence_before_sync();
    __syncthreads();
    if (tid == 0 && *sLate) report(a.status, TV_ERR_TIMEOUT);
    if (warp == kMmaWarp) ptx::tmem_dealloc(tmem, P.tmem_cols);
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
    // persistent: one CTA per resident slot, each taking every grid-th unit
    int dev = 0, sms = 0, per_sm = 0;
    if ((e = cudaGetDevice(&dev)) != cudaSuccess ||
        (e = cudaDeviceGetAttribute(&sms, cudaDevAttrMultiProcessorCount, dev)) != cudaSuccess ||
        (e = resident_ctas(kern, kThreadsD, smem, P.tmem_cols, per_sm)) != cudaSuccess)
        return e;
    const long long units = (long long)a.B * a.H;
    const long long grid = std::min<long long>(units, (long long)sms * per_sm);
    return launch_pdl(kern, dim3((unsigned)grid), dim3(kThreadsD), smem, s, tq, tk, tv_, tg, P);
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
